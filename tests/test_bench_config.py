"""bench.py's JSON contract pieces that need no GPU: both arms report one metric string and one
config, and the config's L2 statement is computed from the shapes of the buffers the step uses."""
import torch

import bench
import sequence_long_context_zigzag_gb300 as usp
from seeded_inputs import WORKLOADS


def test_working_set_matches_the_step_buffers():
    for w in WORKLOADS:
        dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        q = torch.empty(w.bs, w.L, w.hq, w.hd, dtype=dt)  # never written: shapes only
        k = torch.empty(w.bs, w.L, w.hkv, w.hd, dtype=dt)
        step = bench.Step(usp, w, q, k, k)
        ws = sum(t.numel() * t.element_size() for t in (q, k, k, step.qh, step.kh, step.vh, step.oh, step.o_loc))
        assert ws == bench.step_working_set_bytes(w), w.name


def test_l2_statement():
    assert bench.workload_config(WORKLOADS[1])["l2"] == "step working set 512 MiB > L2 (129 MB); no flush"
    assert "fits in L2" in bench.workload_config(WORKLOADS[0])["l2"]


def test_reference_arm_reports_the_same_metric_and_config(capsys, monkeypatch):
    import json
    import sys
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0",
                                      "--workload", "0"])
    bench.main()
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["config"] == bench.workload_config(WORKLOADS[0])
    assert line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
