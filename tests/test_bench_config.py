"""bench.py's JSON contract pieces that need no GPU: both arms report one metric string and one
config, the config's L2 statement is computed from the shapes of the buffers the step uses, and the
clock record keeps the samples of the timed region and the throttle reasons seen in them."""
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


class _DoneProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _sampler_with(lines, tmp_path):
    s = bench.ClockSampler(0)
    path = tmp_path / "clocks.csv"
    path.write_text("".join(x + "\n" for x in lines))
    s.path, s.proc = str(path), _DoneProc()
    return s


def _row(t, mhz, slow="Not Active", cap="Not Active"):
    # timestamp, index, clocks.sm, clocks.max.sm, power, active mask, hw_slowdown, hw_thermal,
    # sw_thermal, sw_power_cap (the sampler's query, csv without header or units)
    return f"2026/01/01 00:00:{t:06.3f}, 0, {mhz}, 2070, 1300.00, 0x0000000000000000, {slow}, Not Active, " \
           f"Not Active, {cap}"


def test_clock_sampler_keeps_the_timed_region(tmp_path):
    import datetime
    base = datetime.datetime(2026, 1, 1).timestamp()
    lines = [_row(1.0, 1200), _row(2.0, 2000, cap="Active"), _row(2.05, 2040), _row(2.1, 2070),
             _row(3.0, 900, slow="Active"), "garbage line", ""]
    got = _sampler_with(lines, tmp_path).stop(base + 1.5, base + 2.5)
    assert got["window"] == "timed region" and got["samples"] == 3
    assert got["sm_mhz"] == 2040 and got["sm_max_mhz"] == 2070
    assert got["reasons"] == ["sw_power_cap"]  # the hw_slowdown sample is outside the region


def test_clock_sampler_falls_back_to_every_sample(tmp_path):
    import datetime
    base = datetime.datetime(2026, 1, 1).timestamp()
    got = _sampler_with([_row(1.0, 1500, slow="Active"), _row(1.2, 1700)], tmp_path).stop(base + 5, base + 6)
    assert got["window"].startswith("sampler run") and got["samples"] == 2
    assert got["reasons"] == ["hw_slowdown"] and got["sm_mhz"] == 1600


def test_traffic_is_reported_only_for_the_captured_source(monkeypatch, tmp_path):
    """roofline.traffic comes from the committed ncu record only while the forward kernel's sources
    hash to the value recorded there, and only for the workload it was captured on."""
    import json
    for w in WORKLOADS:
        rec = bench.traffic_for_current_kernel(w)
        assert rec is None or rec > 0
    f = tmp_path / "traffic.json"
    w = WORKLOADS[bench.DEFAULT_WORKLOAD]
    f.write_text(json.dumps({"records": [{"workload": w.name, "attn_src_sha256_16": "0" * 16,
                                          "dram_bytes_per_launch": 123}]}))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.traffic_for_current_kernel(w) is None
    f.write_text(json.dumps({"records": [{"workload": w.name, "attn_src_sha256_16": bench.attn_src_hash(),
                                          "dram_bytes_per_launch": 123}]}))
    assert bench.traffic_for_current_kernel(w) == 123
    assert bench.traffic_for_current_kernel(WORKLOADS[0]) is None


def test_peak_follows_the_timed_region():
    """A timed region shorter than a second is a burst (the burst cuBLAS rate applies); a longer one
    runs under the power cap (the sustained rate)."""
    peaks = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    v, why = bench.pick_peak(peaks, "measured", 0.01)
    assert v == 1900.0 and "bf16_tflops " in why.replace("=", " ")
    v, why = bench.pick_peak(peaks, "measured", 7.0)
    assert v == 1700.0 and "bf16_tflops_sustained" in why


def test_default_workload_is_the_largest_single_gpu_one():
    w = WORKLOADS[bench.DEFAULT_WORKLOAD]
    assert w.L == max(x.L for x in WORKLOADS) and w.dtype == "bf16" and w.head_chunk == 8


def test_e2e_head_groups_are_valid():
    """The host-buffer pipeline's head groups divide the heads and keep whole KV groups on every
    Ulysses rank (or replicate one KV head)."""
    for w in WORKLOADS:
        hc = bench.e2e_head_chunk(w)
        if hc is None:
            continue
        G = w.hq // w.hkv
        assert w.hq % hc == 0 and hc % G == 0 and hc % w.ud == 0
        hkc = hc // G
        assert hkc % w.ud == 0 or w.ud % hkc == 0
