"""The profiling runner (sequence_long_context_zigzag_gb300.kernel_run) runs each kernel it offers on
a small shape without a device-side error, so the commands recorded with the ncu summaries work."""
import pytest

from sequence_long_context_zigzag_gb300 import kernel_run

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kernel", ["attn", "split_a2a", "a2a_inv", "bwd"])
def test_kernel_run_small(kernel, capsys):
    kernel_run.main(["--L", "1024", "--hq", "8", "--hkv", "2", "--ud", "2", "--rd", "4", "--kernel", kernel,
                     "--launches", "2"])
    assert f"2 launch(es) of {kernel}" in capsys.readouterr().out


def test_kernel_run_packed(capsys):
    kernel_run.main(["--L", "2048", "--hq", "4", "--hkv", "4", "--ud", "2", "--rd", "2", "--nseq", "4"])
    assert "nseq=4" in capsys.readouterr().out
