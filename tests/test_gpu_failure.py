"""Failure detection without a GPU fault: a bounded device-side wait that runs out.

Every kernel of the library waits on mbarriers through one bounded wait that, once its time limit
passes, records USP_ERR_TIMEOUT in the device status word and lets the kernel return. Here the wait
is made to run out on purpose, on a barrier nothing ever arrives on, with a 20 ms limit
(usp_selftest_timeout). Checked: usp_check reports the timeout once and clears it; a tensor-core
attention launch made while the word is set does no work (its output buffer keeps its sentinel) and
is reported too; after the word is cleared the same launch computes the right result, so the context
stays usable."""
import math

import numpy as np
import pytest
import torch

import oracle
import sequence_long_context_zigzag_gb300 as usp
from sequence_long_context_zigzag_gb300 import _abi
from seeded_inputs import make_qkv

pytestmark = pytest.mark.gpu


def test_wait_runs_out_is_reported_once():
    lib = _abi.load()
    torch.cuda.synchronize()
    assert lib.usp_check(None) == _abi.USP_OK
    assert lib.usp_selftest_timeout(20000, None) == _abi.USP_OK
    assert lib.usp_check(None) == _abi.USP_ERR_TIMEOUT
    assert lib.usp_check(None) == _abi.USP_OK


@pytest.mark.parametrize("dt", ["bf16"])
def test_launch_during_a_recorded_timeout_skips_then_recovers(dt):
    lib = _abi.load()
    L, hq, hkv, hd, ud, rd = 1024, 4, 2, 128, 2, 2
    q, k, v = make_qkv(1, L, hq, hkv, hd, dt, seed=31)
    Lr = L // rd
    tdt = q.dtype
    qh = torch.empty(rd, ud, hq // ud, 1, Lr, hd, device="cuda", dtype=tdt)
    kh = torch.empty(rd, ud, hkv // ud, 1, Lr, hd, device="cuda", dtype=tdt)
    vh = torch.empty_like(kh)
    usp.usp_extract_a2a([q.cuda(), k.cuda(), v.cuda()], [qh, kh, vh], rd, ud)
    out = torch.full_like(qh, 7.0)
    lse = torch.full(qh.shape[:5], 7.0, device="cuda")
    torch.cuda.synchronize()
    assert lib.usp_check(None) == _abi.USP_OK
    # the word is set before the attention starts: every CTA sees it and skips its work
    assert lib.usp_selftest_timeout(20000, None) == _abi.USP_OK
    usp.usp_attn_fwd(qh, kh, vh, out, lse, hkv=hkv)
    assert lib.usp_check(None) == _abi.USP_ERR_TIMEOUT
    assert bool((out == 7.0).all()) and bool((lse == 7.0).all())
    # cleared: the same launch computes the attention
    usp.usp_attn_fwd(qh, kh, vh, out, lse, hkv=hkv)
    assert lib.usp_check(None) == _abi.USP_OK
    on = torch.empty(1, L, hq, hd, device="cuda", dtype=tdt)
    ln = torch.empty(1, L, hq, device="cuda")
    usp.usp_extract_a2a([out], [on], rd, ud, inverse=True)
    usp.usp_extract_a2a([lse], [ln], rd, ud, inverse=True)
    rows = list(range(0, L, 37)) + [L - 1]
    o_ref, l_ref = oracle.attn_direct(q, k, v, causal=True, rows=rows)
    tol = 2e-2 if dt == "bf16" else 2e-4
    assert np.abs(on[:, rows].float().cpu().numpy() - o_ref).max() <= tol
    ls = ln[:, rows].cpu().numpy().astype(np.float64)
    assert (np.abs(ls - l_ref) / np.maximum(np.abs(l_ref), 1.0)).max() <= 1e-3
    assert math.isfinite(float(ln.max()))
