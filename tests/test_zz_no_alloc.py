"""usp_forward_noalloc: the forward for callers that cannot allocate device memory (for example a
plugin whose host application owns all device memory, or a latency-critical caller that must not
call cudaMalloc). Its workspace is the library's own fixed scratch array. Through the C ABI, two calls
in a row must give exactly the bytes of the workspace-taking usp_forward (the same kernels on the same
inputs, so any difference would come from the shared scratch), and both must match the oracle within
the parity tolerances. This file is collected last, so a run that stops at the first failure has run
every other test before it."""
import numpy as np
import pytest
import torch

import oracle
import sequence_long_context_zigzag_gb300 as usp
from seeded_inputs import make_qkv

pytestmark = pytest.mark.gpu


def test_no_alloc_forward_matches_forward_twice():
    bs, L, hq, hkv, hd, ud, rd, chunk = 1, 1024, 8, 4, 128, 2, 4, 4
    for seed in (11, 12):   # two calls in a row; the second reuses the scratch the first left behind
        q_h, k_h, v_h = make_qkv(bs, L, hq, hkv, hd, "bf16", seed=seed)
        q, k, v = q_h.cuda(), k_h.cuda(), v_h.cuda()
        ref_o = torch.empty_like(q)
        ref_l = torch.empty(bs, L, hq, device="cuda")
        usp.usp_forward(q, k, v, ref_o, ref_l, ud, rd, head_chunk=chunk)
        out = torch.full_like(q, float("nan"))
        lse = torch.full((bs, L, hq), float("nan"), device="cuda")
        usp.usp_forward_noalloc(q, k, v, out, lse, ud, rd, head_chunk=chunk)
        usp.usp_check()
        assert torch.equal(out.view(torch.int16), ref_o.view(torch.int16))
        assert torch.equal(lse.view(torch.int32), ref_l.view(torch.int32))
        o_ref, l_ref = oracle.attn_direct(q_h, k_h, v_h, causal=True)
        err_o = np.abs(out.float().cpu().numpy() - o_ref).max()
        err_l = (np.abs(lse.cpu().numpy() - l_ref) / np.maximum(np.abs(l_ref), 1.0)).max()
        assert err_o <= 2e-2 and err_l <= 1e-3, (err_o, err_l)


def test_no_alloc_rejects_a_workspace_beyond_the_array():
    """A head group whose workspace exceeds the 32 MiB array is refused before anything runs."""
    bs, L, hq, hkv, hd, ud, rd = 1, 65536, 8, 8, 128, 2, 4
    q = torch.zeros(bs, L, hq, hd, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(bs, L, hkv, hd, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(bs, L, hq, device="cuda")
    with pytest.raises(usp.UspError):
        usp.usp_forward_noalloc(q, k, k, out, lse, ud, rd)
    usp.usp_check()
