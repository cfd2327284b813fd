"""usp_forward_noalloc: the forward for callers that cannot allocate device memory (for example a
plugin whose host application owns all device memory, or a latency-critical caller that must not
call cudaMalloc). Its workspace is the library's own fixed scratch array. Through the C ABI, two calls
in a row must match the workspace-taking usp_forward within the parity tolerances. This file is
collected last, so a run that stops at the first failure has run every other test before it."""
import numpy as np
import pytest
import torch

import sequence_long_context_zigzag_gb300 as usp
from seeded_inputs import make_qkv

pytestmark = pytest.mark.gpu


def test_no_alloc_forward_matches_forward_twice():
    bs, L, hq, hkv, hd, ud, rd, chunk = 1, 1024, 8, 4, 128, 2, 4, 4
    for seed in (11, 12):   # two calls in a row; the second reuses the scratch the first left behind
        q, k, v = (x.cuda() for x in make_qkv(bs, L, hq, hkv, hd, "bf16", seed=seed))
        ref_o = torch.empty_like(q)
        ref_l = torch.empty(bs, L, hq, device="cuda")
        usp.usp_forward(q, k, v, ref_o, ref_l, ud, rd, head_chunk=chunk)
        out = torch.full_like(q, float("nan"))
        lse = torch.full((bs, L, hq), float("nan"), device="cuda")
        usp.usp_forward_noalloc(q, k, v, out, lse, ud, rd, head_chunk=chunk)
        usp.usp_check()
        assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
        assert (out.float() - ref_o.float()).abs().max().item() <= 2e-2
        rel = ((lse - ref_l).abs() / ref_l.abs().clamp_min(1.0)).max().item()
        assert rel <= 1e-3
