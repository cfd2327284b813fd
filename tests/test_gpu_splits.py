"""The plain ring's contiguous split and the round-robin stripe split beside zigzag (through the C ABI):
permutes bit-exact against the oracle's split maps, attention against direct attention, and the
per-ring-rank mode (each ring rank's share computed alone) composing to the full result."""
import numpy as np
import pytest
import torch

import oracle
import sequence_long_context_zigzag_gb300 as usp
from seeded_inputs import make_qkv

pytestmark = pytest.mark.gpu


def bits(t):
    t = t.detach().cpu().contiguous()
    return t.view(torch.int16).numpy() if t.dtype == torch.bfloat16 else t.view(torch.int32).numpy()


@pytest.mark.parametrize("split", ["zigzag", "basic", "stripe"])
@pytest.mark.parametrize("L,rd,ud", [(1024, 4, 2), (768, 3, 2), (512, 8, 1)])
def test_split_permutes_bitexact(split, L, rd, ud):
    x = make_qkv(1, L, 4, 4, 128, "bf16", seed=L + rd)[0]
    xd = x.cuda()
    loc = torch.empty(rd, ud, 1, L // (rd * ud), 4, 128, dtype=torch.bfloat16, device="cuda")
    usp.usp_extract_local(xd, loc, rd, ud, split=split)
    ref = oracle.extract_local(bits(x), rd, ud, split=split)
    assert np.array_equal(bits(loc), ref)
    hs = torch.empty(rd, ud, 4 // ud, 1, L // rd, 128, dtype=torch.bfloat16, device="cuda")
    usp.usp_extract_a2a([xd], [hs], rd, ud, split=split)
    assert np.array_equal(bits(hs), oracle.a2a_fwd(ref, ud))
    back = torch.zeros_like(xd)
    usp.usp_extract_a2a([hs], [back], rd, ud, inverse=True, split=split)
    assert torch.equal(back, xd)
    usp.usp_check()


@pytest.mark.parametrize("split", ["basic", "stripe"])
@pytest.mark.parametrize("L,hq,hkv,hd,dtype,ud,rd", [(1024, 4, 2, 128, "bf16", 2, 2), (1000, 4, 4, 128, "bf16", 2, 4),
                                                     (768, 2, 1, 64, "bf16", 1, 3), (512, 4, 4, 64, "f32", 1, 4)])
def test_split_attention_matches_direct(split, L, hq, hkv, hd, dtype, ud, rd):
    q, k, v = make_qkv(1, L, hq, hkv, hd, dtype, seed=L + hq + rd)
    out, lse = usp.usp_attention(q.cuda(), k.cuda(), v.cuda(), ud=ud, rd=rd, split=split)
    usp.usp_check()
    o_ref, l_ref = oracle.attn_direct(q, k, v)
    assert np.abs(out.float().cpu().numpy() - o_ref).max() <= 2e-2
    assert (np.abs(lse.cpu().numpy() - l_ref) / np.maximum(np.abs(l_ref), 1)).max() <= 1e-3


@pytest.mark.parametrize("split", ["zigzag", "basic", "stripe"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_ring_rank_shares_compose_to_full(split, dtype):
    """Computing each ring rank's query rows alone (the per-rank timing mode) writes exactly the
    rows of the full launch, bit for bit."""
    L, hq, hkv, hd, ud, rd = 1024, 4, 2, 128 if dtype == "bf16" else 64, 2, 4
    q, k, v = make_qkv(1, L, hq, hkv, hd, dtype, seed=5)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    dt = qd.dtype
    qh = torch.empty(rd, ud, hq // ud, 1, L // rd, hd, dtype=dt, device="cuda")
    kh = torch.empty(rd, ud, hkv // ud, 1, L // rd, hd, dtype=dt, device="cuda")
    vh = torch.empty_like(kh)
    usp.usp_extract_a2a([qd, kd, vd], [qh, kh, vh], rd, ud, split=split)
    full_o, full_l = torch.empty_like(qh), torch.empty(qh.shape[:5], device="cuda")
    usp.usp_attn_fwd(qh, kh, vh, full_o, full_l, split=split)
    part_o, part_l = torch.full_like(qh, float("nan")), torch.full(qh.shape[:5], float("nan"), device="cuda")
    for r in range(rd):
        usp.usp_attn_fwd(qh, kh, vh, part_o, part_l, split=split, ring_rank=r)
        # only rank r's rows are written so far
        assert not torch.isnan(part_l[r]).any() and torch.isnan(part_l[r + 1:]).all()
    usp.usp_check()
    assert torch.equal(part_o, full_o) and torch.equal(part_l, full_l)
