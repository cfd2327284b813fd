"""The persistent bf16 forward kernel's walk over its units, through the C ABI.

A unit of work is 256 query rows of one (ring rank, Ulysses rank, head, batch element); one CTA per SM
walks a fixed list of units, carrying its barrier phases, stage ring and tensor-memory hand-offs from
one unit into the next. Checked here at shapes with several units per CTA (more units than the GPU
has SMs), including shapes whose K/V is larger than L2 (units numbered in super-groups of heads, the
super-groups in alternating directions, odd and even counts of them):
every output row is written and matches the oracle on sampled rows; repeated launches give the same
bits; the single-step
modes (whose units can have no visible key at all) fold back into the whole-ring result; one ring
rank's rows alone and packed samples give the bits of the full run.

Bars: out max-abs error <= 2e-2; lse relative error <= 1e-3 with denominator max(|lse|, 1)."""
import numpy as np
import pytest
import torch

import oracle
import sequence_long_context_zigzag_gb300 as usp
from seeded_inputs import make_qkv, make_rows

pytestmark = pytest.mark.gpu
OUT_TOL = 2e-2
LSE_TOL = 1e-3

SHAPES = [  # bs, L, hq, hkv, hd, ud, rd; units = rd * hq * bs * ceil(L / rd / 256)
    (1, 4096, 16, 4, 128, 2, 4),     # 256 units, GQA
    (2, 3072, 8, 8, 64, 1, 3),       # 192 units, hd 64, odd ring degree
    (1, 6000, 8, 2, 128, 2, 2),      # 192 units, Lr = 3000: ragged last unit of every head
    (1, 65536, 8, 8, 128, 1, 2),     # 2048 units; K/V 256 MiB: four super-groups of 2 heads
    (1, 65536, 6, 6, 128, 1, 2),     # 1536 units; K/V 192 MiB: three super-groups (alternating order)
    (4, 32768, 8, 4, 128, 2, 2),     # 4096 units; K/V 256 MiB over 16 (u, kv head, b) groups
    (1, 262144, 2, 2, 128, 1, 2),    # 2048 units; two 128 MiB groups, one per super-group
]


def sharded(q, k, v, ud, rd):
    bs, L, hq, hd = q.shape
    hkv = k.shape[2]
    Lr = L // rd
    qh = torch.empty(rd, ud, hq // ud, bs, Lr, hd, device="cuda", dtype=q.dtype)
    kh = torch.empty(rd, ud, usp.heads_per_rank(hkv, ud), bs, Lr, hd, device="cuda", dtype=q.dtype)
    vh = torch.empty_like(kh)
    usp.usp_extract_a2a([q.cuda(), k.cuda(), v.cuda()], [qh, kh, vh], rd, ud)
    return qh, kh, vh


def natural(oh, lh, bs, L, hq, hd, ud, rd):
    out = torch.empty(bs, L, hq, hd, device="cuda", dtype=oh.dtype)
    lse = torch.empty(bs, L, hq, device="cuda", dtype=torch.float32)
    usp.usp_extract_a2a([oh], [out], rd, ud, inverse=True)
    usp.usp_extract_a2a([lh], [lse], rd, ud, inverse=True)
    return out, lse


def run(qh, kh, vh, hkv, **kw):
    # NaN-filled, so that a unit the walk missed shows up
    oh = torch.full_like(qh, float("nan"))
    lh = torch.full(qh.shape[:5], float("nan"), device="cuda", dtype=torch.float32)
    usp.usp_attn_fwd(qh, kh, vh, oh, lh, hkv=hkv, **kw)
    usp.usp_check()  # a hand-off stall shows as a bounded wait running out, not as wrong bits
    return oh, lh


@pytest.mark.parametrize("bs,L,hq,hkv,hd,ud,rd", SHAPES)
def test_many_units_per_cta_match_oracle(bs, L, hq, hkv, hd, ud, rd):
    q, k, v = make_qkv(bs, L, hq, hkv, hd, "bf16", seed=L + hq + bs)
    qh, kh, vh = sharded(q, k, v, ud, rd)
    o1, l1 = run(qh, kh, vh, hkv)
    o2, l2 = run(qh, kh, vh, hkv)
    # every row of every unit written (causal: each row sees at least its own key), the same bits twice
    assert bool(torch.isfinite(o1).all()) and bool(torch.isfinite(l1).all())
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    out, lse = natural(o1, l1, bs, L, hq, hd, ud, rd)
    rows = make_rows(L, L // (2 * rd), 40, seed=L)
    o_ref, l_ref = oracle.attn_direct(q, k, v, causal=True, rows=rows)
    o = out[:, rows].float().cpu().numpy().astype(np.float64)
    assert np.abs(o - o_ref).max() <= OUT_TOL
    ls = lse[:, rows].cpu().numpy().astype(np.float64)
    assert (np.abs(ls - l_ref) / np.maximum(np.abs(l_ref), 1.0)).max() <= LSE_TOL


def test_single_steps_fold_into_the_whole_ring():
    """One ring step at a time (units of later steps can see no key at all and only write the empty
    partial), merged in place step by step, reproduces the whole-ring launch; every step twice gives
    the same bits."""
    bs, L, hq, hkv, hd, ud, rd = SHAPES[0]
    q, k, v = make_qkv(bs, L, hq, hkv, hd, "bf16", seed=5)
    qh, kh, vh = sharded(q, k, v, ud, rd)
    ref_o, ref_l = run(qh, kh, vh, hkv)
    for t in range(rd):
        o1, l1 = run(qh, kh, vh, hkv, mode=usp.USP_MODE_STEP, step=t)
        o2, l2 = run(qh, kh, vh, hkv, mode=usp.USP_MODE_STEP, step=t)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
    ao = torch.empty_like(qh)
    al = torch.empty(qh.shape[:5], device="cuda", dtype=torch.float32)
    for t in range(rd):
        usp.usp_attn_fwd(qh, kh, vh, ao, al, hkv=hkv, mode=usp.USP_MODE_STEP if t == 0 else usp.USP_MODE_ACCUM,
                         step=t)
    usp.usp_check()
    assert (ao.float() - ref_o.float()).abs().max().item() <= OUT_TOL
    d = (al - ref_l).abs() / ref_l.abs().clamp(min=1.0)
    assert d.max().item() <= LSE_TOL


def test_one_ring_rank_and_packed_samples():
    """ring_rank_only (a subset of the units) writes exactly the full run's rows of that rank; packed
    samples (units that skip tiles, or have none in a ring step) run twice to the same bits."""
    bs, L, hq, hkv, hd, ud, rd = SHAPES[0]
    q, k, v = make_qkv(bs, L, hq, hkv, hd, "bf16", seed=9)
    qh, kh, vh = sharded(q, k, v, ud, rd)
    full_o, full_l = run(qh, kh, vh, hkv)
    for r in range(rd):
        o, l = run(qh, kh, vh, hkv, ring_rank=r)
        assert torch.equal(o[r], full_o[r]) and torch.equal(l[r], full_l[r])
    cu = torch.tensor([0, 1000, 1100, 3000, L], dtype=torch.int32, device="cuda")
    o1, l1 = run(qh, kh, vh, hkv, cu_seqlens=cu)
    o2, l2 = run(qh, kh, vh, hkv, cu_seqlens=cu)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.isfinite(l1).all()
