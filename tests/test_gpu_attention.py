"""GPU parity of the ring attention forward (steps a3 + a4) and of the whole USP-Attention forward
(a1 - a6) against the oracle, through the C ABI.

Bars: out max-abs error <= 2e-2; lse relative error <= 1e-3 with denominator max(|lse|, 1)."""
import math

import numpy as np
import pytest
import torch

import oracle
import sequence_long_context_zigzag_gb300 as usp
from seeded_inputs import make_qkv

pytestmark = pytest.mark.gpu
OUT_TOL = 2e-2
LSE_TOL = 1e-3


def lse_err(lse, ref):
    lse = np.asarray(lse, dtype=np.float64)
    both_inf = np.isneginf(lse) & np.isneginf(ref)
    d = np.where(both_inf, 0.0, np.abs(lse - ref) / np.maximum(np.abs(ref), 1.0))
    return float(np.nan_to_num(d, nan=np.inf).max()) if d.size else 0.0


def out_err(out, ref):
    return float(np.abs(out.float().cpu().numpy().astype(np.float64) - ref).max()) if ref.size else 0.0


CASES = [  # bs, L, hq, hkv, hd, dtype, ud, rd, causal
    (1, 1024, 4, 4, 64, "f32", 1, 4, True),       # the tiny fp32 workload, all rows
    (1, 512, 4, 2, 128, "bf16", 2, 2, True),
    (2, 1000, 4, 4, 128, "bf16", 2, 4, True),     # c = 125: tiles straddle chunks, ragged tails
    (1, 768, 8, 2, 128, "bf16", 2, 3, True),      # GQA G = 4, odd ring degree
    (1, 640, 4, 1, 64, "bf16", 1, 5, True),       # MQA (ud = 1)
    (1, 512, 4, 4, 128, "bf16", 4, 1, True),      # pure Ulysses
    (1, 2048, 2, 2, 128, "bf16", 1, 8, True),     # pure ring, several 128-row tiles per chunk
    (1, 512, 2, 2, 64, "bf16", 1, 1, False),      # non-causal
    (1, 384, 4, 2, 128, "f32", 2, 2, False),
    (1, 1536, 4, 2, 128, "bf16", 2, 2, True),     # chunks of 384 rows: 3 tiles per chunk
]


@pytest.mark.parametrize("bs,L,hq,hkv,hd,dtype,ud,rd,causal", CASES)
def test_usp_attention_matches_direct(bs, L, hq, hkv, hd, dtype, ud, rd, causal):
    q, k, v = make_qkv(bs, L, hq, hkv, hd, dtype, seed=L + hq + 10 * rd + ud)
    out, lse = usp.usp_attention(q.cuda(), k.cuda(), v.cuda(), ud=ud, rd=rd, causal=causal)
    usp.usp_check()
    o_ref, l_ref = oracle.attn_direct(q, k, v, causal=causal)
    assert out_err(out, o_ref) <= OUT_TOL
    assert lse_err(lse.cpu().numpy(), l_ref) <= LSE_TOL


def test_head_chunks_identical_to_unchunked():
    """Processing heads in groups (a6) gives exactly the unchunked result."""
    q, k, v = make_qkv(1, 512, 8, 4, 128, "bf16", seed=5)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = usp.usp_attention(q, k, v, ud=2, rd=2)
    o2, l2 = usp.usp_attention(q, k, v, ud=2, rd=2, head_chunk=4)
    usp.usp_check()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def ring_inputs(L, hq, hkv, hd, dtype, ud, rd, seed):
    q, k, v = make_qkv(1, L, hq, hkv, hd, dtype, seed=seed)
    Lu, Lr = L // (rd * ud), L // rd
    dev = [x.cuda() for x in (q, k, v)]
    hs = []
    for x, H in zip(dev, (hq, hkv, hkv)):
        loc = torch.empty(rd, ud, 1, Lu, H, hd, dtype=x.dtype, device="cuda")
        usp.usp_extract_local(x, loc, rd, ud)
        h = torch.empty(rd, ud, H // ud, 1, Lr, hd, dtype=x.dtype, device="cuda")
        usp.usp_a2a4d(loc, h, rd, ud, 1)
        hs.append(h)
    return (q, k, v), hs


@pytest.mark.parametrize("L,hq,hkv,hd,dtype,ud,rd", [(512, 4, 2, 128, "bf16", 2, 2), (768, 2, 2, 64, "bf16", 1, 3),
                                                     (1000, 4, 4, 128, "bf16", 2, 4),
                                                     (256, 2, 1, 64, "f32", 1, 4)])
def test_ring_steps_match_oracle_blocks(L, hq, hkv, hd, dtype, ud, rd):
    """USP_MODE_STEP writes the partial (o_t, lse_t) of ring step t; it matches the oracle's block
    attention of rank r's queries against rank (r - t) mod rd's keys (Fig. 1 schedule). Folding the
    steps with USP_MODE_ACCUM reproduces USP_MODE_FUSED."""
    (q, k, v), (qh, kh, vh) = ring_inputs(L, hq, hkv, hd, dtype, ud, rd, seed=L + rd)
    c, Lr = L // (2 * rd), L // rd
    scale = 1.0 / math.sqrt(hd)
    Q = oracle.a2a_fwd(oracle.extract_local(q.double().numpy(), rd, ud), ud)
    K = oracle.a2a_fwd(oracle.extract_local(k.double().numpy(), rd, ud), ud)
    V = oracle.a2a_fwd(oracle.extract_local(v.double().numpy(), rd, ud), ud)
    acc_o, acc_l = torch.empty_like(qh), torch.empty(qh.shape[:5], device="cuda", dtype=torch.float32)
    for t in range(rd):
        o_t, l_t = torch.empty_like(qh), torch.empty_like(acc_l)
        usp.usp_attn_fwd(qh, kh, vh, o_t, l_t, mode=usp.USP_MODE_STEP, step=t)
        usp.usp_attn_fwd(qh, kh, vh, acc_o, acc_l, mode=usp.USP_MODE_STEP if t == 0 else usp.USP_MODE_ACCUM,
                         step=t)
        usp.usp_check()
        o_np, l_np = o_t.float().cpu().numpy(), l_t.cpu().numpy()
        for r in range(rd):
            s = oracle.ring_source(r, t, rd)
            for u in range(ud):
                o_ref, l_ref = oracle.attn_block(Q[r, u, :, 0], oracle.zig(r, np.arange(Lr), c, rd), K[s, u, :, 0],
                                                 V[s, u, :, 0], oracle.zig(s, np.arange(Lr), c, rd), scale)
                assert np.abs(o_np[r, u, :, 0] - o_ref).max() <= OUT_TOL
                assert lse_err(l_np[r, u, :, 0], l_ref) <= LSE_TOL
    fo, fl = torch.empty_like(qh), torch.empty_like(acc_l)
    usp.usp_attn_fwd(qh, kh, vh, fo, fl)
    usp.usp_check()
    assert (acc_o.float() - fo.float()).abs().max().item() <= OUT_TOL
    assert lse_err(acc_l.cpu().numpy(), fl.cpu().numpy().astype(np.float64)) <= LSE_TOL
