"""Packed sequences on the GPU (several samples concatenated into one sequence, each attending only
within itself -- the sequence packing of the Context-Parallel page's ByteScale section): parity of
the forward with the oracle's per-sample attention (out max-abs 2e-2, lse relative 1e-3 with
denominator max(|lse|, 1)), across sample boundaries inside tiles, zigzag chunks and ring ranks."""
import numpy as np
import pytest
import torch

import oracle
import sequence_long_context_zigzag_gb300 as usp
from seeded_inputs import make_qkv

pytestmark = pytest.mark.gpu


def check(out, lse, q, k, v, cu, causal=True):
    o_ref, l_ref = oracle.attn_direct(q, k, v, causal=causal, cu_seqlens=cu)
    o, l = out.float().cpu().numpy(), lse.cpu().numpy()
    err_o = np.abs(o - o_ref).max()
    err_l = (np.abs(l - l_ref) / np.maximum(np.abs(l_ref), 1)).max()
    assert err_o <= 2e-2, err_o
    assert err_l <= 1e-3, err_l


CASES = [
    (2048, 8, 2, 128, 2, 4, "bf16", [0, 100, 700, 701, 1500, 2048]),     # boundaries inside tiles and chunks
    (2048, 8, 8, 64, 1, 4, "bf16", [0, 1024, 2048]),                      # two halves
    (4096, 8, 2, 128, 2, 2, "bf16", list(range(0, 4097, 256))),         # 16 samples of 256
    (1000, 4, 4, 128, 2, 5, "bf16", [0, 1, 2, 3, 400, 999, 1000]),       # one-token samples, ragged tiles
    (512, 8, 1, 128, 4, 2, "bf16", [0, 130, 512]),                        # MQA, replicated K/V
    (512, 4, 2, 64, 2, 2, "f32", [0, 17, 300, 512]),                      # fp32 path
]


@pytest.mark.parametrize("L,hq,hkv,hd,ud,rd,dt,cu", CASES)
def test_packed_forward_matches_oracle(L, hq, hkv, hd, ud, rd, dt, cu):
    q, k, v = make_qkv(1, L, hq, hkv, hd, dt, seed=L + len(cu))
    cud = torch.tensor(cu, dtype=torch.int32, device="cuda")
    out, lse = usp.usp_attention(q.cuda(), k.cuda(), v.cuda(), ud=ud, rd=rd, cu_seqlens=cud)
    usp.usp_check()
    check(out, lse, q, k, v, cu)
    # the sequence-sharded path (usp_attn_fwd per head group) gives the same bytes
    out_s, _ = usp.usp_attention(q.cuda(), k.cuda(), v.cuda(), ud=ud, rd=rd, cu_seqlens=cud, natural_output=False)
    nat = torch.empty_like(out)
    usp.usp_extract_local(out_s, nat, rd, ud, inverse=True)
    usp.usp_check()
    assert torch.equal(nat, out)


@pytest.mark.parametrize("split", ["basic", "stripe"])
def test_packed_other_splits(split):
    L, hq, hkv, hd, ud, rd, cu = 2048, 4, 2, 128, 2, 4, [0, 300, 301, 1100, 2048]
    q, k, v = make_qkv(1, L, hq, hkv, hd, "bf16", seed=5)
    cud = torch.tensor(cu, dtype=torch.int32, device="cuda")
    out, lse = usp.usp_attention(q.cuda(), k.cuda(), v.cuda(), ud=ud, rd=rd, split=split, cu_seqlens=cud)
    usp.usp_check()
    check(out, lse, q, k, v, cu)


def test_packed_noncausal():
    L, hq, hkv, hd, ud, rd, cu = 1024, 4, 4, 128, 2, 2, [0, 200, 900, 1024]
    q, k, v = make_qkv(1, L, hq, hkv, hd, "bf16", seed=6)
    cud = torch.tensor(cu, dtype=torch.int32, device="cuda")
    out, lse = usp.usp_attention(q.cuda(), k.cuda(), v.cuda(), ud=ud, rd=rd, causal=False, cu_seqlens=cud)
    usp.usp_check()
    check(out, lse, q, k, v, cu, causal=False)


def test_one_sample_equals_unpacked():
    L, hq, hd, ud, rd = 2048, 8, 128, 2, 4
    q, k, v = make_qkv(1, L, hq, hq, hd, "bf16", seed=7)
    cud = torch.tensor([0, L], dtype=torch.int32, device="cuda")
    a, la = usp.usp_attention(q.cuda(), k.cuda(), v.cuda(), ud=ud, rd=rd)
    b, lb = usp.usp_attention(q.cuda(), k.cuda(), v.cuda(), ud=ud, rd=rd, cu_seqlens=cud)
    usp.usp_check()
    assert torch.equal(a, b) and torch.equal(la, lb)


def test_many_samples_past_the_shared_memory_copy():
    """More samples than the forward kernel keeps in shared memory (4095): the sample search falls
    back to global memory. L = 8192 as 5462 samples of 1 or 2 tokens, every row against the oracle."""
    L, hq, hkv, hd, ud, rd = 8192, 4, 2, 128, 2, 2
    lens = [1 + (i % 2) for i in range(5462)]
    lens[-1] = L - sum(lens[:-1])
    cu = [0]
    for n in lens:
        cu.append(cu[-1] + n)
    assert cu[-1] == L and len(cu) - 1 > 4095 and min(lens) >= 1
    q, k, v = make_qkv(1, L, hq, hkv, hd, "bf16", seed=77)
    cud = torch.tensor(cu, dtype=torch.int32, device="cuda")
    out, lse = usp.usp_attention(q.cuda(), k.cuda(), v.cuda(), ud=ud, rd=rd, cu_seqlens=cud)
    usp.usp_check()
    check(out, lse, q, k, v, cu)


def test_packing_full_size_sampled():
    """The L = 32768 GQA workload packed as 32 samples of 1024, at full size: sampled rows against
    the oracle's per-sample attention."""
    from seeded_inputs import WORKLOADS, default_seed, make_rows, make_workload_qkv
    w = WORKLOADS[2]
    q, k, v = make_workload_qkv(w, default_seed(2))
    cu = list(range(0, w.L + 1, 1024))
    cud = torch.tensor(cu, dtype=torch.int32, device="cuda")
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out, lse = usp.usp_attention(qd, kd, vd, ud=w.ud, rd=w.rd, cu_seqlens=cud)
    usp.usp_check()
    rows = np.array(make_rows(w.L, w.c, 64, 3))
    o_ref, l_ref = oracle.attn_direct(q, k, v, rows=rows, cu_seqlens=cu)
    rt = torch.as_tensor(rows, device="cuda")
    assert np.abs(out.index_select(1, rt).float().cpu().numpy() - o_ref).max() <= 2e-2
    l = lse.index_select(1, rt).cpu().numpy()
    assert (np.abs(l - l_ref) / np.maximum(np.abs(l_ref), 1)).max() <= 1e-3


BWD_CASES = [
    (2048, 8, 2, 128, 2, 4, "bf16", [0, 100, 700, 701, 1500, 2048], True),
    (1000, 4, 4, 64, 2, 5, "bf16", [0, 1, 2, 3, 400, 999, 1000], True),
    (512, 8, 1, 128, 4, 2, "bf16", [0, 130, 512], True),                 # MQA, replica sums
    (1024, 4, 4, 128, 2, 2, "bf16", [0, 200, 900, 1024], False),        # non-causal
    (512, 4, 2, 64, 2, 2, "f32", [0, 17, 300, 512], True),
]


@pytest.mark.parametrize("L,hq,hkv,hd,ud,rd,dt,cu,causal", BWD_CASES)
def test_packed_backward_matches_oracle(L, hq, hkv, hd, ud, rd, dt, cu, causal):
    q, k, v = make_qkv(1, L, hq, hkv, hd, dt, seed=L + 3 * len(cu))
    g, _, _ = make_qkv(1, L, hq, hkv, hd, dt, seed=L + 3 * len(cu) + 500)
    cud = torch.tensor(cu, dtype=torch.int32, device="cuda")
    qd, kd, vd, gd = q.cuda(), k.cuda(), v.cuda(), g.cuda()
    out = torch.empty_like(qd)
    lse = torch.empty(1, L, hq, device="cuda")
    usp.usp_forward(qd, kd, vd, out, lse, ud, rd, causal=causal, cu_seqlens=cud)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    usp.usp_backward(qd, kd, vd, out, lse, gd, dq, dk, dv, ud, rd, causal=causal, cu_seqlens=cud)
    usp.usp_check()
    rq, rk, rv = oracle.attn_direct_bwd(q, k, v, g, causal=causal, cu_seqlens=cu)
    tol = 2e-2 if dt == "bf16" else 2e-4
    for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
        err = np.abs(got.float().cpu().numpy() - ref).max() / max(np.abs(ref).max(), 1.0)
        assert err <= tol, err


def test_packed_autograd():
    L, hq, hkv, hd, ud, rd, cu = 1024, 4, 2, 128, 2, 2, [0, 300, 301, 1024]
    q, k, v = make_qkv(1, L, hq, hkv, hd, "bf16", seed=71)
    g, _, _ = make_qkv(1, L, hq, hkv, hd, "bf16", seed=72)
    cud = torch.tensor(cu, dtype=torch.int32, device="cuda")
    qd, kd, vd = (x.cuda().requires_grad_(True) for x in (q, k, v))
    out = usp.UspAttentionFunction.apply(qd, kd, vd, ud, rd, True, None, None, "zigzag", cud)
    (out.float() * g.cuda().float()).sum().backward()
    usp.usp_check()
    rq, rk, rv = oracle.attn_direct_bwd(q, k, v, g, cu_seqlens=cu)
    for got, ref in ((qd.grad, rq), (kd.grad, rk), (vd.grad, rv)):
        assert np.abs(got.float().cpu().numpy() - ref).max() / max(np.abs(ref).max(), 1.0) <= 2e-2


@pytest.mark.parametrize("L,hq,hkv,hd,ud,rd,cu", [(2048, 4, 2, 128, 2, 4, [0, 100, 700, 701, 1500, 2048]),
                                                  (1024, 4, 4, 64, 1, 2, list(range(0, 1025, 128)))])
def test_packed_ring_steps_match_oracle_blocks(L, hq, hkv, hd, ud, rd, cu):
    """Packed samples in the single-step modes: USP_MODE_STEP's partial of ring step t matches the
    oracle's block attention of rank r's queries against rank (r - t) mod rd's keys restricted to each
    query's sample (rows with no key in that block: (0, -inf)); folding the steps with
    USP_MODE_ACCUM reproduces USP_MODE_FUSED."""
    import math
    q, k, v = make_qkv(1, L, hq, hkv, hd, "bf16", seed=L + 3 * len(cu))
    cud = torch.tensor(cu, dtype=torch.int32, device="cuda")
    Lu, Lr, c = L // (rd * ud), L // rd, L // (2 * rd)
    hs = []
    for x, H in zip((q, k, v), (hq, hkv, hkv)):
        h = torch.empty(rd, ud, H // ud, 1, Lr, hd, dtype=x.dtype, device="cuda")
        usp.usp_extract_a2a([x.cuda()], [h], rd, ud)
        hs.append(h)
    qh, kh, vh = hs
    Q = oracle.a2a_fwd(oracle.extract_local(q.double().numpy(), rd, ud), ud)
    K = oracle.a2a_fwd(oracle.extract_local(k.double().numpy(), rd, ud), ud)
    V = oracle.a2a_fwd(oracle.extract_local(v.double().numpy(), rd, ud), ud)
    _, _, seg = oracle.seg_bounds(cu, L)
    scale = 1.0 / math.sqrt(hd)
    acc_o, acc_l = torch.empty_like(qh), torch.empty(qh.shape[:5], device="cuda", dtype=torch.float32)
    for t in range(rd):
        o_t, l_t = torch.empty_like(qh), torch.empty_like(acc_l)
        usp.usp_attn_fwd(qh, kh, vh, o_t, l_t, mode=usp.USP_MODE_STEP, step=t, cu_seqlens=cud)
        usp.usp_attn_fwd(qh, kh, vh, acc_o, acc_l, mode=usp.USP_MODE_STEP if t == 0 else usp.USP_MODE_ACCUM,
                         step=t, cu_seqlens=cud)
        usp.usp_check()
        o_np, l_np = o_t.float().cpu().numpy(), l_t.cpu().numpy()
        for r in range(rd):
            s = oracle.ring_source(r, t, rd)
            qpos, kpos = oracle.zig(r, np.arange(Lr), c, rd), oracle.zig(s, np.arange(Lr), c, rd)
            for u in range(ud):
                o_ref, l_ref = oracle.attn_block(Q[r, u, :, 0], qpos, K[s, u, :, 0], V[s, u, :, 0], kpos, scale,
                                                 qseg=seg[qpos], kseg=seg[kpos])
                assert np.abs(o_np[r, u, :, 0] - o_ref).max() <= 2e-2
                both = np.isneginf(l_np[r, u, :, 0]) & np.isneginf(l_ref)
                assert np.array_equal(np.isneginf(l_np[r, u, :, 0]), np.isneginf(l_ref))
                d = np.abs(np.where(both, 0, l_np[r, u, :, 0]) - np.where(both, 0, l_ref))
                assert (d / np.maximum(np.abs(np.where(both, 0, l_ref)), 1)).max() <= 1e-3
    fo, fl = torch.empty_like(qh), torch.empty_like(acc_l)
    usp.usp_attn_fwd(qh, kh, vh, fo, fl, cu_seqlens=cud)
    usp.usp_check()
    assert (acc_o.float() - fo.float()).abs().max().item() <= 2e-2
    assert ((acc_l - fl).abs() / fl.abs().clamp_min(1.0)).max().item() <= 1e-3
