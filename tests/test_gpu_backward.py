"""The backward pass through the C ABI: the row term D, the replica-summing inverse all-to-all, the
ring backward on head-sharded buffers, the one-call backward in natural order and the autograd
wrapper, against the oracle's gradients (fp64 on the same inputs).

Tolerance: gradients are compared as max|g - g_ref| / max(max|g_ref|, 1); 2e-2 for bf16 inputs and
outputs (the forward's out tolerance; bf16 rounding of the inputs and of each gradient is 2^-9
relative, fp32 accumulation), 2e-4 for fp32."""
import numpy as np
import pytest
import torch

import oracle
import sequence_long_context_zigzag_gb300 as usp
from seeded_inputs import make_qkv

pytestmark = pytest.mark.gpu


def rel_err(g, ref):
    g = g.float().cpu().numpy() if isinstance(g, torch.Tensor) else np.asarray(g)
    return np.abs(g - ref).max() / max(np.abs(ref).max(), 1.0)


def tol(dt):
    return 2e-2 if dt == "bf16" else 2e-4


def _inputs(L, hq, hkv, hd, dt, seed):
    q, k, v = make_qkv(1, L, hq, hkv, hd, dt, seed=seed)
    g, _, _ = make_qkv(1, L, hq, hkv, hd, dt, seed=seed + 500)
    return q, k, v, g


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_delta_is_row_dot(dt):
    _, _, _, g = _inputs(256, 4, 4, 128, dt, seed=1)
    o, _, _, _ = _inputs(256, 4, 4, 128, dt, seed=2)
    delta = torch.empty(1, 256, 4, device="cuda")
    usp.usp_attn_bwd_delta(o.cuda(), g.cuda(), delta)
    usp.usp_check()
    ref = np.einsum("blhd,blhd->blh", o.double().numpy(), g.double().numpy())
    assert np.abs(delta.cpu().numpy() - ref).max() <= 1e-4 * max(np.abs(ref).max(), 1)


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("L,H,ud,rd", [(512, 1, 4, 2), (480, 2, 4, 3), (1024, 2, 8, 2)])
def test_inverse_a2a_sums_replicas(dt, L, H, ud, rd):
    """Small integers make every sum exact in bf16 and fp32, so the result is compared bit for bit."""
    g = torch.Generator().manual_seed(L + H)
    Lr = L // rd
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    hs = torch.randint(-8, 9, (rd, ud, 1, 1, Lr, 64), generator=g).to(tdt)
    seq = torch.empty(rd, ud, 1, Lr // ud, H, 64, dtype=tdt, device="cuda")
    usp.usp_a2a4d(hs.cuda(), seq, rd, ud, -1)
    nat = torch.empty(1, L, H, 64, dtype=tdt, device="cuda")
    usp.usp_extract_a2a([hs.cuda()], [nat], rd, ud, inverse=True)
    usp.usp_check()
    ref = oracle.a2a_inv_sum(hs.double().numpy(), ud, H)
    assert np.array_equal(seq.double().cpu().numpy(), ref)
    assert np.array_equal(nat.double().cpu().numpy(), oracle.extract_inverse(ref, L, rd, ud))


CASES = [
    (512, 4, 4, 128, 2, 2, "bf16", None),
    (768, 8, 2, 64, 2, 3, "bf16", None),       # GQA, ragged tiles
    (512, 8, 1, 128, 4, 2, "bf16", None),      # MQA: K/V replicated on 4 ranks, replica sum
    (1024, 8, 4, 128, 2, 2, "bf16", 2),        # head groups of 2 (one KV head each, replicated on 2 ranks)
    (256, 4, 2, 64, 1, 4, "f32", None),
    (384, 4, 4, 128, 2, 3, "f32", None),
]


@pytest.mark.parametrize("L,hq,hkv,hd,ud,rd,dt,chunk", CASES)
def test_backward_matches_oracle(L, hq, hkv, hd, ud, rd, dt, chunk):
    q, k, v, g = _inputs(L, hq, hkv, hd, dt, seed=L + hq * 3 + hkv)
    qd, kd, vd, gd = q.cuda(), k.cuda(), v.cuda(), g.cuda()
    out = torch.empty_like(qd)
    lse = torch.empty(1, L, hq, device="cuda")
    usp.usp_forward(qd, kd, vd, out, lse, ud, rd, head_chunk=chunk)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    usp.usp_backward(qd, kd, vd, out, lse, gd, dq, dk, dv, ud, rd, head_chunk=chunk)
    usp.usp_check()
    rq, rk, rv = oracle.attn_direct_bwd(q, k, v, g)
    errs = [rel_err(dq, rq), rel_err(dk, rk), rel_err(dv, rv)]
    print(f"L={L} hq={hq} hkv={hkv} ud={ud} rd={rd} {dt}: rel err dq {errs[0]:.2e} dk {errs[1]:.2e} dv {errs[2]:.2e}")
    assert max(errs) <= tol(dt)


@pytest.mark.parametrize("split", ["basic", "stripe"])
def test_backward_other_splits(split):
    L, hq, hkv, hd, ud, rd = 512, 4, 2, 128, 2, 4
    q, k, v, g = _inputs(L, hq, hkv, hd, "bf16", seed=9)
    qd, kd, vd, gd = q.cuda(), k.cuda(), v.cuda(), g.cuda()
    out = torch.empty_like(qd)
    lse = torch.empty(1, L, hq, device="cuda")
    usp.usp_forward(qd, kd, vd, out, lse, ud, rd, split=split)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    usp.usp_backward(qd, kd, vd, out, lse, gd, dq, dk, dv, ud, rd, split=split)
    usp.usp_check()
    rq, rk, rv = oracle.attn_direct_bwd(q, k, v, g)
    assert max(rel_err(dq, rq), rel_err(dk, rk), rel_err(dv, rv)) <= 2e-2


def test_head_sharded_backward_matches_mapped_oracle():
    """usp_attn_bwd on head-sharded buffers equals the oracle's gradients moved by the same maps."""
    L, hq, hkv, hd, ud, rd = 512, 4, 2, 64, 2, 2
    q, k, v, g = _inputs(L, hq, hkv, hd, "f32", seed=31)
    Lr = L // rd
    sh = lambda H: torch.empty(rd, ud, H // ud, 1, Lr, hd, device="cuda")  # noqa: E731
    qh, kh, vh, gh = sh(hq), sh(hkv), sh(hkv), sh(hq)
    usp.usp_extract_a2a([q.cuda(), k.cuda(), v.cuda(), g.cuda()], [qh, kh, vh, gh], rd, ud)
    o_ref, l_ref = oracle.attn_direct(q, k, v)
    oh = torch.empty_like(qh)
    lh = torch.empty(qh.shape[:5], device="cuda")
    usp.usp_attn_fwd(qh, kh, vh, oh, lh)
    dh = torch.empty_like(lh)
    usp.usp_attn_bwd_delta(oh, gh, dh)
    dq, dk, dv = torch.empty_like(qh), torch.empty_like(kh), torch.empty_like(vh)
    usp.usp_attn_bwd(qh, kh, vh, gh, lh, dh, dq, dk, dv)
    usp.usp_check()
    rq, rk, rv = oracle.attn_direct_bwd(q, k, v, g)
    hs = lambda x: oracle.a2a_fwd(oracle.extract_local(x, rd, ud), ud)  # noqa: E731
    assert rel_err(dq, hs(rq)) <= 2e-4 and rel_err(dk, hs(rk)) <= 2e-4 and rel_err(dv, hs(rv)) <= 2e-4


def test_head_sharded_backward_bf16_replicated():
    """Tensor-core backward on head-sharded buffers with replicated K/V (MQA, ud = 4): each replica
    carries its own rank's share; summing the replicas (the inverse all-to-all) gives the oracle's."""
    L, hq, hkv, hd, ud, rd = 1024, 8, 1, 128, 4, 2
    q, k, v, g = _inputs(L, hq, hkv, hd, "bf16", seed=33)
    Lr = L // rd
    qh = torch.empty(rd, ud, hq // ud, 1, Lr, hd, device="cuda", dtype=torch.bfloat16)
    gh = torch.empty_like(qh)
    kh = torch.empty(rd, ud, 1, 1, Lr, hd, device="cuda", dtype=torch.bfloat16)
    vh = torch.empty_like(kh)
    usp.usp_extract_a2a([q.cuda(), k.cuda(), v.cuda(), g.cuda()], [qh, kh, vh, gh], rd, ud)
    oh = torch.empty_like(qh)
    lh = torch.empty(qh.shape[:5], device="cuda")
    usp.usp_attn_fwd(qh, kh, vh, oh, lh, hkv=hkv)
    dh = torch.empty_like(lh)
    usp.usp_attn_bwd_delta(oh, gh, dh)
    dq, dk, dv = torch.empty_like(qh), torch.empty_like(kh), torch.empty_like(vh)
    usp.usp_attn_bwd(qh, kh, vh, gh, lh, dh, dq, dk, dv, hkv=hkv)
    dk_n = torch.empty(1, L, hkv, hd, device="cuda", dtype=torch.bfloat16)
    dv_n = torch.empty_like(dk_n)
    usp.usp_extract_a2a([dk, dv], [dk_n, dv_n], rd, ud, inverse=True)
    usp.usp_check()
    rq, rk, rv = oracle.attn_direct_bwd(q, k, v, g)
    hs = lambda x: oracle.a2a_fwd(oracle.extract_local(x, rd, ud), ud)  # noqa: E731
    assert rel_err(dq, hs(rq)) <= 2e-2 and rel_err(dk_n, rk) <= 2e-2 and rel_err(dv_n, rv) <= 2e-2


def test_autograd_function():
    L, hq, hkv, hd, ud, rd = 512, 4, 2, 128, 2, 2
    q, k, v, g = _inputs(L, hq, hkv, hd, "bf16", seed=41)
    qd, kd, vd = (x.cuda().requires_grad_(True) for x in (q, k, v))
    out = usp.UspAttentionFunction.apply(qd, kd, vd, ud, rd)
    (out.float() * g.cuda().float()).sum().backward()
    usp.usp_check()
    rq, rk, rv = oracle.attn_direct_bwd(q, k, v, g)
    assert max(rel_err(qd.grad, rq), rel_err(kd.grad, rk), rel_err(vd.grad, rv)) <= 2e-2
    o_ref, _ = oracle.attn_direct(q, k, v)
    assert np.abs(out.detach().float().cpu().numpy() - o_ref).max() <= 2e-2


@pytest.mark.parametrize("L,hq,hkv,hd,ud,rd", [(4096, 8, 2, 128, 2, 4), (2000, 4, 4, 64, 1, 5), (3072, 8, 1, 128, 4, 3)])
def test_backward_many_tiles(L, hq, hkv, hd, ud, rd):
    """Several 128-key CTAs and 64-row tiles per block, ragged block ends (Lr = 400 at L = 2000),
    and the dk/dv kernel's walk over every ring rank's visible query tiles."""
    q, k, v, g = _inputs(L, hq, hkv, hd, "bf16", seed=L + rd)
    qd, kd, vd, gd = q.cuda(), k.cuda(), v.cuda(), g.cuda()
    out = torch.empty_like(qd)
    lse = torch.empty(1, L, hq, device="cuda")
    usp.usp_forward(qd, kd, vd, out, lse, ud, rd)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    usp.usp_backward(qd, kd, vd, out, lse, gd, dq, dk, dv, ud, rd)
    usp.usp_check()
    rq, rk, rv = oracle.attn_direct_bwd(q, k, v, g)
    errs = [rel_err(dq, rq), rel_err(dk, rk), rel_err(dv, rv)]
    print(f"L={L} hq={hq} hkv={hkv} hd={hd} ud={ud} rd={rd}: rel err dq {errs[0]:.2e} dk {errs[1]:.2e} dv {errs[2]:.2e}")
    assert max(errs) <= 2e-2


def test_backward_noncausal():
    L, hq, hkv, hd, ud, rd = 1024, 4, 2, 128, 2, 2
    q, k, v, g = _inputs(L, hq, hkv, hd, "bf16", seed=12)
    qd, kd, vd, gd = q.cuda(), k.cuda(), v.cuda(), g.cuda()
    out = torch.empty_like(qd)
    lse = torch.empty(1, L, hq, device="cuda")
    usp.usp_forward(qd, kd, vd, out, lse, ud, rd, causal=False)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    usp.usp_backward(qd, kd, vd, out, lse, gd, dq, dk, dv, ud, rd, causal=False)
    usp.usp_check()
    rq, rk, rv = oracle.attn_direct_bwd(q, k, v, g, causal=False)
    assert max(rel_err(dq, rq), rel_err(dk, rk), rel_err(dv, rv)) <= 2e-2


@pytest.mark.parametrize("wi", [1, 2])
def test_backward_full_size_sampled(wi):
    """At the workloads' full sizes: dq on seeded sampled rows (plus chunk-boundary rows) and dk, dv
    on the last 256 keys (seen only by the last queries, so the oracle stays cheap); and the
    invariants that hold at any size, sum_j dk_j = 0 and sum_j dv_j = sum of dout over the group."""
    from seeded_inputs import WORKLOADS, default_seed, make_rows, make_workload_qkv
    w = WORKLOADS[wi]
    seed = default_seed(wi)
    q, k, v = make_workload_qkv(w, seed)
    g, _, _ = make_qkv(w.bs, w.L, w.hq, w.hkv, w.hd, w.dtype, seed=seed + 500)
    qd, kd, vd, gd = q.cuda(), k.cuda(), v.cuda(), g.cuda()
    out = torch.empty_like(qd)
    lse = torch.empty(w.bs, w.L, w.hq, device="cuda")
    usp.usp_forward(qd, kd, vd, out, lse, w.ud, w.rd, head_chunk=w.head_chunk)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    usp.usp_backward(qd, kd, vd, out, lse, gd, dq, dk, dv, w.ud, w.rd, head_chunk=w.head_chunk)
    usp.usp_check()
    rows = np.array(make_rows(w.L, w.c, 128, seed))
    j0 = w.L - 256
    rq, rk, rv = oracle.attn_direct_bwd(q, k, v, g, q_rows=rows, kv_from=j0)
    e_q = rel_err(dq[:, torch.as_tensor(rows, device="cuda")], rq)
    e_k, e_v = rel_err(dk[:, j0:], rk), rel_err(dv[:, j0:], rv)
    print(f"{w.name}: dq rows {len(rows)} rel {e_q:.2e}; dk/dv tail rel {e_k:.2e} / {e_v:.2e}")
    assert max(e_q, e_k, e_v) <= 2e-2
    G = w.hq // w.hkv
    dk_sum = dk.double().sum(dim=1)
    assert dk_sum.abs().max().item() <= 2e-2 * max(dk.double().abs().sum(dim=1).max().item(), 1.0)
    dv_sum = dv.double().sum(dim=1)
    g_sum = gd.double().reshape(w.bs, w.L, w.hkv, G, w.hd).sum(dim=(1, 3))
    assert (dv_sum - g_sum).abs().max().item() <= 2e-2 * max(g_sum.abs().max().item(), 1.0) + 1e-2 * w.L ** 0.5
