"""Pins of the oracle's backward (CPU only): the gradients of attention with respect to q, k, v.

  * torch autograd through a plain fp64 softmax attention (a library routine, differentiated by
    torch, not by the formulas the oracle writes out);
  * central finite differences of the oracle's own forward (the definition of a derivative);
  * invariants that hold at any size: the rows of dS sum to zero, so sum_j dk_j = 0; the rows of P
    sum to one, so sum_j dv_j = sum of dout over the group's query heads and rows;
  * the literal ring backward (rank by rank, Fig. 1 order, dk/dv partials returned to their owner)
    against the direct gradients on brute-force tiny inputs, for every split, GQA and K/V replication;
  * the replica sum is the adjoint of the replicating all-to-all (<A x, y> = <x, A^T y>).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from seeded_inputs import make_qkv


def torch_grads(q, k, v, dout, scale, causal):
    """fp64 autograd of softmax(scale q k^T + mask) v, GQA by repeat_interleave of the KV heads."""
    q, k, v, dout = (torch.as_tensor(np.asarray(x, dtype=np.float64)).clone() for x in (q, k, v, dout))
    q.requires_grad_(True)
    k.requires_grad_(True)
    v.requires_grad_(True)
    G = q.shape[2] // k.shape[2]
    qt, kt, vt = q.transpose(1, 2), k.repeat_interleave(G, 2).transpose(1, 2), v.repeat_interleave(G, 2).transpose(1, 2)
    s = scale * qt @ kt.transpose(-1, -2)
    if causal:
        L = s.shape[-1]
        s = s.masked_fill(torch.triu(torch.ones(L, L, dtype=torch.bool), 1), float("-inf"))
    out = (torch.softmax(s, -1) @ vt).transpose(1, 2)
    (out * dout).sum().backward()
    return q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


def _inputs(bs, L, hq, hkv, hd, seed):
    q, k, v = make_qkv(bs, L, hq, hkv, hd, "f32", seed=seed)
    g, _, _ = make_qkv(bs, L, hq, hkv, hd, "f32", seed=seed + 500)
    return q, k, v, g


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("bs,L,hq,hkv,hd", [(1, 24, 2, 2, 8), (2, 17, 4, 2, 5), (1, 32, 4, 1, 16)])
def test_bwd_matches_torch_autograd(causal, bs, L, hq, hkv, hd):
    q, k, v, g = _inputs(bs, L, hq, hkv, hd, seed=L + hq)
    scale = 1.0 / math.sqrt(hd)
    dq, dk, dv = oracle.attn_direct_bwd(q, k, v, g, scale=scale, causal=causal)
    tq, tk, tv = torch_grads(q, k, v, g, scale, causal)
    np.testing.assert_allclose(dq, tq, atol=1e-12, rtol=1e-10)
    np.testing.assert_allclose(dk, tk, atol=1e-12, rtol=1e-10)
    np.testing.assert_allclose(dv, tv, atol=1e-12, rtol=1e-10)


def test_bwd_matches_finite_differences():
    bs, L, hq, hkv, hd = 1, 6, 2, 1, 3
    q, k, v, g = (np.asarray(x, dtype=np.float64) for x in _inputs(bs, L, hq, hkv, hd, seed=3))
    scale = 0.7
    dq, dk, dv = oracle.attn_direct_bwd(q, k, v, g, scale=scale)

    def f(q_, k_, v_):
        o, _ = oracle.attn_direct(q_, k_, v_, scale=scale)
        return float((o * g).sum())

    eps = 1e-6
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args = {"q": (q, k, v), "k": (q, k, v), "v": (q, k, v)}[name]
            ap = [xp if a is x else a for a in args]
            am = [xm if a is x else a for a in args]
            num[idx] = (f(*ap) - f(*am)) / (2 * eps)
        np.testing.assert_allclose(grad, num, atol=1e-8, err_msg=name)


def test_bwd_restricted_rows_equal_full():
    q, k, v, g = _inputs(2, 40, 4, 2, 8, seed=11)
    dq, dk, dv = oracle.attn_direct_bwd(q, k, v, g)
    rows = np.array([0, 5, 39, 17])
    dq_r, dk_t, dv_t = oracle.attn_direct_bwd(q, k, v, g, q_rows=rows, kv_from=30)
    assert np.array_equal(dq_r, dq[:, rows])
    assert np.array_equal(dk_t, dk[:, 30:]) and np.array_equal(dv_t, dv[:, 30:])
    _, dk_n, _ = oracle.attn_direct_bwd(q, k, v, g, q_rows=[], kv_from=40)
    assert dk_n.shape == (2, 0, 2, 8)
    # non-causal tail still needs every query row
    dq_f, dk_f, _ = oracle.attn_direct_bwd(q, k, v, g, causal=False)
    _, dk_nt, _ = oracle.attn_direct_bwd(q, k, v, g, causal=False, q_rows=[], kv_from=25)
    assert np.array_equal(dk_nt, dk_f[:, 25:])


@pytest.mark.parametrize("causal", [True, False])
def test_bwd_invariants(causal):
    bs, L, hq, hkv, hd = 2, 48, 6, 2, 8
    q, k, v, g = _inputs(bs, L, hq, hkv, hd, seed=21)
    dq, dk, dv = oracle.attn_direct_bwd(q, k, v, g, causal=causal)
    np.testing.assert_allclose(dk.sum(axis=1), 0, atol=1e-12)
    G = hq // hkv
    gsum = np.asarray(g, dtype=np.float64).reshape(bs, L, hkv, G, hd).sum(axis=(1, 3))
    np.testing.assert_allclose(dv.sum(axis=1), gsum, atol=1e-11)
    # the gradient of the row sum of out w.r.t. v is the column sum of P: dout = 1 gives sum_j dv_j = L * G
    ones = torch.ones_like(g)
    _, _, dv1 = oracle.attn_direct_bwd(q, k, v, ones, causal=causal)
    np.testing.assert_allclose(dv1.sum(axis=1), L * G, rtol=1e-12)


def test_row0_only_sees_key0():
    """Causal: key 0 is the only key of query 0, so P_00 = 1, dS_00 = 0 and dq_0 = 0; the last key
    is seen by the last query only, so dv_{L-1} = sum_h P_{L-1,L-1} dout_{L-1,h}."""
    q, k, v, g = _inputs(1, 12, 2, 1, 4, seed=5)
    dq, dk, dv = oracle.attn_direct_bwd(q, k, v, g)
    np.testing.assert_allclose(dq[0, 0], 0, atol=1e-15)
    qa, ka, ga = (np.asarray(x, dtype=np.float64) for x in (q, k, g))
    s = 0.5 * qa[0, 11] @ ka[0, :, 0].T            # scale 1/sqrt(4), query 11 vs all keys, both heads
    p_last = np.exp(s[:, 11] - np.log(np.exp(s).sum(axis=1)))
    np.testing.assert_allclose(dv[0, 11, 0], (p_last[:, None] * ga[0, 11]).sum(axis=0), atol=1e-14)


CASES = [(L, rd, ud, hq, hkv, split) for (L, rd, ud, hq, hkv) in
         [(16, 2, 1, 2, 2), (16, 2, 2, 4, 2), (24, 3, 2, 4, 2), (32, 4, 2, 8, 2), (16, 1, 2, 2, 1),
          (16, 2, 4, 4, 1), (32, 2, 4, 8, 2), (24, 2, 1, 3, 1), (32, 4, 1, 2, 2)]
         for split in ("zigzag", "basic", "stripe")]


@pytest.mark.parametrize("L,rd,ud,hq,hkv,split", CASES)
def test_literal_ring_bwd_equals_direct(L, rd, ud, hq, hkv, split):
    q, k, v, g = _inputs(1, L, hq, hkv, 4, seed=L + 7 * rd + 13 * ud + hkv)
    dq, dk, dv = oracle.attn_direct_bwd(q, k, v, g)
    lq, lk, lv = oracle.literal_pipeline_bwd(q, k, v, g, rd, ud, split=split)
    np.testing.assert_allclose(lq, dq, atol=1e-12)
    np.testing.assert_allclose(lk, dk, atol=1e-12)
    np.testing.assert_allclose(lv, dv, atol=1e-12)


def test_literal_ring_bwd_noncausal_batch():
    q, k, v, g = _inputs(2, 24, 4, 2, 4, seed=77)
    dq, dk, dv = oracle.attn_direct_bwd(q, k, v, g, causal=False)
    lq, lk, lv = oracle.literal_pipeline_bwd(q, k, v, g, 3, 2, causal=False)
    for a, b in ((lq, dq), (lk, dk), (lv, dv)):
        np.testing.assert_allclose(a, b, atol=1e-12)


@pytest.mark.parametrize("ud,H", [(4, 1), (4, 2), (2, 2), (8, 2)])
def test_replica_sum_is_adjoint_of_replicating_a2a(ud, H):
    rng = np.random.default_rng(ud * 10 + H)
    rd, bs, Lu = 2, 2, 3
    x = rng.standard_normal((rd, ud, bs, Lu, H, 2))
    ax = oracle.a2a_fwd(x, ud)
    y = rng.standard_normal(ax.shape)
    assert np.isclose((ax * y).sum(), (x * oracle.a2a_inv_sum(y, ud, H)).sum(), rtol=1e-12)
