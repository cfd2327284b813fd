"""Pins of the oracle's packed-sequence (varlen) attention (CPU only): several samples concatenated
into one sequence, each attending only within itself (the sequence packing that motivates ByteScale
on the Context-Parallel page).

  * packed attention equals the samples attended one by one (slicing and separate calls -- an
    independent computation) and concatenated;
  * the literal rank-by-rank pipeline with the per-sample mask equals it, for every split, with
    samples that straddle zigzag chunk and rank boundaries and samples of one token;
  * one sample spanning the sequence is plain causal attention.
"""
import numpy as np
import pytest

import oracle
from seeded_inputs import make_qkv


def by_parts(q, k, v, cu, causal=True):
    outs, lses = [], []
    for a, b in zip(cu[:-1], cu[1:]):
        o, l = oracle.attn_direct(q[:, a:b], k[:, a:b], v[:, a:b], causal=causal, scale=0.5)
        outs.append(o)
        lses.append(l)
    return np.concatenate(outs, 1), np.concatenate(lses, 1)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("cu", [[0, 10, 30, 48], [0, 1, 2, 47, 48], [0, 48], [0, 16, 32, 48], [0, 5, 6, 40, 48]])
def test_packed_equals_samples_one_by_one(causal, cu):
    q, k, v = make_qkv(2, 48, 4, 2, 4, "f32", seed=len(cu) + 7 * causal)
    o, l = oracle.attn_direct(q, k, v, causal=causal, scale=0.5, cu_seqlens=cu)
    ro, rl = by_parts(q, k, v, cu, causal)
    np.testing.assert_allclose(o, ro, atol=1e-13)
    np.testing.assert_allclose(l, rl, atol=1e-13)


def test_single_sample_is_plain_attention():
    q, k, v = make_qkv(1, 32, 2, 2, 4, "f32", seed=2)
    o, l = oracle.attn_direct(q, k, v, cu_seqlens=[0, 32])
    ro, rl = oracle.attn_direct(q, k, v)
    assert np.array_equal(o, ro) and np.array_equal(l, rl)


@pytest.mark.parametrize("split", ["zigzag", "basic", "stripe"])
@pytest.mark.parametrize("L,rd,ud,cu", [(48, 3, 2, [0, 7, 20, 21, 48]), (64, 4, 2, [0, 32, 64]),
                                        (64, 2, 4, [0, 3, 50, 64]), (32, 4, 1, [0, 1, 2, 3, 31, 32])])
def test_literal_pipeline_packed_equals_direct(split, L, rd, ud, cu):
    q, k, v = make_qkv(1, L, 4, 2, 4, "f32", seed=L + rd + len(cu))
    ro, rl = oracle.attn_direct(q, k, v, cu_seqlens=cu)
    o, l = oracle.literal_pipeline(q, k, v, rd, ud, split=split, cu_seqlens=cu)
    np.testing.assert_allclose(o, ro, atol=1e-12)
    np.testing.assert_allclose(l, rl, atol=1e-12)


@pytest.mark.parametrize("cu", [[0, 10, 40], [1, 48], [0, 20, 10, 48], [0, 48, 48]])
def test_bad_cu_seqlens(cu):
    q, k, v = make_qkv(1, 48, 2, 2, 4, "f32", seed=1)
    with pytest.raises(ValueError):
        oracle.attn_direct(q, k, v, cu_seqlens=cu)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("cu", [[0, 10, 30, 48], [0, 1, 2, 47, 48], [0, 48]])
def test_packed_grads_equal_samples_one_by_one(causal, cu):
    q, k, v = make_qkv(1, 48, 4, 2, 4, "f32", seed=11 + len(cu))
    g, _, _ = make_qkv(1, 48, 4, 2, 4, "f32", seed=99)
    dq, dk, dv = oracle.attn_direct_bwd(q, k, v, g, scale=0.5, causal=causal, cu_seqlens=cu)
    parts = [oracle.attn_direct_bwd(q[:, a:b], k[:, a:b], v[:, a:b], g[:, a:b], scale=0.5, causal=causal)
             for a, b in zip(cu[:-1], cu[1:])]
    for got, i in ((dq, 0), (dk, 1), (dv, 2)):
        np.testing.assert_allclose(got, np.concatenate([p[i] for p in parts], 1), atol=1e-13)
    # restricted rows agree with the full call
    rows = np.array([0, 9, 10, 47])
    dq_r, dk_t, _ = oracle.attn_direct_bwd(q, k, v, g, scale=0.5, causal=causal, cu_seqlens=cu, q_rows=rows,
                                           kv_from=40)
    assert np.array_equal(dq_r, dq[:, rows]) and np.array_equal(dk_t, dk[:, 40:])


@pytest.mark.parametrize("split", ["zigzag", "basic", "stripe"])
@pytest.mark.parametrize("L,rd,ud,hkv,cu", [(48, 3, 2, 2, [0, 7, 20, 21, 48]), (32, 2, 4, 1, [0, 3, 30, 32])])
def test_literal_ring_bwd_packed_equals_direct(split, L, rd, ud, hkv, cu):
    q, k, v = make_qkv(1, L, 4, hkv, 4, "f32", seed=L + rd)
    g, _, _ = make_qkv(1, L, 4, hkv, 4, "f32", seed=L + rd + 500)
    dq, dk, dv = oracle.attn_direct_bwd(q, k, v, g, cu_seqlens=cu)
    lq, lk, lv = oracle.literal_pipeline_bwd(q, k, v, g, rd, ud, split=split, cu_seqlens=cu)
    for a, b in ((lq, dq), (lk, dk), (lv, dv)):
        np.testing.assert_allclose(a, b, atol=1e-12)
