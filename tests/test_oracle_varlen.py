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
