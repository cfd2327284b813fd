"""Pins of the CPU oracle to things other than itself (CPU only).

Each pin is chosen so that a plausible slip in the oracle (a dropped term, a wrong sign, an
off-by-one in the causal mask, a transposed index in a permutation) fails at least one test:
  * library routines on the special cases they cover (torch SDPA and torch's CPU flash routine,
    which also returns the row log-sum-exp; torch.chunk / torch.cat for Algorithm 2 and
    AllToAll4D; plain transposes for the ud = 1 all-to-all);
  * closed forms (q = 0 gives lse = log(i + 1) and prefix means; row 0 gives o = v_0);
  * the pages' printed numbers (tests/golden/*.txt, each citing its figure or table);
  * brute force on tiny inputs (the literal rank-by-rank pipeline against direct attention).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from seeded_inputs import make_qkv

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, _, val = line.partition("=") if "=" in line else line.partition(":")
            vals[key.strip()] = val.strip()
    return vals


def torch_lib_attn(q, k, v, scale, causal):
    """Library reference: torch's CPU flash routine (out and natural-log lse), fp64.
    q (bs,L,hq,hd) -> out (bs,L,hq,hd), lse (bs,L,hq); GQA by repeat_interleave of KV heads."""
    q = torch.as_tensor(q, dtype=torch.float64).transpose(1, 2)
    k = torch.as_tensor(k, dtype=torch.float64).transpose(1, 2)
    v = torch.as_tensor(v, dtype=torch.float64).transpose(1, 2)
    G = q.shape[1] // k.shape[1]
    k = k.repeat_interleave(G, dim=1)
    v = v.repeat_interleave(G, dim=1)
    out, lse = torch.ops.aten._scaled_dot_product_flash_attention_for_cpu(q, k, v, 0.0, causal, scale=scale)
    return out.transpose(1, 2).numpy(), lse.transpose(1, 2).numpy()


# ---------------------------------------------------------------------------------------------
# direct attention
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("hq,hkv", [(2, 2), (4, 2), (4, 1)])
def test_direct_matches_library(causal, hq, hkv):
    q, k, v = make_qkv(2, 37, hq, hkv, 8, "f32", seed=3)
    q, k, v = q.double(), k.double(), v.double()
    scale = 0.3
    o, l = oracle.attn_direct(q, k, v, scale=scale, causal=causal)
    o_ref, l_ref = torch_lib_attn(q, k, v, scale, causal)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, l_ref, rtol=1e-13, atol=1e-13)


def test_direct_matches_sdpa_gqa():
    q, k, v = make_qkv(1, 50, 8, 2, 16, "f32", seed=4)
    q, k, v = q.double(), k.double(), v.double()
    o, _ = oracle.attn_direct(q, k, v, causal=True)
    ref = torch.nn.functional.scaled_dot_product_attention(
        q.transpose(1, 2), k.transpose(1, 2), v.transpose(1, 2), is_causal=True, enable_gqa=True)
    np.testing.assert_allclose(o, ref.transpose(1, 2).numpy(), atol=1e-12, rtol=0)


def test_direct_closed_form_zero_queries():
    """q = 0: every visible score is 0, so lse_i = log(i+1) and o_i is the mean of v_0..v_i."""
    L, hd = 23, 4
    _, k, v = make_qkv(1, L, 3, 3, hd, "f32", seed=5)
    q = torch.zeros(1, L, 3, hd)
    o, l = oracle.attn_direct(q, k, v, causal=True)
    i = np.arange(L)
    np.testing.assert_allclose(l[0], np.log(i + 1.0)[:, None].repeat(3, 1), atol=1e-14, rtol=0)
    prefix_mean = np.cumsum(v[0].double().numpy(), axis=0) / (i + 1.0)[:, None, None]
    np.testing.assert_allclose(o[0], prefix_mean, atol=1e-13, rtol=0)
    # non-causal: the mean over all L keys and lse = log L
    o, l = oracle.attn_direct(q, k, v, causal=False)
    np.testing.assert_allclose(l, math.log(L), atol=1e-14, rtol=0)
    np.testing.assert_allclose(o[0], np.broadcast_to(v[0].double().mean(0).numpy(), o[0].shape), atol=1e-13)


def test_direct_row0_and_identical_keys():
    """Row 0 sees only key 0 (o = v_0, lse = s_00); identical keys give equal weights."""
    L, hd, scale = 9, 8, 0.25
    q, k, v = make_qkv(1, L, 2, 2, hd, "f32", seed=6)
    o, l = oracle.attn_direct(q, k, v, scale=scale, causal=True)
    qd, kd, vd = q.double().numpy(), k.double().numpy(), v.double().numpy()
    np.testing.assert_allclose(o[0, 0], vd[0, 0], atol=1e-15)
    np.testing.assert_allclose(l[0, 0], scale * np.einsum("hd,hd->h", qd[0, 0], kd[0, 0]), atol=1e-14)
    kk = np.broadcast_to(kd[:, :1], kd.shape).copy()
    o, l = oracle.attn_direct(qd, kk, vd, scale=scale, causal=True)
    s = scale * np.einsum("lhd,hd->lh", qd[0], kd[0, 0])
    np.testing.assert_allclose(l[0], s + np.log(np.arange(L) + 1.0)[:, None], atol=1e-13)


def test_direct_widening_is_exact():
    """bf16 and fp32 inputs are widened exactly: same result as passing fp64 copies."""
    q, k, v = make_qkv(1, 40, 2, 1, 8, "bf16", seed=7)
    o1, l1 = oracle.attn_direct(q, k, v)
    o2, l2 = oracle.attn_direct(q.double(), k.double(), v.double())
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_direct_row_subset():
    q, k, v = make_qkv(1, 64, 2, 2, 8, "f32", seed=8)
    o, l = oracle.attn_direct(q, k, v)
    rows = [63, 0, 17, 40]
    o2, l2 = oracle.attn_direct(q, k, v, rows=rows)
    assert np.array_equal(o2, o[:, rows]) and np.array_equal(l2, l[:, rows])


# ---------------------------------------------------------------------------------------------
# LSE merge and blocks
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("nblocks", [2, 3, 5])
def test_merge_of_blocks_equals_direct(nblocks):
    """Context-Parallel page: merging the per-block (o_j, lse_j) equals one pass over all keys."""
    L, hd, scale = 48, 8, 0.35
    q, k, v = make_qkv(1, L, 4, 2, hd, "f32", seed=10 + nblocks)
    qd, kd, vd = (x.double().numpy()[0].transpose(1, 0, 2) for x in (q, k, v))   # (H, L, hd)
    pos = np.arange(L)
    o_ref, l_ref = oracle.attn_direct(q, k, v, scale=scale, causal=True)
    rng = np.random.default_rng(nblocks)
    perm = rng.permutation(L)                       # keys split into scattered blocks
    o_acc = np.zeros((4, L, hd))
    l_acc = np.full((4, L), -np.inf)
    for blk in np.array_split(perm, nblocks):
        o_b, l_b = oracle.attn_block(qd, pos, kd[:, blk], vd[:, blk], pos[blk], scale, causal=True)
        o_acc, l_acc = oracle.lse_merge(o_acc, l_acc, o_b, l_b)
    np.testing.assert_allclose(o_acc.transpose(1, 0, 2), o_ref[0], atol=1e-12, rtol=0)
    np.testing.assert_allclose(l_acc.T, l_ref[0], atol=1e-12, rtol=1e-12)


def test_merge_identities():
    rng = np.random.default_rng(0)
    o = rng.standard_normal((6, 5))
    l = rng.standard_normal(6) * 3
    # merging with an empty partial (-inf) returns the other operand exactly
    om, lm = oracle.lse_merge(o, l, np.zeros_like(o), np.full(6, -np.inf))
    assert np.array_equal(om, o) and np.array_equal(lm, l)
    om, lm = oracle.lse_merge(np.zeros_like(o), np.full(6, -np.inf), o, l)
    assert np.array_equal(om, o) and np.array_equal(lm, l)
    # two empty partials stay empty
    om, lm = oracle.lse_merge(np.zeros_like(o), np.full(6, -np.inf), np.zeros_like(o), np.full(6, -np.inf))
    assert np.all(om == 0) and np.all(np.isneginf(lm))
    # merge(x, x) = (o, lse + log 2)
    om, lm = oracle.lse_merge(o, l, o, l)
    np.testing.assert_allclose(om, o, atol=1e-15)
    np.testing.assert_allclose(lm, l + math.log(2), atol=1e-14)
    # weights e^(l1-lse) and e^(l2-lse) sum to 1: merging o1 = o2 = 1 gives 1
    l2 = rng.standard_normal(6) * 3
    om, lm = oracle.lse_merge(np.ones((6, 5)), l, np.ones((6, 5)), l2)
    np.testing.assert_allclose(om, 1.0, atol=1e-14)
    np.testing.assert_allclose(lm, np.log(np.exp(l) + np.exp(l2)), atol=1e-13)
    # very different magnitudes do not overflow
    om, lm = oracle.lse_merge(o, l + 800.0, o * 2, l - 800.0)
    np.testing.assert_allclose(om, o, atol=1e-15)
    np.testing.assert_allclose(lm, l + 800.0, atol=1e-12)


def test_block_empty_rows():
    """A block whose keys all lie after the queries yields (0, -inf) for every row."""
    q = np.ones((1, 3, 4))
    k = np.ones((1, 2, 4))
    o, l = oracle.attn_block(q, [0, 1, 2], k, k, [5, 6], 1.0, causal=True)
    assert np.all(o == 0) and np.all(np.isneginf(l))


# ---------------------------------------------------------------------------------------------
# index maps
# ---------------------------------------------------------------------------------------------
def alg2_with_torch(x, r, u, rd, ud):
    """Algorithm 2 literally with torch.chunk / torch.cat on the sequence dimension (dim 1)."""
    chunks = torch.as_tensor(x).chunk(2 * rd, dim=1)
    reorder = torch.cat([chunks[r], chunks[2 * rd - r - 1]], dim=1)
    return reorder.chunk(ud, dim=1)[u]


@pytest.mark.parametrize("rd,ud,L", [(1, 1, 8), (2, 1, 16), (4, 2, 32), (2, 4, 48), (8, 1, 64), (3, 2, 36)])
def test_extract_matches_algorithm2(rd, ud, L):
    x = np.arange(2 * L * 4 * 3, dtype=np.int64).reshape(2, L, 4, 3)
    loc = oracle.extract_local(x, rd, ud)
    assert loc.shape == (rd, ud, 2, L // (rd * ud), 4, 3)
    for r in range(rd):
        for u in range(ud):
            assert np.array_equal(loc[r, u], alg2_with_torch(x, r, u, rd, ud).numpy())
    assert np.array_equal(oracle.extract_inverse(loc, L, rd, ud), x)
    # a bijection: every element appears exactly once
    assert np.array_equal(np.sort(loc.ravel()), np.arange(x.size))


def test_extract_head_window_and_identity():
    x = np.arange(1 * 16 * 6 * 2).reshape(1, 16, 6, 2)
    loc = oracle.extract_local(x, 2, 2, h0=2, H=3)
    assert np.array_equal(loc, oracle.extract_local(x[:, :, 2:5], 2, 2))
    ident = oracle.extract_local(x, 1, 1)
    assert np.array_equal(ident[0, 0], x)


def a2a_with_torch(loc, ud):
    """AllToAll4D per destination Ulysses rank u': concatenate over source ranks u (ascending) the
    head slice u' of every rank's (bs, Lu, H, hd) tensor along the sequence, then lay it out as
    (H/ud, bs, Lr, hd) (the head-major shape the USP review prints)."""
    rd, _, bs, Lu, H, hd = loc.shape
    Hl = H // ud
    out = []
    for r in range(rd):
        row = []
        for up in range(ud):
            parts = [torch.as_tensor(loc[r, u])[:, :, up * Hl:(up + 1) * Hl] for u in range(ud)]
            row.append(torch.cat(parts, dim=1).permute(2, 0, 1, 3).numpy())
        out.append(row)
    return np.array(out)


@pytest.mark.parametrize("rd,ud,H", [(1, 1, 2), (2, 2, 4), (1, 4, 8), (4, 2, 2), (2, 3, 6)])
def test_a2a_matches_library_and_inverts(rd, ud, H):
    L = 2 * rd * ud * 3
    x = np.arange(2 * L * H * 5).reshape(2, L, H, 5)
    loc = oracle.extract_local(x, rd, ud)
    hs = oracle.a2a_fwd(loc, ud)
    assert hs.shape == (rd, ud, H // ud, 2, L // rd, 5)
    assert np.array_equal(hs, a2a_with_torch(loc, ud))
    assert np.array_equal(oracle.a2a_inv(hs, ud), loc)
    assert np.array_equal(np.sort(hs.ravel()), np.arange(x.size))


def test_a2a_ud1_is_transpose():
    loc = np.arange(3 * 1 * 2 * 5 * 4 * 2).reshape(3, 1, 2, 5, 4, 2)
    hs = oracle.a2a_fwd(loc, 1)
    assert np.array_equal(hs[:, 0], loc[:, 0].transpose(0, 3, 1, 2, 4))


@pytest.mark.parametrize("rd,ud,H", [(2, 4, 1), (1, 4, 2), (2, 2, 1), (3, 8, 2)])
def test_a2a_replicates_when_fewer_heads_than_ranks(rd, ud, H):
    """hkv < ud: rank u' of every Ulysses group receives head u' // (ud/H) for the whole ring-local
    sequence, i.e. exactly what the ud = 1 split gives for that head (an independent map)."""
    L = 2 * rd * ud * 2
    x = np.arange(2 * L * H * 3).reshape(2, L, H, 3)
    hs = oracle.a2a_fwd(oracle.extract_local(x, rd, ud), ud)
    assert hs.shape == (rd, ud, 1, 2, L // rd, 3)
    rep = ud // H
    for h in range(H):
        ring_local = oracle.extract_local(x, rd, 1, h0=h, H=1)       # [rd][1][bs][Lr][1][3]
        for u in range(h * rep, (h + 1) * rep):
            assert np.array_equal(hs[:, u, 0], ring_local[:, 0, :, :, 0])
    # every element of x shows up exactly rep times
    counts = np.bincount(hs.ravel(), minlength=x.size)
    assert np.all(counts == rep)


def test_lse_as_rows_of_one():
    """lse is permuted as a tensor whose rows hold one value: same maps with a trailing axis of 1."""
    hs = np.arange(2 * 2 * 3 * 1 * 8).reshape(2, 2, 3, 1, 8).astype(float)
    a = oracle.a2a_inv(hs[..., None], 2)[..., 0]
    b = oracle.a2a_inv(hs, 2)
    assert np.array_equal(a, b)


# ---------------------------------------------------------------------------------------------
# the literal pipeline against direct attention (brute force on tiny inputs)
# ---------------------------------------------------------------------------------------------
CASES = [(L, hd, rd, ud, G) for L in (8, 16, 32) for hd in (4, 8) for rd in (1, 2, 4) for ud in (1, 2)
         for G in (1, 2) if L % (2 * rd) == 0 and (L // rd) % ud == 0]


@pytest.mark.parametrize("L,hd,rd,ud,G", CASES)
def test_literal_pipeline_equals_direct(L, hd, rd, ud, G):
    hkv = 2
    hq = hkv * G
    q, k, v = make_qkv(1, L, hq, hkv, hd, "f32", seed=L * 100 + hd * 10 + rd + ud + G)
    o_ref, l_ref = oracle.attn_direct(q, k, v, causal=True)
    o, l = oracle.literal_pipeline(q, k, v, rd, ud)
    np.testing.assert_allclose(o, o_ref, atol=1e-12, rtol=0)
    np.testing.assert_allclose(l, l_ref, atol=1e-12, rtol=1e-12)


@pytest.mark.parametrize("L,rd,ud,hq,hkv", [(16, 2, 4, 4, 1), (16, 2, 4, 8, 2), (16, 1, 4, 4, 1),
                                              (24, 3, 2, 2, 1), (32, 2, 8, 8, 2), (32, 4, 2, 4, 1)])
def test_literal_pipeline_kv_replication_equals_direct(L, rd, ud, hq, hkv):
    """MQA / GQA with ud > hkv: the replicated K/V all-to-all still gives plain causal attention
    (checked against torch's CPU flash routine as well)."""
    q, k, v = make_qkv(1, L, hq, hkv, 4, "f32", seed=L + rd * 10 + ud * 100 + hkv)
    o_ref, l_ref = oracle.attn_direct(q, k, v, causal=True)
    o, l = oracle.literal_pipeline(q, k, v, rd, ud)
    np.testing.assert_allclose(o, o_ref, atol=1e-12, rtol=0)
    np.testing.assert_allclose(l, l_ref, atol=1e-12, rtol=1e-12)
    o_lib, l_lib = torch_lib_attn(q, k, v, 0.5, True)
    np.testing.assert_allclose(o, o_lib, atol=1e-10)
    np.testing.assert_allclose(l, l_lib, atol=1e-10)


def test_literal_pipeline_rejects_uneven_kv_heads():
    q, k, v = make_qkv(1, 16, 6, 3, 4, "f32", seed=5)
    with pytest.raises(ValueError):
        oracle.literal_pipeline(q, k, v, 2, 2)


def test_literal_pipeline_noncausal_and_batch():
    q, k, v = make_qkv(2, 24, 4, 2, 4, "f32", seed=99)
    o_ref, l_ref = oracle.attn_direct(q, k, v, causal=False)
    o, l = oracle.literal_pipeline(q, k, v, 3, 2, causal=False)
    np.testing.assert_allclose(o, o_ref, atol=1e-12)
    np.testing.assert_allclose(l, l_ref, atol=1e-12)


# ---------------------------------------------------------------------------------------------
# the pages' numbers
# ---------------------------------------------------------------------------------------------
def test_ring_schedule_matches_fig1():
    g = read_golden("ring_schedule_cp4.txt")
    table = oracle.ring_schedule(4)
    for step in range(4):
        assert table[step] == [int(t) for t in g[str(step + 1)].split()]


def test_zigzag_balance_matches_fig2():
    g = read_golden("zigzag_balance_cp4.txt")
    assert oracle.zigzag_rank_work(4) == [float(x) for x in g["zigzag"].split()]
    cont = oracle.contiguous_rank_work(4)
    assert cont == [float(x) for x in g["contiguous"].split()]
    assert max(cont) / (sum(cont) / 4) == float(g["contiguous_max_over_mean"])
    assert max(cont) / min(cont) == float(g["contiguous_max_over_min"])
    for a, owner, w in oracle.zigzag_chunk_work(4):
        exp_owner, exp_w = g[f"chunk{a}"].split()
        assert owner == int(exp_owner) and w == float(exp_w)


@pytest.mark.parametrize("rd", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("c", [1, 4, 7])
def test_zigzag_exact_pairs_equal(rd, c):
    """Brute-force pair counts per rank: zigzag gives c^2 (2rd-1) + c (c+1) on every rank;
    the general block count is 2*rd small blocks per rank."""
    counts = [oracle.visible_pairs(oracle.zig(r, np.arange(2 * c), c, rd)) for r in range(rd)]
    assert counts == [c * c * (2 * rd - 1) + c * (c + 1)] * rd
    if c > 1:   # a 1 x 1 diagonal block is fully visible, so the half-block convention needs c > 1
        assert oracle.zigzag_rank_work(rd, c) == [2.0 * rd] * rd


def test_comm_volumes_hand_example():
    g = read_golden("comm_volume_hand_example.txt")
    s, h, cp, eb = (int(g[k]) for k in ("s_tokens", "hidden", "cp", "bytes_per_elem"))
    hkv = int(g["gqa_hkv_hidden"])
    MiB = 2 ** 20
    assert oracle.comm_ring_elems(s, h, cp) * eb / MiB == int(g["mha_ring_mib"])
    assert oracle.comm_ulysses_elems(s, h, h, cp) * eb / MiB == int(g["mha_ulysses_mib"])
    assert oracle.comm_ring_elems(s, hkv, cp) * eb / MiB == int(g["gqa_ring_mib"])
    assert oracle.comm_ulysses_elems(s, h, hkv, cp) * eb / MiB == int(g["gqa_ulysses_mib"])


def test_comm_volumes_counted_from_schedule():
    """Counting the bytes the virtual schedule moves off-rank reproduces the closed forms."""
    s, cp, hd = 131072, 8, 128
    for heads, heads_kv in ((32, 32), (32, 8)):
        h, hkv = heads * hd, heads_kv * hd
        assert oracle.counted_ring_elems(s, heads_kv, hd, cp) == oracle.comm_ring_elems(s, hkv, cp)
        assert oracle.counted_ulysses_elems(s, heads, heads_kv, hd, cp) == \
            oracle.comm_ulysses_elems(s, h, hkv, cp)


# ---------------------------------------------------------------------------------------------
# other sequence splits (the plain ring's contiguous split, Striped Attention's round robin)
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("rd,ud,L", [(2, 1, 16), (4, 2, 32), (3, 2, 36), (1, 1, 8)])
def test_basic_and_stripe_splits_match_library(rd, ud, L):
    x = np.arange(2 * L * 3 * 2).reshape(2, L, 3, 2)
    xt = torch.as_tensor(x)
    for r in range(rd):
        basic = xt.chunk(rd, dim=1)[r]              # contiguous: rank r holds its L/rd block
        stripe = xt[:, r::rd]                       # round robin: tokens r, r + rd, ...
        for u in range(ud):
            assert np.array_equal(oracle.extract_local(x, rd, ud, split="basic")[r, u],
                                  basic.chunk(ud, dim=1)[u].numpy())
            assert np.array_equal(oracle.extract_local(x, rd, ud, split="stripe")[r, u],
                                  stripe.chunk(ud, dim=1)[u].numpy())
    for split in oracle.SPLITS:
        loc = oracle.extract_local(x, rd, ud, split=split)
        assert np.array_equal(oracle.extract_inverse(loc, L, rd, ud, split=split), x)


@pytest.mark.parametrize("split", ["basic", "stripe"])
@pytest.mark.parametrize("L,rd,ud", [(16, 2, 1), (32, 4, 2), (24, 3, 2)])
def test_literal_pipeline_other_splits_equal_direct(split, L, rd, ud):
    q, k, v = make_qkv(1, L, 4, 2, 8, "f32", seed=L + rd + ud)
    o_ref, l_ref = oracle.attn_direct(q, k, v, causal=True)
    o, l = oracle.literal_pipeline(q, k, v, rd, ud, split=split)
    np.testing.assert_allclose(o, o_ref, atol=1e-12)
    np.testing.assert_allclose(l, l_ref, atol=1e-12)


@pytest.mark.parametrize("rd,Lr", [(4, 16), (8, 32), (3, 10)])
def test_split_rank_pairs_closed_forms(rd, Lr):
    """Causal pairs per rank: basic r*Lr^2 + Lr(Lr+1)/2 (grows with r, max/mean -> 1.75 at rd = 4 for
    long blocks, the Context-Parallel page's figure); stripe rd*Lr(Lr-1)/2 + (r+1)*Lr (nearly equal);
    zigzag identical on every rank."""
    L = rd * Lr
    basic = oracle.split_rank_pairs("basic", L, rd)
    stripe = oracle.split_rank_pairs("stripe", L, rd)
    assert basic == [r * Lr * Lr + Lr * (Lr + 1) // 2 for r in range(rd)]
    assert stripe == [rd * Lr * (Lr - 1) // 2 + (r + 1) * Lr for r in range(rd)]
    if Lr % 2 == 0:
        zz = oracle.split_rank_pairs("zigzag", L, rd)
        assert len(set(zz)) == 1 and sum(zz) == sum(basic) == L * (L + 1) // 2
    if rd == 4:
        big = oracle.split_rank_pairs("basic", 4 * 4096, 4)
        assert abs(max(big) / (sum(big) / 4) - 1.75) < 1e-3
