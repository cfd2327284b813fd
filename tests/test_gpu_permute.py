"""GPU parity of the permutes (zigzag split, AllToAll4D and their inverses): bit-exact against the
oracle's index maps, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import sequence_long_context_zigzag_gb300 as usp
from seeded_inputs import WORKLOADS

pytestmark = pytest.mark.gpu
DEV = "cuda"


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw bit patterns of a tensor as an integer numpy array (bit-exact comparisons)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy()
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy()
    raise TypeError(t.dtype)


def rand(shape, dtype, seed):
    g = torch.Generator("cpu").manual_seed(seed)
    return torch.randn(*shape, generator=g).to(dtype)


CASES = [  # bs, L, H, hd, dtype, rd, ud
    (1, 64, 4, 128, torch.bfloat16, 2, 2),
    (2, 1000, 4, 128, torch.bfloat16, 4, 2),   # c = 125, Lu = 125: nothing aligned to 128
    (1, 768, 6, 64, torch.bfloat16, 3, 2),
    (1, 1024, 4, 64, torch.float32, 4, 1),
    (2, 96, 8, 128, torch.float32, 1, 4),
    (1, 240, 4, 96, torch.bfloat16, 5, 2),     # 192-byte rows: 12 vectors per row
    (1, 128, 4, 1, torch.float32, 2, 2),       # lse-like 4-byte rows
    (3, 48, 2, 8, torch.float32, 2, 1),        # 32-byte rows
]


@pytest.mark.parametrize("bs,L,H,hd,dtype,rd,ud", CASES)
def test_extract_and_inverse_bitexact(bs, L, H, hd, dtype, rd, ud):
    shape = (bs, L, H) if hd == 1 else (bs, L, H, hd)
    x = rand(shape, dtype, seed=L + H + hd)
    xd = x.to(DEV)
    Lu = L // (rd * ud)
    loc = torch.empty((rd, ud, bs, Lu, H) + (() if hd == 1 else (hd,)), dtype=dtype, device=DEV)
    usp.usp_extract_local(xd, loc, rd, ud)
    assert np.array_equal(bits(loc), oracle.extract_local(bits(x), rd, ud))
    back = torch.full_like(xd, float("nan"))
    usp.usp_extract_local(loc, back, rd, ud, inverse=True)
    assert np.array_equal(bits(back), bits(x))
    # one virtual rank at a time, as the pages' per-rank extract call does
    ref = oracle.extract_local(bits(x), rd, ud)
    for vr in range(rd * ud):
        one = torch.empty(loc.shape[2:], dtype=dtype, device=DEV)
        usp.usp_extract_local(xd, one, rd, ud, vr=vr)
        assert np.array_equal(bits(one), ref[vr // ud, vr % ud])
    usp.usp_check()


@pytest.mark.parametrize("bs,L,H,hd,dtype,rd,ud", CASES)
def test_a2a_and_inverse_bitexact(bs, L, H, hd, dtype, rd, ud):
    Lu, Lr = L // (rd * ud), L // rd
    tail = () if hd == 1 else (hd,)
    loc = rand((rd, ud, bs, Lu, H) + tail, dtype, seed=7 * L + H)
    locd = loc.to(DEV)
    hs = torch.empty((rd, ud, H // ud, bs, Lr) + tail, dtype=dtype, device=DEV)
    usp.usp_a2a4d(locd, hs, rd, ud, 1)
    assert np.array_equal(bits(hs), oracle.a2a_fwd(bits(loc), ud))
    back = torch.full_like(locd, float("nan"))
    usp.usp_a2a4d(hs, back, rd, ud, -1)
    assert np.array_equal(bits(back), bits(loc))
    usp.usp_check()


def test_head_windows_bitexact():
    """Head groups (the head-chunk loop) read and write windows of the full tensors."""
    bs, L, Ht, hd, rd, ud = 1, 256, 12, 128, 2, 2
    x = rand((bs, L, Ht, hd), torch.bfloat16, seed=11)
    xd = x.to(DEV)
    Lu, Lr = L // (rd * ud), L // rd
    for h0, H in ((0, 4), (4, 4), (8, 4), (2, 6)):
        loc = torch.empty(rd, ud, bs, Lu, H, hd, dtype=torch.bfloat16, device=DEV)
        usp.usp_extract_local(xd, loc, rd, ud, h0=h0, H=H)
        assert np.array_equal(bits(loc), oracle.extract_local(bits(x), rd, ud, h0=h0, H=H))
        hs = torch.empty(rd, ud, H // ud, bs, Lr, hd, dtype=torch.bfloat16, device=DEV)
        usp.usp_a2a4d(loc, hs, rd, ud, 1)
        # windowed inverse all-to-all into a full sequence-sharded tensor leaves other heads alone
        full = torch.zeros(rd, ud, bs, Lu, Ht, hd, dtype=torch.bfloat16, device=DEV)
        usp.usp_a2a4d(hs, full, rd, ud, -1, h0=h0, H=H)
        f = bits(full)
        assert np.array_equal(f[:, :, :, :, h0:h0 + H], bits(loc))
        assert not f[:, :, :, :, :h0].any() and not f[:, :, :, :, h0 + H:].any()
        # windowed inverse split into a natural tensor
        nat = torch.zeros_like(xd)
        usp.usp_extract_local(loc, nat, rd, ud, inverse=True, h0=h0, H=H)
        n = bits(nat)
        assert np.array_equal(n[:, :, h0:h0 + H], bits(x)[:, :, h0:h0 + H])
        assert not n[:, :, :h0].any() and not n[:, :, h0 + H:].any()
    usp.usp_check()


@pytest.mark.parametrize("wi", [1, 2, 3, 4])
def test_full_size_permutes(wi):
    """At the workloads' full sizes and launch configuration: the composed split -> AllToAll4D ->
    inverse AllToAll4D -> inverse split is the identity, and both intermediates equal the oracle's
    index maps applied to the same bytes (bit-exact)."""
    w = WORKLOADS[wi]
    H = w.head_chunk or w.hq
    rd, ud, bs, L, hd = w.rd, w.ud, w.bs, w.L, w.hd
    Lu, Lr = L // (rd * ud), L // rd
    # arbitrary 16-bit patterns moved as bf16 rows
    g = torch.Generator(device=DEV).manual_seed(wi)
    x = torch.randint(-30000, 30000, (bs, L, w.hq, hd), generator=g, device=DEV, dtype=torch.int16)
    h0 = w.hq - H  # last head group
    loc = torch.empty(rd, ud, bs, Lu, H, hd, dtype=torch.int16, device=DEV)
    hs = torch.empty(rd, ud, H // ud, bs, Lr, hd, dtype=torch.int16, device=DEV)
    bf = torch.bfloat16
    usp.usp_extract_local(x.view(bf), loc.view(bf), rd, ud, h0=h0, H=H)
    usp.usp_a2a4d(loc.view(bf), hs.view(bf), rd, ud, 1)
    loc2 = torch.empty_like(loc)
    usp.usp_a2a4d(hs.view(bf), loc2.view(bf), rd, ud, -1)
    nat = torch.zeros_like(x)
    usp.usp_extract_local(loc2.view(bf), nat.view(bf), rd, ud, inverse=True, h0=h0, H=H)
    usp.usp_check()
    assert torch.equal(nat[:, :, h0:], x[:, :, h0:])
    assert torch.equal(loc2, loc)
    xs = x.cpu().numpy()
    ref_loc = oracle.extract_local(xs, rd, ud, h0=h0, H=H)
    assert np.array_equal(loc.cpu().numpy(), ref_loc)
    assert np.array_equal(hs.cpu().numpy(), oracle.a2a_fwd(ref_loc, ud))


FUSED_CASES = [  # bs, L, hq, hkv, hd, dtype, rd, ud
    (1, 256, 4, 2, 128, torch.bfloat16, 2, 2),
    (2, 1000, 4, 4, 128, torch.bfloat16, 4, 2),
    (1, 768, 8, 2, 64, torch.bfloat16, 3, 2),
    (1, 1024, 4, 4, 64, torch.float32, 4, 1),
    (1, 240, 4, 4, 96, torch.bfloat16, 5, 2),
]


@pytest.mark.parametrize("bs,L,hq,hkv,hd,dtype,rd,ud", FUSED_CASES)
def test_fused_extract_a2a_bitexact(bs, L, hq, hkv, hd, dtype, rd, ud):
    """One launch moves Q, K, V natural -> head-sharded; equal to the oracle's split then all-to-all."""
    nat = [rand((bs, L, h, hd), dtype, seed=L + h + i) for i, h in enumerate((hq, hkv, hkv))]
    natd = [x.to(DEV) for x in nat]
    hs = [torch.empty(rd, ud, h // ud, bs, L // rd, hd, dtype=dtype, device=DEV) for h in (hq, hkv, hkv)]
    usp.usp_extract_a2a(natd, hs, rd, ud)
    for x, h in zip(nat, hs):
        assert np.array_equal(bits(h), oracle.a2a_fwd(oracle.extract_local(bits(x), rd, ud), ud))
    back = [torch.full_like(x, float("nan")) for x in natd]
    usp.usp_extract_a2a(hs, back, rd, ud, inverse=True)
    for x, b in zip(nat, back):
        assert np.array_equal(bits(b), bits(x))
    usp.usp_check()


def test_fused_head_windows_and_lse_rows():
    """Head windows of a wider natural tensor, and 4-byte lse rows through the inverse."""
    bs, L, Ht, hd, rd, ud = 1, 512, 12, 128, 4, 2
    x = rand((bs, L, Ht, hd), torch.bfloat16, seed=3)
    xd = x.to(DEV)
    hs = torch.empty(rd, ud, 3, bs, L // rd, hd, dtype=torch.bfloat16, device=DEV)
    usp.usp_extract_a2a([xd], [hs], rd, ud, h0s=[6], Hs=[6])
    ref = oracle.a2a_fwd(oracle.extract_local(bits(x), rd, ud, h0=6, H=6), ud)
    assert np.array_equal(bits(hs), ref)
    lse_hs = rand((rd, ud, 3, bs, L // rd), torch.float32, seed=4)
    lse_nat = torch.zeros(bs, L, Ht, device=DEV)
    usp.usp_extract_a2a([lse_hs.to(DEV)], [lse_nat], rd, ud, inverse=True, h0s=[6], Hs=[6])
    want = oracle.extract_inverse(oracle.a2a_inv(bits(lse_hs)[..., None], ud), L, rd, ud)[..., 0]
    got = bits(lse_nat)
    assert np.array_equal(got[:, :, 6:], want) and not got[:, :, :6].any()
    usp.usp_check()


@pytest.mark.parametrize("dtype,hd,rd,ud,bs,L", [(torch.bfloat16, 128, 4, 2, 1, 1024), (torch.float32, 64, 3, 2, 2, 768),
                                                (torch.bfloat16, 64, 5, 1, 1, 1000)])
def test_out_and_lse_rows_in_one_launch(dtype, hd, rd, ud, bs, L):
    """out (rows of hd elements) and lse (rows of one fp32) back to natural order in one launch, for a
    head window of wider natural tensors: equal to the oracle's inverse all-to-all then inverse split
    of each, and to one launch per tensor; heads outside the window untouched."""
    Ht, h0, H = 3 * ud, ud, 2 * ud
    Lr = L // rd
    o_hs = rand((rd, ud, H // ud, bs, Lr, hd), dtype, seed=L + hd)
    l_hs = rand((rd, ud, H // ud, bs, Lr), torch.float32, seed=L + 1)
    od, ld = o_hs.to(DEV), l_hs.to(DEV)
    o_nat = torch.zeros(bs, L, Ht, hd, dtype=dtype, device=DEV)
    l_nat = torch.zeros(bs, L, Ht, device=DEV)
    usp.usp_extract_a2a([od, ld], [o_nat, l_nat], rd, ud, inverse=True, h0s=[h0, h0], Hs=[H, H])
    o_want = oracle.extract_inverse(oracle.a2a_inv(bits(o_hs), ud), L, rd, ud)
    l_want = oracle.extract_inverse(oracle.a2a_inv(bits(l_hs)[..., None], ud), L, rd, ud)[..., 0]
    og, lg = bits(o_nat), bits(l_nat)
    assert np.array_equal(og[:, :, h0:h0 + H], o_want) and np.array_equal(lg[:, :, h0:h0 + H], l_want)
    assert not og[:, :, :h0].any() and not og[:, :, h0 + H:].any()
    assert not lg[:, :, :h0].any() and not lg[:, :, h0 + H:].any()
    o1, l1 = torch.zeros_like(o_nat), torch.zeros_like(l_nat)
    usp.usp_extract_a2a([od], [o1], rd, ud, inverse=True, h0s=[h0], Hs=[H])
    usp.usp_extract_a2a([ld], [l1], rd, ud, inverse=True, h0s=[h0], Hs=[H])
    assert torch.equal(o1, o_nat) and torch.equal(l1, l_nat)
    usp.usp_check()


@pytest.mark.parametrize("dtype,hd,rd,ud,bs,L", [(torch.bfloat16, 128, 4, 2, 1, 1024), (torch.float32, 64, 2, 4, 2, 512)])
def test_a2a4d_multi_out_and_lse(dtype, hd, rd, ud, bs, L):
    """usp_a2a4d_multi: step a5 of out (rows of hd elements) and lse (rows of one fp32) in one launch
    for a head window of wider sequence-sharded tensors, equal to the oracle's inverse all-to-all and
    to one launch per tensor; then the forward direction of Q-like and replicated K-like tensors in
    one launch, equal to one launch per tensor."""
    Ht, h0, H = 3 * ud, ud, 2 * ud
    Lr, Lu = L // rd, L // (rd * ud)
    o_hs = rand((rd, ud, H // ud, bs, Lr, hd), dtype, seed=L + hd + 7)
    l_hs = rand((rd, ud, H // ud, bs, Lr), torch.float32, seed=L + 8)
    od, ld = o_hs.to(DEV), l_hs.to(DEV)
    o_seq = torch.zeros(rd, ud, bs, Lu, Ht, hd, dtype=dtype, device=DEV)
    l_seq = torch.zeros(rd, ud, bs, Lu, Ht, device=DEV)
    usp.usp_a2a4d_multi([od, ld], [o_seq, l_seq], rd, ud, -1, h0s=[h0, h0], Hs=[H, H])
    og, lg = bits(o_seq), bits(l_seq)
    assert np.array_equal(og[:, :, :, :, h0:h0 + H], oracle.a2a_inv(bits(o_hs), ud))
    assert np.array_equal(lg[:, :, :, :, h0:h0 + H], oracle.a2a_inv(bits(l_hs)[..., None], ud)[..., 0])
    assert not og[..., :h0, :].any() and not og[..., h0 + H:, :].any()
    assert not lg[..., :h0].any() and not lg[..., h0 + H:].any()
    o1, l1 = torch.zeros_like(o_seq), torch.zeros_like(l_seq)
    usp.usp_a2a4d(od, o1, rd, ud, -1, h0=h0, H=H)
    usp.usp_a2a4d(ld, l1, rd, ud, -1, h0=h0, H=H)
    assert torch.equal(o1, o_seq) and torch.equal(l1, l_seq)
    # forward: ud query heads and one KV head (replicated on every Ulysses rank) in one launch
    q_seq = rand((rd, ud, bs, Lu, ud, hd), dtype, seed=L + 9).to(DEV)
    k_seq = rand((rd, ud, bs, Lu, 1, hd), dtype, seed=L + 10).to(DEV)
    q_hs = torch.empty(rd, ud, 1, bs, Lr, hd, dtype=dtype, device=DEV)
    k_hs = torch.empty(rd, ud, 1, bs, Lr, hd, dtype=dtype, device=DEV)
    usp.usp_a2a4d_multi([q_seq, k_seq], [q_hs, k_hs], rd, ud, 1)
    q1, k1 = torch.empty_like(q_hs), torch.empty_like(k_hs)
    usp.usp_a2a4d(q_seq, q1, rd, ud, 1)
    usp.usp_a2a4d(k_seq, k1, rd, ud, 1)
    assert torch.equal(q1, q_hs) and torch.equal(k1, k_hs)
    usp.usp_check()
