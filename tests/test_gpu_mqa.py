"""GQA / MQA with fewer KV heads than Ulysses ranks (hkv < ud, ud % hkv == 0): the forward
all-to-all replicates each KV head on the ud / hkv ranks whose query heads read it. Permutes are
compared bit-exactly with the oracle's maps; attention with the oracle's direct attention (out
max-abs 2e-2, lse relative 1e-3 with denominator max(|lse|, 1))."""
import numpy as np
import pytest
import torch

import oracle
import sequence_long_context_zigzag_gb300 as usp
from seeded_inputs import make_qkv

pytestmark = pytest.mark.gpu


def _check_attn(out, lse, q, k, v):
    o_ref, l_ref = oracle.attn_direct(q, k, v)
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    assert np.abs(o - o_ref).max() <= 2e-2
    assert (np.abs(l - l_ref) / np.maximum(np.abs(l_ref), 1)).max() <= 1e-3


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("L,H,ud,rd", [(512, 1, 4, 2), (480, 2, 4, 3), (256, 1, 2, 1), (1024, 2, 8, 2)])
def test_a2a_replicates_kv_heads(dt, L, H, ud, rd):
    _, k, _ = make_qkv(1, L, H, H, 64, dt, seed=L + H + ud)
    kd = k.cuda()
    Lu, Lr = L // (rd * ud), L // rd
    loc = torch.empty(rd, ud, 1, Lu, H, 64, dtype=kd.dtype, device="cuda")
    usp.usp_extract_local(kd, loc, rd, ud)
    hs = torch.empty(rd, ud, 1, 1, Lr, 64, dtype=kd.dtype, device="cuda")
    usp.usp_a2a4d(loc, hs, rd, ud, 1)
    fused = torch.full_like(hs, 7)
    usp.usp_extract_a2a([kd], [fused], rd, ud)
    usp.usp_check()
    ref = oracle.a2a_fwd(oracle.extract_local(k.numpy() if dt == "f32" else k.view(torch.int16).numpy(),
                                              rd, ud), ud)
    got = hs.cpu()
    got = got.numpy() if dt == "f32" else got.view(torch.int16).numpy()
    assert np.array_equal(got, ref)
    assert torch.equal(fused, hs)


@pytest.mark.parametrize("split", ["basic", "stripe"])
def test_fused_replication_other_splits(split):
    _, k, _ = make_qkv(1, 512, 2, 2, 128, "bf16", seed=11)
    hs = torch.empty(2, 4, 1, 1, 256, 128, dtype=torch.bfloat16, device="cuda")
    usp.usp_extract_a2a([k.cuda()], [hs], 2, 4, split=split)
    usp.usp_check()
    ref = oracle.a2a_fwd(oracle.extract_local(k.view(torch.int16).numpy(), 2, 4, split=split), 4)
    assert np.array_equal(hs.cpu().view(torch.int16).numpy(), ref)


@pytest.mark.parametrize("L,hq,hkv,hd,ud,rd,dt", [
    (1024, 8, 1, 128, 4, 2, "bf16"),     # MQA, tensor-core kernel, 4 replicas
    (1000, 8, 2, 64, 4, 5, "bf16"),      # GQA hkv = 2 < ud = 4, ragged tiles (Lr = 200)
    (2048, 16, 2, 128, 8, 1, "bf16"),    # pure Ulysses, 8 ranks over 2 KV heads
    (512, 4, 1, 64, 2, 2, "f32"),        # fp32 path
])
def test_attention_with_replicated_kv_matches_oracle(L, hq, hkv, hd, ud, rd, dt):
    q, k, v = make_qkv(1, L, hq, hkv, hd, dt, seed=3 * L + hq + hkv)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out, lse = usp.usp_attention(qd, kd, vd, ud=ud, rd=rd)
    usp.usp_check()
    _check_attn(out, lse, q, k, v)
    # the sequence-sharded path (per-call head-sharded buffers, a5 only) agrees with it exactly
    out_s, lse_s = usp.usp_attention(qd, kd, vd, ud=ud, rd=rd, natural_output=False)
    nat = torch.empty_like(out)
    usp.usp_extract_local(out_s, nat, rd, ud, inverse=True)
    usp.usp_check()
    assert torch.equal(nat, out)


def test_forward_chunks_that_replicate_equal_unchunked():
    """Head groups of 4 query heads carry one KV head each, below ud = 2, so the group's K/V are
    replicated; the result is bit-identical to the unchunked forward (no replication)."""
    L, hq, hkv, ud, rd = 1024, 16, 4, 2, 2
    q, k, v = make_qkv(1, L, hq, hkv, 128, "bf16", seed=21)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    outs = []
    for chunk in (None, 4):
        out = torch.empty_like(qd)
        lse = torch.empty(1, L, hq, device="cuda")
        usp.usp_forward(qd, kd, vd, out, lse, ud, rd, head_chunk=chunk)
        outs.append((out, lse))
    usp.usp_check()
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    _check_attn(outs[1][0], outs[1][1], q, k, v)


def test_ring_steps_with_replicated_kv():
    """STEP then ACCUM over the ring on replicated K/V equals the fused ring."""
    L, hq, hkv, ud, rd = 1024, 4, 1, 2, 4
    q, k, v = make_qkv(1, L, hq, hkv, 128, "bf16", seed=5)
    Lr = L // rd
    qh = torch.empty(rd, ud, hq // ud, 1, Lr, 128, dtype=torch.bfloat16, device="cuda")
    kh = torch.empty(rd, ud, 1, 1, Lr, 128, dtype=torch.bfloat16, device="cuda")
    vh = torch.empty_like(kh)
    usp.usp_extract_a2a([q.cuda(), k.cuda(), v.cuda()], [qh, kh, vh], rd, ud)
    o_f, l_f = torch.empty_like(qh), torch.empty(qh.shape[:5], device="cuda")
    usp.usp_attn_fwd(qh, kh, vh, o_f, l_f, hkv=hkv)
    o_s, l_s = torch.empty_like(qh), torch.empty(qh.shape[:5], device="cuda")
    usp.usp_attn_fwd(qh, kh, vh, o_s, l_s, mode=usp.USP_MODE_STEP, step=0, hkv=hkv)
    for t in range(1, rd):
        usp.usp_attn_fwd(qh, kh, vh, o_s, l_s, mode=usp.USP_MODE_ACCUM, step=t, hkv=hkv)
    usp.usp_check()
    o_ref, l_ref = oracle.attn_direct(q, k, v)
    O_ref = oracle.a2a_fwd(oracle.extract_local(o_ref, rd, ud), ud)
    L_ref = oracle.a2a_fwd(oracle.extract_local(l_ref[..., None], rd, ud), ud)[..., 0]
    for o, l in ((o_f, l_f), (o_s, l_s)):
        assert np.abs(o.float().cpu().numpy() - O_ref).max() <= 2e-2
        assert (np.abs(l.cpu().numpy() - L_ref) / np.maximum(np.abs(L_ref), 1)).max() <= 1e-3
