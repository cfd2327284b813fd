"""The one-call forward (usp_forward on device buffers, usp_forward_host pipelined from pinned host
buffers) through the C ABI: parity with the oracle, and bit-identity between the two paths and across
head-group sizes (the same kernels run on the same data)."""
import numpy as np
import pytest
import torch

import oracle
import sequence_long_context_zigzag_gb300 as usp
from seeded_inputs import make_qkv

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("L,hq,hkv,hd,ud,rd,chunk", [(1024, 16, 4, 128, 2, 2, 8), (768, 8, 8, 64, 2, 3, 2),
                                                     (1000, 16, 4, 128, 2, 4, 8)])
def test_forward_device_matches_oracle_and_is_chunk_invariant(L, hq, hkv, hd, ud, rd, chunk):
    q, k, v = make_qkv(1, L, hq, hkv, hd, "bf16", seed=L + hq + chunk)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out = torch.empty_like(qd)
    lse = torch.empty(1, L, hq, device="cuda")
    usp.usp_forward(qd, kd, vd, out, lse, ud, rd, head_chunk=chunk)
    out2 = torch.empty_like(qd)
    lse2 = torch.empty(1, L, hq, device="cuda")
    usp.usp_forward(qd, kd, vd, out2, lse2, ud, rd)
    usp.usp_check()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    o_ref, l_ref = oracle.attn_direct(q, k, v)
    assert np.abs(out.float().cpu().numpy() - o_ref).max() <= 2e-2
    assert (np.abs(lse.cpu().numpy() - l_ref) / np.maximum(np.abs(l_ref), 1)).max() <= 1e-3


@pytest.mark.parametrize("mem", ["pinned", "pageable", "mixed"])
@pytest.mark.parametrize("L,hq,hkv,hd,ud,rd,chunk", [(1024, 32, 8, 128, 2, 2, 8), (512, 8, 8, 64, 1, 4, 2),
                                                     (256, 4, 4, 128, 2, 1, None)])
def test_forward_host_equals_device(L, hq, hkv, hd, ud, rd, chunk, mem):
    """Host-buffer forward gives exactly the device-buffer result on both of its paths: pinned
    buffers (the kernels read and write host memory directly), pageable or partly pageable buffers
    (the pipelined copies; 4 groups exercise both staging slots and their reuse). Two calls in a row
    on one workspace stay correct."""
    q, k, v = make_qkv(1, L, hq, hkv, hd, "bf16", seed=7 * L + hq)
    pin_in, pin_out = {"pinned": (True, True), "pageable": (False, False), "mixed": (True, False)}[mem]
    qp, kp, vp = ((x.pin_memory() if pin_in else x.clone()) for x in (q, k, v))
    out = torch.empty_like(q)
    lse = torch.empty(1, L, hq)
    if pin_out:
        out, lse = out.pin_memory(), lse.pin_memory()
    ws = torch.empty(usp.usp_forward_workspace_size(q, k, ud, rd, chunk, host=True), dtype=torch.uint8,
                     device="cuda")
    od = torch.empty(q.shape, dtype=q.dtype, device="cuda")
    ld = torch.empty(1, L, hq, device="cuda")
    usp.usp_forward(q.cuda(), k.cuda(), v.cuda(), od, ld, ud, rd, head_chunk=chunk)
    for _ in range(2):
        out.zero_()
        lse.zero_()
        usp.usp_forward_host(qp, kp, vp, out, lse, ud, rd, head_chunk=chunk, workspace=ws)
        torch.cuda.current_stream().synchronize()
        usp.usp_check()
        assert torch.equal(out, od.cpu()) and torch.equal(lse, ld.cpu())


def test_attention_host_helper():
    q, k, v = make_qkv(1, 512, 4, 2, 128, "bf16", seed=3)
    out, lse = usp.usp_attention_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), ud=1, rd=4, head_chunk=2)
    o_ref, l_ref = oracle.attn_direct(q, k, v)
    assert np.abs(out.float().numpy() - o_ref).max() <= 2e-2
    assert (np.abs(lse.numpy() - l_ref) / np.maximum(np.abs(l_ref), 1)).max() <= 1e-3


@pytest.mark.parametrize("L,hq,hkv,ud,rd", [(32768, 32, 8, 1, 8), (16384, 24, 6, 2, 4)])
def test_forward_host_overlapped_transfers(L, hq, hkv, ud, rd):
    """Pinned buffers at lengths where each head group's attention is long enough for the library to
    run the neighbouring groups' host transfers beside it, on a few thread blocks, with the attention
    on the remaining SMs (4 and 3 head groups of 8 query heads: both buffer slots, an odd count).
    Bit-identical to the device-buffer forward (the same units, on fewer CTAs), three calls in a row
    on one workspace."""
    q, k, v = make_qkv(1, L, hq, hkv, 128, "bf16", seed=L + hq)
    qp, kp, vp = (x.pin_memory() for x in (q, k, v))
    out = torch.empty_like(q).pin_memory()
    lse = torch.empty(1, L, hq).pin_memory()
    ws = torch.empty(usp.usp_forward_workspace_size(q, k, ud, rd, 8, host=True), dtype=torch.uint8, device="cuda")
    od = torch.empty(q.shape, dtype=q.dtype, device="cuda")
    ld = torch.empty(1, L, hq, device="cuda")
    usp.usp_forward(q.cuda(), k.cuda(), v.cuda(), od, ld, ud, rd, head_chunk=8)
    od, ld = od.cpu(), ld.cpu()
    for _ in range(3):
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        usp.usp_forward_host(qp, kp, vp, out, lse, ud, rd, head_chunk=8, workspace=ws)
        torch.cuda.current_stream().synchronize()
        usp.usp_check()
        assert torch.equal(out, od) and torch.equal(lse, ld)
