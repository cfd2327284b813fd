"""Host-side checks of the C ABI: the library loads, exports every declared symbol, and rejects bad
arguments before anything touches a device. Runs without a GPU: none of these calls launches."""
import ctypes
import os
import re

import pytest

import sequence_long_context_zigzag_gb300 as usp
from sequence_long_context_zigzag_gb300 import _abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"USP_API\s+[\w\s\*]*?\b(usp_\w+)\s*\(", txt)
    return sorted(set(names))


def test_library_loads_and_exports_every_declared_symbol():
    lib = _abi.load()
    names = declared_symbols()
    assert {"usp_extract_local", "usp_a2a4d", "usp_attn_fwd", "usp_lse_merge", "usp_check",
            "usp_strerror", "usp_version"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
        assert ctypes.cast(getattr(lib, n), ctypes.c_void_p).value


def test_version_and_strerror():
    lib = _abi.load()
    assert lib.usp_version() >> 16 == 1
    for code in range(0, -8, -1):
        assert _abi.strerror(code)
    assert _abi.strerror(0) == "success"
    assert "unknown" in _abi.strerror(12345)


def dims(bs=1, L=64, H=4, hd=128, dtype=_abi.USP_BF16, rd=2, ud=2, H_total=0, h0=0, split=0):
    return _abi.UspDims(bs, L, H, hd, dtype, rd, ud, H_total, h0, split)


BAD = 0x1001  # never dereferenced: every case below is rejected before a launch


@pytest.mark.parametrize("d,code", [
    (dims(L=62), _abi.USP_ERR_SHAPE),            # L % (2 rd) != 0
    (dims(L=68, rd=2, ud=4), _abi.USP_ERR_SHAPE),  # (L/rd) % ud != 0
    (dims(H=3), _abi.USP_ERR_SHAPE),             # heads % ud != 0 and ud % heads != 0 (a2a only)
    (dims(H=3, ud=4, L=64), _abi.USP_ERR_SHAPE),  # fewer heads than ranks but not a divisor of ud
    (dims(dtype=7), _abi.USP_ERR_DTYPE),
    (dims(rd=0), _abi.USP_ERR_INVALID_ARG),
    (dims(hd=0), _abi.USP_ERR_INVALID_ARG),
    (dims(H_total=4, h0=2), _abi.USP_ERR_SHAPE),  # window past the end
    (dims(split=3), _abi.USP_ERR_INVALID_ARG),     # unknown split
])
def test_a2a_rejects(d, code):
    assert _abi.load().usp_a2a4d(BAD, BAD, d, 1, None) == code


def test_a2a_rejects_direction_and_alignment():
    lib = _abi.load()
    # fewer heads than ranks (ud % H == 0): replication forward, replica sum backward; both accepted
    assert lib.usp_a2a4d(BAD, BAD, dims(H=1, ud=4), 1, None) == _abi.USP_ERR_ALIGN
    assert lib.usp_a2a4d(BAD, BAD, dims(H=1, ud=4), -1, None) == _abi.USP_ERR_ALIGN
    assert lib.usp_a2a4d(BAD, BAD, dims(H=3, ud=4), -1, None) == _abi.USP_ERR_SHAPE
    assert lib.usp_a2a4d(BAD, BAD, dims(), 0, None) == _abi.USP_ERR_INVALID_ARG
    assert lib.usp_a2a4d(BAD, BAD, dims(), 1, None) == _abi.USP_ERR_ALIGN
    assert lib.usp_a2a4d(None, BAD, dims(), 1, None) == _abi.USP_ERR_INVALID_ARG


def test_extract_rejects():
    lib = _abi.load()
    assert lib.usp_extract_local(BAD, BAD, dims(L=62), -1, 0, None) == _abi.USP_ERR_SHAPE
    assert lib.usp_extract_local(BAD, BAD, dims(), 4, 0, None) == _abi.USP_ERR_INVALID_ARG   # vr >= ud*rd
    assert lib.usp_extract_local(BAD, BAD, dims(), -2, 0, None) == _abi.USP_ERR_INVALID_ARG
    assert lib.usp_extract_local(BAD, BAD, dims(), -1, 0, None) == _abi.USP_ERR_ALIGN
    assert lib.usp_extract_local(BAD, BAD, dims(hd=3, dtype=_abi.USP_BF16), -1, 0, None) == \
        _abi.USP_ERR_UNSUPPORTED   # 6-byte rows
    # empty work is a no-op that succeeds without touching the device
    assert lib.usp_extract_local(None, None, dims(L=0), -1, 0, None) == _abi.USP_OK
    assert lib.usp_extract_local(None, None, dims(bs=0), -1, 1, None) == _abi.USP_OK


def desc(**kw):
    base = dict(bs=1, L=256, hq=4, hkv=2, hd=128, rd=2, ud=2, dtype=_abi.USP_BF16, causal=1, scale=0.0,
                mode=0, step=0, split=0, ring_rank_only=0, nseq=0, cu_seqlens=None)
    base.update(kw)
    return _abi.UspAttnDesc(*[base[f] for f, _ in _abi.UspAttnDesc._fields_])


@pytest.mark.parametrize("kw,code", [
    (dict(hd=96), _abi.USP_ERR_UNSUPPORTED),
    (dict(hq=6, hkv=4), _abi.USP_ERR_SHAPE),
    (dict(hq=6, hkv=3, ud=2), _abi.USP_ERR_SHAPE),   # hkv neither divides by ud nor divides ud
    (dict(hq=4, hkv=1, ud=2), _abi.USP_ERR_ALIGN),   # MQA with ud > hkv is accepted (replicated K/V)
    (dict(L=250), _abi.USP_ERR_SHAPE),
    (dict(mode=3), _abi.USP_ERR_INVALID_ARG),
    (dict(mode=1, step=2), _abi.USP_ERR_INVALID_ARG),
    (dict(dtype=5), _abi.USP_ERR_DTYPE),
    (dict(scale=float("nan")), _abi.USP_ERR_INVALID_ARG),
    (dict(split=5), _abi.USP_ERR_INVALID_ARG),
    (dict(ring_rank_only=3), _abi.USP_ERR_INVALID_ARG),   # rank 2 of rd = 2 does not exist
    (dict(), _abi.USP_ERR_ALIGN),
])
def test_attn_rejects(kw, code):
    assert _abi.load().usp_attn_fwd(BAD, BAD, BAD, BAD, BAD, desc(**kw), None) == code


def test_selftest_timeout_rejects_limits():
    lib = _abi.load()
    assert lib.usp_selftest_timeout(0, None) == _abi.USP_ERR_INVALID_ARG
    assert lib.usp_selftest_timeout(1000001, None) == _abi.USP_ERR_INVALID_ARG


def test_attn_null_and_empty():
    lib = _abi.load()
    assert lib.usp_attn_fwd(None, None, None, None, None, desc(), None) == _abi.USP_ERR_INVALID_ARG
    assert lib.usp_attn_fwd(None, None, None, None, None, desc(L=0), None) == _abi.USP_OK


def test_merge_rejects():
    lib = _abi.load()
    assert lib.usp_lse_merge(BAD, BAD, BAD, BAD, 10, 128, 9, None) == _abi.USP_ERR_DTYPE
    assert lib.usp_lse_merge(BAD, BAD, BAD, BAD, 10, 4, _abi.USP_BF16, None) == _abi.USP_ERR_UNSUPPORTED
    assert lib.usp_lse_merge(BAD, BAD, BAD, BAD, -1, 128, _abi.USP_BF16, None) == _abi.USP_ERR_INVALID_ARG
    assert lib.usp_lse_merge(BAD, BAD, BAD, BAD, 10, 128, _abi.USP_BF16, None) == _abi.USP_ERR_ALIGN
    assert lib.usp_lse_merge(None, None, None, None, 0, 128, _abi.USP_BF16, None) == _abi.USP_OK


def test_binding_rejects_cpu_tensors():
    import torch
    x = torch.zeros(1, 8, 2, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        usp.usp_extract_local(x, x, 2, 1)


def test_extract_a2a_rejects():
    import ctypes
    lib = _abi.load()
    vp = ctypes.c_void_p
    two = (vp * 2)(BAD, BAD)
    d_ok = dims()
    assert lib.usp_extract_a2a(0, two, two, (_abi.UspDims * 1)(d_ok), 0, None) == _abi.USP_ERR_INVALID_ARG
    assert lib.usp_extract_a2a(5, two, two, (_abi.UspDims * 1)(d_ok), 0, None) == _abi.USP_ERR_INVALID_ARG
    # tensors of one launch must share L / grid / row size
    mixed = (_abi.UspDims * 2)(dims(), dims(L=128))
    assert lib.usp_extract_a2a(2, two, two, mixed, 0, None) == _abi.USP_ERR_SHAPE
    # a head count the Ulysses degree does not divide
    assert lib.usp_extract_a2a(1, two, two, (_abi.UspDims * 1)(dims(H=3)), 0, None) == _abi.USP_ERR_SHAPE
    assert lib.usp_extract_a2a(2, two, two, (_abi.UspDims * 2)(dims(), dims(H=2)), 0, None) == _abi.USP_ERR_ALIGN
    # rows may differ between the tensors of one launch (out with lse): past the shape checks, the
    # misaligned pointers are what is rejected
    out_lse = (_abi.UspDims * 2)(dims(), dims(hd=1, dtype=_abi.USP_F32))
    assert lib.usp_extract_a2a(2, two, two, out_lse, 1, None) == _abi.USP_ERR_ALIGN
    # but not the split
    assert lib.usp_extract_a2a(2, two, two, (_abi.UspDims * 2)(dims(), dims(split=1)), 1, None) == _abi.USP_ERR_SHAPE


def test_a2a4d_multi_rejects():
    import ctypes
    lib = _abi.load()
    vp = ctypes.c_void_p
    two = (vp * 2)(BAD, BAD)
    one = (_abi.UspDims * 1)(dims())
    assert lib.usp_a2a4d_multi(0, two, two, one, 1, None) == _abi.USP_ERR_INVALID_ARG
    assert lib.usp_a2a4d_multi(5, two, two, one, 1, None) == _abi.USP_ERR_INVALID_ARG
    assert lib.usp_a2a4d_multi(1, two, two, one, 0, None) == _abi.USP_ERR_INVALID_ARG
    assert lib.usp_a2a4d_multi(2, two, two, (_abi.UspDims * 2)(dims(), dims(L=128)), -1, None) == _abi.USP_ERR_SHAPE
    # out with lse rows, and a split the all-to-all alone does not use: past the shape checks
    out_lse = (_abi.UspDims * 2)(dims(), dims(hd=1, dtype=_abi.USP_F32, split=1))
    assert lib.usp_a2a4d_multi(2, two, two, out_lse, -1, None) == _abi.USP_ERR_ALIGN


def test_forward_workspace_and_rejects():
    lib = _abi.load()
    d = desc(L=1024, hq=8, hkv=2, ud=2, rd=2)
    n_dev = lib.usp_forward_workspace_size(d, 8, 0)
    n_host = lib.usp_forward_workspace_size(d, 8, 1)
    # q group 1024*8*128*2 = 2 MiB, kv group 512 KiB, lse group 32 KiB: q, out, k, v, lse on the device
    assert n_dev == 2 * 2 ** 21 + 2 * 2 ** 19 + 2 ** 15
    assert n_host > n_dev
    assert lib.usp_forward_workspace_size(d, 3, 0) == 0            # 3 does not divide 8
    # 1 KV head per group with ud = 2: each Ulysses rank gets a replica, so head-sharded k and v
    # hold 2 heads' worth (2 * 512 KiB) beside q and out (2 * 1 MiB) and lse (16 KiB)
    assert lib.usp_forward_workspace_size(d, 4, 0) == 2 * 2 ** 20 + 2 * 2 ** 19 + 2 ** 14
    assert lib.usp_forward_workspace_size(desc(L=1024, hq=6, hkv=3, ud=2), 0, 0) == 0  # 3 vs ud 2
    assert lib.usp_forward_workspace_size(desc(mode=1), 0, 0) == 0  # only the fused mode
    ws = BAD - 1  # 0x1000: 256-byte aligned, never dereferenced (rejected before any launch)
    assert lib.usp_forward(BAD, BAD, BAD, BAD, BAD, d, 8, ws, n_dev - 1, None) == _abi.USP_ERR_INVALID_ARG
    assert lib.usp_forward(BAD, BAD, BAD, BAD, BAD, d, 8, BAD, n_dev, None) == _abi.USP_ERR_ALIGN
    assert lib.usp_forward_host(BAD, BAD, BAD, BAD, BAD, d, 8, ws, n_host - 1, None) == _abi.USP_ERR_INVALID_ARG


def test_forward_noalloc_rejects_before_launch():
    lib = _abi.load()
    # workspace above the fixed scratch: L = 65536 MHA, 16 heads per group, hd 128 bf16 (> 32 MiB)
    big = desc(L=65536, hq=16, hkv=16, ud=2, rd=2)
    assert lib.usp_forward_workspace_size(big, 0, 0) > _abi.USP_NOALLOC_SCRATCH_BYTES
    assert lib.usp_forward_noalloc(BAD, BAD, BAD, BAD, BAD, big, 0, None) == _abi.USP_ERR_UNSUPPORTED
    # invalid shapes report the same status as usp_forward
    assert lib.usp_forward_noalloc(BAD, BAD, BAD, BAD, BAD, desc(L=250), 0, None) == _abi.USP_ERR_SHAPE
    assert lib.usp_forward_noalloc(None, None, None, None, None, desc(L=0), 0, None) == _abi.USP_OK


def test_backward_rejects_before_launch():
    lib = _abi.load()
    nine = [BAD] * 9
    assert lib.usp_attn_bwd(*nine, desc(mode=1), None) == _abi.USP_ERR_INVALID_ARG       # whole ring only
    assert lib.usp_attn_bwd(*nine, desc(ring_rank_only=1), None) == _abi.USP_ERR_INVALID_ARG
    assert lib.usp_attn_bwd(*nine, desc(hd=96), None) == _abi.USP_ERR_UNSUPPORTED
    assert lib.usp_attn_bwd(*nine, desc(hq=6, hkv=3), None) == _abi.USP_ERR_SHAPE
    assert lib.usp_attn_bwd(*nine, desc(), None) == _abi.USP_ERR_ALIGN
    assert lib.usp_attn_bwd(None, *nine[1:], desc(), None) == _abi.USP_ERR_INVALID_ARG
    assert lib.usp_attn_bwd(None, *nine[1:], desc(L=0), None) == _abi.USP_OK
    assert lib.usp_attn_bwd_delta(BAD, BAD, BAD, 10, 4, _abi.USP_BF16, None) == _abi.USP_ERR_UNSUPPORTED
    assert lib.usp_attn_bwd_delta(BAD, BAD, BAD, 10, 128, 9, None) == _abi.USP_ERR_DTYPE
    assert lib.usp_attn_bwd_delta(BAD, BAD, BAD, 10, 128, _abi.USP_BF16, None) == _abi.USP_ERR_ALIGN
    assert lib.usp_attn_bwd_delta(None, None, None, 0, 128, _abi.USP_BF16, None) == _abi.USP_OK


def test_backward_workspace_size():
    lib = _abi.load()
    d = desc(L=1024, hq=8, hkv=2, ud=2, rd=2)
    # D of all rows (1024*8*4 = 32 KiB), q/dout/dq groups (2 MiB each), k/v/dk/dv (512 KiB each),
    # lse and D groups (32 KiB each)
    assert lib.usp_backward_workspace_size(d, 0) == 2 ** 15 + 3 * 2 ** 21 + 4 * 2 ** 19 + 2 * 2 ** 15
    assert lib.usp_backward_workspace_size(desc(mode=1), 0) == 0
    ws = BAD - 1
    n = lib.usp_backward_workspace_size(d, 0)
    assert lib.usp_backward(*([BAD] * 9), d, 0, ws, n - 1, None) == _abi.USP_ERR_INVALID_ARG
    assert lib.usp_backward(*([BAD] * 9), d, 0, BAD, n, None) == _abi.USP_ERR_ALIGN


def test_packed_samples_rejects():
    lib = _abi.load()
    assert lib.usp_attn_fwd(BAD, BAD, BAD, BAD, BAD, desc(nseq=3, cu_seqlens=None), None) == _abi.USP_ERR_INVALID_ARG
    assert lib.usp_attn_fwd(BAD, BAD, BAD, BAD, BAD, desc(nseq=-1), None) == _abi.USP_ERR_INVALID_ARG
    assert lib.usp_attn_fwd(BAD, BAD, BAD, BAD, BAD, desc(nseq=3, cu_seqlens=0x1002), None) == _abi.USP_ERR_INVALID_ARG
    assert lib.usp_attn_fwd(BAD, BAD, BAD, BAD, BAD, desc(L=256, nseq=300, cu_seqlens=0x1000), None) == \
        _abi.USP_ERR_SHAPE
    assert lib.usp_attn_fwd(BAD, BAD, BAD, BAD, BAD, desc(nseq=3, cu_seqlens=0x1000), None) == _abi.USP_ERR_ALIGN
    assert lib.usp_attn_bwd(*([BAD] * 9), desc(nseq=3, cu_seqlens=None), None) == _abi.USP_ERR_INVALID_ARG
    assert lib.usp_attn_bwd(*([BAD] * 9), desc(nseq=3, cu_seqlens=0x1000), None) == _abi.USP_ERR_ALIGN
