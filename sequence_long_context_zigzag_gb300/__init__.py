"""USP-Attention forward (zigzag Ulysses x Ring) on one GB300, over a virtual rank grid.

Thin Python binding of the C ABI in include/usp.h: functions with the ABI's names take torch CUDA
tensors, check their shapes, and pass raw device pointers and the current CUDA stream to libusp.so.
Every step of the path runs in the library's CUDA kernels; torch only allocates memory and supplies
streams. There is no CPU fallback: if libusp.so cannot be loaded, every call raises.

Layouts (all row-major; see include/usp.h for the index formulas):
  natural            (bs, L, H, hd)                      token order of the model
  local              [rd][ud][bs][Lu][H][hd]             after the zigzag split (Algorithm 2)
  head-sharded       [rd][ud][H/ud][bs][Lr][hd]          after AllToAll4D
  lse (head-sharded) [rd][ud][hq/ud][bs][Lr] fp32; lse (natural) (bs, L, hq)
"""
from __future__ import annotations

import ctypes
import math
from typing import Optional

import torch

from . import _abi
from ._abi import (USP_BF16, USP_F32, USP_MODE_ACCUM, USP_MODE_FUSED, USP_MODE_STEP, UspAttnDesc, UspDims,
                   UspError)

__all__ = ["usp_extract_local", "usp_a2a4d", "usp_a2a4d_multi", "usp_extract_a2a", "usp_attn_fwd", "usp_lse_merge", "usp_check", "usp_attention",
           "usp_attention_host", "usp_forward", "usp_forward_host", "usp_forward_workspace_size",
           "usp_forward_noalloc", "heads_per_rank",
           "usp_attn_bwd_delta", "usp_attn_bwd", "usp_backward", "usp_backward_workspace_size", "UspAttentionFunction",
           "UspAttention", "UspError", "USP_MODE_FUSED", "USP_MODE_STEP", "USP_MODE_ACCUM", "lib_path"]

lib_path = _abi.LIB_PATH


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return USP_BF16
    if t.dtype == torch.float32:
        return USP_F32
    raise TypeError(f"unsupported dtype {t.dtype} (bf16 or fp32)")


def _split_code(split) -> int:
    if isinstance(split, str):
        if split not in _abi.SPLITS:
            raise ValueError(f"unknown split {split!r} (zigzag, basic or stripe)")
        return _abi.SPLITS[split]
    return int(split)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(*ts):
    for t in ts:
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError("expected CUDA tensors")
        if not t.is_contiguous():
            raise ValueError("expected contiguous tensors")


def _ptr(t: torch.Tensor) -> int:
    return t.data_ptr()


def _need(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


def usp_extract_local(src: torch.Tensor, dst: torch.Tensor, rd: int, ud: int, vr: int = -1, inverse: bool = False,
                      h0: int = 0, H: Optional[int] = None, split="zigzag", stream=None) -> torch.Tensor:
    """Zigzag split (inverse=False: natural -> local) or its inverse (local -> natural).

    natural: (bs, L, H_total, hd), or (bs, L, H_total) for an lse tensor; local:
    [rd][ud][bs][Lu][H][hd] (or (bs, Lu, H, hd) when vr >= 0). Heads [h0, h0+H) of the natural tensor.
    """
    _dev(src, dst)
    nat, loc = (dst, src) if inverse else (src, dst)
    _need(nat.dtype == loc.dtype, "dtype mismatch")
    if nat.dim() == 3:
        bs, L, Ht = nat.shape
        hd = 1
    else:
        _need(nat.dim() == 4, "natural tensor must be (bs, L, H, hd) or (bs, L, H)")
        bs, L, Ht, hd = nat.shape
    H = Ht - h0 if H is None else H
    _need(0 <= h0 and h0 + H <= Ht, "head window out of range")
    _need(L % (2 * rd) == 0 and (L // rd) % ud == 0, "L must split into 2*rd chunks and L/rd into ud parts")
    Lu = L // (rd * ud)
    ranks = rd * ud if vr < 0 else 1
    _need(loc.numel() == ranks * bs * Lu * H * hd, f"local tensor has {loc.numel()} elements, "
          f"expected {ranks * bs * Lu * H * hd}")
    d = UspDims(bs, L, H, hd, _dtype_code(nat), rd, ud, Ht, h0, _split_code(split))
    _abi.check("usp_extract_local", _abi.load().usp_extract_local(
        _ptr(src), _ptr(dst), d, int(vr), int(bool(inverse)), _stream(stream)))
    return dst


def heads_per_rank(H: int, ud: int) -> int:
    """Heads each Ulysses rank holds after the forward all-to-all: H // ud when ud divides H, 1 when
    H divides ud (K/V replicated for GQA/MQA with fewer KV heads than Ulysses ranks), else 0."""
    if H <= 0 or ud <= 0:
        return 0
    if H % ud == 0:
        return H // ud
    return 1 if ud % H == 0 else 0


def _a2a4d_dims(src: torch.Tensor, dst: torch.Tensor, rd: int, ud: int, dir: int, h0: int, H: Optional[int]):
    _dev(src, dst)
    seq, hs = (src, dst) if dir > 0 else (dst, src)
    _need(seq.dtype == hs.dtype, "dtype mismatch")
    if seq.dim() == 5:
        rd_, ud_, bs, Lu, Ht = seq.shape
        hd = 1
    else:
        _need(seq.dim() == 6, "sequence-sharded tensor must be [rd][ud][bs][Lu][H][hd]")
        rd_, ud_, bs, Lu, Ht, hd = seq.shape
    _need(rd_ == rd and ud_ == ud, "grid mismatch")
    H = Ht - h0 if H is None else H
    _need(0 <= h0 and h0 + H <= Ht, "head window out of range")
    Hl = heads_per_rank(H, ud)
    _need(Hl > 0, "heads must divide by ud or divide ud")
    L = Lu * ud * rd
    _need(hs.numel() == rd * ud * Hl * bs * ud * Lu * hd, "head-sharded tensor has the wrong size")
    return UspDims(bs, L, H, hd, _dtype_code(seq), rd, ud, Ht, h0, 0)


def usp_a2a4d(src: torch.Tensor, dst: torch.Tensor, rd: int, ud: int, dir: int = 1, h0: int = 0,
              H: Optional[int] = None, stream=None) -> torch.Tensor:
    """AllToAll4D inside every Ulysses group: dir=+1 sequence-sharded [rd][ud][bs][Lu][H_total][hd]
    -> head-sharded [rd][ud][H/ud][bs][Lr][hd]; dir=-1 back. lse tensors drop the trailing hd axis.
    dir=+1 with H < ud (ud % H == 0, K/V under GQA/MQA) replicates: head-sharded is
    [rd][ud][1][bs][Lr][hd], rank u' holding head u' // (ud // H); dir=-1 then sums each head's
    replicas (the adjoint, for gradients)."""
    d = _a2a4d_dims(src, dst, rd, ud, dir, h0, H)
    _abi.check("usp_a2a4d", _abi.load().usp_a2a4d(_ptr(src), _ptr(dst), d, 1 if dir > 0 else -1,
                                                 _stream(stream)))
    return dst


def usp_a2a4d_multi(srcs, dsts, rd: int, ud: int, dir: int = 1, h0s=None, Hs=None, stream=None):
    """usp_a2a4d for up to four tensors in one launch (their rows may differ: out and lse together);
    tensor k moves heads [h0s[k], h0s[k] + Hs[k]) of its sequence-sharded tensor."""
    srcs, dsts = list(srcs), list(dsts)
    n = len(srcs)
    _need(1 <= n <= 4 and len(dsts) == n, "one to four tensors")
    h0s = [0] * n if h0s is None else list(h0s)
    Hs = [None] * n if Hs is None else list(Hs)
    dims = [_a2a4d_dims(srcs[k], dsts[k], rd, ud, dir, h0s[k], Hs[k]) for k in range(n)]
    vp = ctypes.c_void_p
    _abi.check("usp_a2a4d_multi", _abi.load().usp_a2a4d_multi(
        n, (vp * n)(*[_ptr(x) for x in srcs]), (vp * n)(*[_ptr(x) for x in dsts]), (UspDims * n)(*dims),
        1 if dir > 0 else -1, _stream(stream)))
    return dsts


def usp_extract_a2a(srcs, dsts, rd: int, ud: int, inverse: bool = False, h0s=None, Hs=None, split="zigzag",
                    stream=None):
    """Zigzag split then AllToAll4D in one pass (inverse: AllToAll4D's inverse then the inverse split),
    for up to four tensors in one launch (their rows may differ: out and lse go back together). inverse=False: srcs[k] natural (bs, L, H_total, hd) (or
    (bs, L, H_total) for lse) -> dsts[k] head-sharded [rd][ud][H/ud][bs][Lr](, hd) ([rd][ud][1]... with
    replicated heads when H < ud, as usp_a2a4d); inverse=True the other way round. Tensor k moves heads
    [h0s[k], h0s[k] + Hs[k]) of its natural tensor."""
    srcs, dsts = list(srcs), list(dsts)
    n = len(srcs)
    _need(1 <= n <= 4 and len(dsts) == n, "one to four tensors")
    h0s = [0] * n if h0s is None else list(h0s)
    Hs = [None] * n if Hs is None else list(Hs)
    dims, sp, dp = [], [], []
    for k in range(n):
        src, dst = srcs[k], dsts[k]
        _dev(src, dst)
        nat, hs = (dst, src) if inverse else (src, dst)
        _need(nat.dtype == hs.dtype, "dtype mismatch")
        if nat.dim() == 3:
            bs, L, Ht = nat.shape
            hd = 1
        else:
            _need(nat.dim() == 4, "natural tensor must be (bs, L, H, hd) or (bs, L, H)")
            bs, L, Ht, hd = nat.shape
        H = Ht - h0s[k] if Hs[k] is None else Hs[k]
        _need(0 <= h0s[k] and h0s[k] + H <= Ht, "head window out of range")
        Hl = heads_per_rank(H, ud)
        _need(L % (2 * rd) == 0 and (L // rd) % ud == 0 and Hl > 0, "shape not divisible")
        _need(hs.numel() == bs * L * Hl * ud * hd, "head-sharded tensor has the wrong size")
        dims.append(UspDims(bs, L, H, hd, _dtype_code(nat), rd, ud, Ht, h0s[k], _split_code(split)))
        sp.append(_ptr(src))
        dp.append(_ptr(dst))
    vp = ctypes.c_void_p
    _abi.check("usp_extract_a2a", _abi.load().usp_extract_a2a(
        n, (vp * n)(*sp), (vp * n)(*dp), (UspDims * n)(*dims), int(bool(inverse)), _stream(stream)))
    return dsts


def usp_attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor, lse: torch.Tensor,
                 causal: bool = True, scale: Optional[float] = None, mode: int = USP_MODE_FUSED, step: int = 0,
                 split="zigzag", ring_rank: Optional[int] = None, hkv: Optional[int] = None, cu_seqlens=None,
                 stream=None):
    """Ring attention over all virtual ring ranks (or only ring rank ``ring_rank``'s query rows).
    cu_seqlens: packed samples' cumulative lengths (int32, device; a query sees only its own sample).
    q/out [rd][ud][hq/ud][bs][Lr][hd], k/v [rd][ud][hkv/ud][bs][Lr][hd], lse [rd][ud][hq/ud][bs][Lr] fp32.
    Replicated K/V (hkv < ud): k/v [rd][ud][1][bs][Lr][hd] and ``hkv`` gives the global KV head count
    (default: k's heads per rank times ud)."""
    _dev(q, k, v, out, lse)
    _need(q.dim() == 6 and k.dim() == 6 and v.dim() == 6, "q, k, v must be [rd][ud][H/ud][bs][Lr][hd]")
    rd, ud, Hl, bs, Lr, hd = q.shape
    Hkl = k.shape[2]
    _need(k.shape == (rd, ud, Hkl, bs, Lr, hd) and v.shape == k.shape, "k/v shape mismatch")
    _need(out.shape == q.shape and out.dtype == q.dtype, "out must match q")
    _need(lse.shape == (rd, ud, Hl, bs, Lr) and lse.dtype == torch.float32, "lse must be fp32 [rd][ud][Hl][bs][Lr]")
    _need(k.dtype == q.dtype and v.dtype == q.dtype, "dtype mismatch")
    L = Lr * rd
    hkv = Hkl * ud if hkv is None else int(hkv)
    _need(hkv > 0 and heads_per_rank(hkv, ud) == Hkl, "k/v heads per rank do not match hkv and ud")
    nseq, cu = _packed(cu_seqlens, L, q.device)
    d = UspAttnDesc(bs, L, Hl * ud, hkv, hd, rd, ud, _dtype_code(q), int(bool(causal)),
                    float(scale) if scale is not None else 0.0, int(mode), int(step), _split_code(split),
                    0 if ring_rank is None else int(ring_rank) + 1, nseq, cu)
    _abi.check("usp_attn_fwd", _abi.load().usp_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), d,
                                                       _stream(stream)))
    return out, lse


def usp_lse_merge(o_acc: torch.Tensor, lse_acc: torch.Tensor, o_new: torch.Tensor, lse_new: torch.Tensor,
                  stream=None):
    """In place: (o_acc, lse_acc) <- LSE-merge((o_acc, lse_acc), (o_new, lse_new)); o (..., hd)."""
    _dev(o_acc, lse_acc, o_new, lse_new)
    _need(o_acc.shape == o_new.shape and o_acc.dtype == o_new.dtype, "o shapes/dtypes differ")
    _need(lse_acc.dtype == torch.float32 and lse_new.dtype == torch.float32, "lse must be fp32")
    hd = o_acc.shape[-1]
    rows = o_acc.numel() // hd
    _need(lse_acc.numel() == rows and lse_new.numel() == rows, "lse must hold one value per row")
    _abi.check("usp_lse_merge", _abi.load().usp_lse_merge(_ptr(o_acc), _ptr(lse_acc), _ptr(o_new), _ptr(lse_new),
                                                         rows, hd, _dtype_code(o_acc), _stream(stream)))
    return o_acc, lse_acc


def usp_check(stream=None) -> None:
    """Synchronise the stream and raise if a kernel's bounded device-side wait ran out."""
    _abi.check("usp_check", _abi.load().usp_check(_stream(stream)))


def usp_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, ud: int, rd: int, causal: bool = True,
                  scale: Optional[float] = None, head_chunk: Optional[int] = None, natural_output: bool = True,
                  split="zigzag", cu_seqlens=None, stream=None):
    """USP-Attention forward (Algorithm 1 of the USP review) over a virtual ud x rd grid on one GPU.

    q: (bs, L, hq, hd), k/v: (bs, L, hkv, hd) CUDA tensors in natural token order. For every head group
    of ``head_chunk`` query heads (all heads when None): zigzag split, AllToAll4D, ring attention with
    LSE merging, inverse AllToAll4D (steps a1-a6). Returns (out, lse): natural (bs, L, hq, hd) and
    (bs, L, hq) when ``natural_output``, else the sequence-sharded [rd][ud][bs][Lu][hq][hd] and
    [rd][ud][bs][Lu][hq] a model would keep.
    """
    _dev(q, k, v)
    bs, L, hq, hd = q.shape
    hkv = k.shape[2]
    _need(k.shape == (bs, L, hkv, hd) and v.shape == k.shape, "k/v shape mismatch")
    _need(hq % hkv == 0, "hq must divide by hkv")
    G = hq // hkv
    hc = hq if head_chunk is None else head_chunk
    _need(hq % hc == 0 and hc % G == 0, "head_chunk must divide hq and be a multiple of hq/hkv")
    hkc = hc // G
    Hkl = heads_per_rank(hkc, ud)
    _need(hc % ud == 0 and Hkl > 0, "query head groups must divide by ud, KV groups divide or be divided by ud")
    _need(L % (2 * rd) == 0 and (L // rd) % ud == 0, "L must split into 2*rd chunks and L/rd into ud parts")
    Lu, Lr = L // (rd * ud), L // rd
    dev, dt = q.device, q.dtype
    if natural_output:
        out = torch.empty(bs, L, hq, hd, device=dev, dtype=dt)
        lse = torch.empty(bs, L, hq, device=dev, dtype=torch.float32)
        usp_forward(q, k, v, out, lse, ud, rd, causal=causal, scale=scale, head_chunk=head_chunk, split=split,
                    cu_seqlens=cu_seqlens, stream=stream)
        return out, lse
    out = torch.empty(rd, ud, bs, Lu, hq, hd, device=dev, dtype=dt)
    lse = torch.empty(rd, ud, bs, Lu, hq, device=dev, dtype=torch.float32)
    # per-group workspace, reused across groups
    qh = torch.empty(rd, ud, hc // ud, bs, Lr, hd, device=dev, dtype=dt)
    kh = torch.empty(rd, ud, Hkl, bs, Lr, hd, device=dev, dtype=dt)
    vh = torch.empty_like(kh)
    oh = torch.empty_like(qh)
    lh = torch.empty(rd, ud, hc // ud, bs, Lr, device=dev, dtype=torch.float32)
    for g0 in range(0, hq, hc):
        gk = g0 // G
        # a1 + a2: zigzag split and AllToAll4D of Q, K, V in one launch
        usp_extract_a2a([q, k, v], [qh, kh, vh], rd, ud, h0s=[g0, gk, gk], Hs=[hc, hkc, hkc], split=split,
                        stream=stream)
        # a3 + a4: the ring with the fused LSE merge
        usp_attn_fwd(qh, kh, vh, oh, lh, causal=causal, scale=scale, split=split, hkv=hkc, cu_seqlens=cu_seqlens,
                     stream=stream)
        # a5 on out and lse: back to the sequence-sharded layout a model keeps
        usp_a2a4d(oh, out, rd, ud, -1, h0=g0, H=hc, stream=stream)
        usp_a2a4d(lh, lse, rd, ud, -1, h0=g0, H=hc, stream=stream)
    return out, lse


def _packed(cu_seqlens, L, device):
    """(nseq, device pointer) of packed samples' cumulative lengths (int32 on the tensors' device)."""
    if cu_seqlens is None:
        return 0, None
    _need(isinstance(cu_seqlens, torch.Tensor) and cu_seqlens.dtype == torch.int32 and cu_seqlens.dim() == 1
          and cu_seqlens.is_contiguous() and cu_seqlens.device == device,
          "cu_seqlens must be a contiguous 1-D int32 tensor on the tensors' device")
    n = cu_seqlens.numel() - 1
    _need(n >= 1 and n <= L, "cu_seqlens needs 2 to L + 1 entries")
    return n, cu_seqlens.data_ptr()


def _forward_desc(q, k, ud, rd, causal, scale, split="zigzag", cu_seqlens=None):
    bs, L, hq, hd = q.shape
    hkv = k.shape[2]
    nseq, cu = _packed(cu_seqlens, L, q.device)
    return UspAttnDesc(bs, L, hq, hkv, hd, rd, ud, _dtype_code(q), int(bool(causal)),
                       float(scale) if scale is not None else 0.0, USP_MODE_FUSED, 0, _split_code(split), 0,
                       nseq, cu)


def usp_forward_workspace_size(q, k, ud: int, rd: int, head_chunk: Optional[int] = None, host: bool = False,
                               causal: bool = True) -> int:
    """Workspace bytes usp_forward / usp_forward_host need for these shapes."""
    d = _forward_desc(q, k, ud, rd, causal, None)
    n = _abi.load().usp_forward_workspace_size(d, int(head_chunk or 0), int(bool(host)))
    _need(n > 0, "invalid forward shapes")
    return int(n)


def _check_natural(q, k, v, out, lse):
    bs, L, hq, hd = q.shape
    hkv = k.shape[2]
    _need(k.shape == (bs, L, hkv, hd) and v.shape == k.shape, "k/v shape mismatch")
    _need(out.shape == q.shape and out.dtype == q.dtype, "out must match q")
    _need(lse.shape == (bs, L, hq) and lse.dtype == torch.float32, "lse must be fp32 (bs, L, hq)")
    _need(k.dtype == q.dtype and v.dtype == q.dtype, "dtype mismatch")


def usp_forward(q, k, v, out, lse, ud: int, rd: int, causal: bool = True, scale: Optional[float] = None,
                head_chunk: Optional[int] = None, workspace: Optional[torch.Tensor] = None, split="zigzag",
                cu_seqlens=None, stream=None):
    """The whole forward on device buffers in one C call (natural-order in and out). cu_seqlens:
    packed samples' cumulative lengths (int32 on the device), each sample attending only within itself."""
    _dev(q, k, v, out, lse)
    _check_natural(q, k, v, out, lse)
    d = _forward_desc(q, k, ud, rd, causal, scale, split, cu_seqlens)
    n = usp_forward_workspace_size(q, k, ud, rd, head_chunk, host=False, causal=causal)
    if workspace is None:
        workspace = torch.empty(n, dtype=torch.uint8, device=q.device)
    _need(workspace.numel() >= n and workspace.is_cuda, "workspace too small")
    _abi.check("usp_forward", _abi.load().usp_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), d,
                                                     int(head_chunk or 0), _ptr(workspace), workspace.numel(),
                                                     _stream(stream)))
    return out, lse


def usp_forward_noalloc(q, k, v, out, lse, ud: int, rd: int, causal: bool = True, scale: Optional[float] = None,
                        head_chunk: Optional[int] = None, stream=None):
    """usp_forward with the library's own fixed scratch array instead of a caller workspace: for
    callers that cannot allocate device memory (see include/usp.h). Shapes whose workspace exceeds
    the array (32 MiB) raise UspError (USP_ERR_UNSUPPORTED); calls must not overlap on the GPU.
    The library uses the current device's array, so the call runs with the tensors' device current
    (all five tensors must be on one device)."""
    _dev(q, k, v, out, lse)
    _need(all(t.device == q.device for t in (k, v, out, lse)), "q, k, v, out, lse must be on one device")
    _check_natural(q, k, v, out, lse)
    d = _forward_desc(q, k, ud, rd, causal, scale)
    with torch.cuda.device(q.device):
        _abi.check("usp_forward_noalloc", _abi.load().usp_forward_noalloc(
            _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), d, int(head_chunk or 0), _stream(stream)))
    return out, lse


def usp_forward_host(q, k, v, out, lse, ud: int, rd: int, causal: bool = True, scale: Optional[float] = None,
                     head_chunk: Optional[int] = None, workspace: Optional[torch.Tensor] = None, device=None,
                     stream=None):
    """The whole forward from host tensors to host tensors, pipelined per head group inside the
    library. With all five tensors pinned, the library's kernels read and write them directly over the
    CPU-GPU link, beside the attention of the neighbouring head group; otherwise each group's window is
    copied in and out (pageable tensors: without overlap). Work is queued on ``stream`` (the current
    stream of ``device``); synchronise it before reading ``out`` / ``lse``."""
    for t in (q, k, v, out, lse):
        _need(isinstance(t, torch.Tensor) and not t.is_cuda and t.is_contiguous(), "expected contiguous host tensors")
    _check_natural(q, k, v, out, lse)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    d = _forward_desc(q, k, ud, rd, causal, scale)
    n = usp_forward_workspace_size(q, k, ud, rd, head_chunk, host=True, causal=causal)
    if workspace is None:
        workspace = torch.empty(n, dtype=torch.uint8, device=dev)
    _need(workspace.numel() >= n and workspace.is_cuda, "workspace too small")
    with torch.cuda.device(dev):
        _abi.check("usp_forward_host", _abi.load().usp_forward_host(
            _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), d, int(head_chunk or 0), _ptr(workspace),
            workspace.numel(), _stream(stream)))
    return out, lse


def usp_attention_host(q, k, v, ud: int, rd: int, causal: bool = True, scale: Optional[float] = None,
                       head_chunk: Optional[int] = None, device=None):
    """usp_attention for host tensors: allocates pinned outputs, runs usp_forward_host, waits."""
    bs, L, hq, hd = q.shape
    out = torch.empty(bs, L, hq, hd, dtype=q.dtype).pin_memory()
    lse = torch.empty(bs, L, hq, dtype=torch.float32).pin_memory()
    usp_forward_host(q, k, v, out, lse, ud, rd, causal=causal, scale=scale, head_chunk=head_chunk, device=device)
    torch.cuda.current_stream(device).synchronize()
    return out, lse


def usp_attn_bwd_delta(out: torch.Tensor, dout: torch.Tensor, delta: torch.Tensor, stream=None) -> torch.Tensor:
    """delta[row] = <dout[row], out[row]> (fp32) for every row of hd elements (any row-contiguous layout)."""
    _dev(out, dout, delta)
    _need(out.shape == dout.shape and out.dtype == dout.dtype, "out / dout differ")
    hd = out.shape[-1]
    rows = out.numel() // hd
    _need(delta.numel() == rows and delta.dtype == torch.float32, "delta must hold one fp32 value per row")
    _abi.check("usp_attn_bwd_delta", _abi.load().usp_attn_bwd_delta(_ptr(out), _ptr(dout), _ptr(delta), rows, hd,
                                                                   _dtype_code(out), _stream(stream)))
    return delta


def usp_attn_bwd(q, k, v, dout, lse, delta, dq, dk, dv, causal: bool = True, scale: Optional[float] = None,
                 split="zigzag", hkv: Optional[int] = None, cu_seqlens=None, stream=None):
    """Backward of usp_attn_fwd (whole ring) on head-sharded buffers: q/dout/dq [rd][ud][hq/ud][bs][Lr][hd],
    k/v/dk/dv [rd][ud][Hkl][bs][Lr][hd], lse/delta [rd][ud][hq/ud][bs][Lr] fp32 (delta from
    usp_attn_bwd_delta). Replicated K/V (hkv < ud): each replica gets its own rank's share."""
    _dev(q, k, v, dout, lse, delta, dq, dk, dv)
    _need(q.dim() == 6 and k.dim() == 6, "q, k must be [rd][ud][H/ud][bs][Lr][hd]")
    rd, ud, Hl, bs, Lr, hd = q.shape
    Hkl = k.shape[2]
    _need(k.shape == (rd, ud, Hkl, bs, Lr, hd) and v.shape == k.shape, "k/v shape mismatch")
    _need(dout.shape == q.shape and dq.shape == q.shape and dk.shape == k.shape and dv.shape == k.shape,
          "gradient shapes must match their inputs")
    for t in (k, v, dout, dq, dk, dv):
        _need(t.dtype == q.dtype, "dtype mismatch")
    for t in (lse, delta):
        _need(t.shape == (rd, ud, Hl, bs, Lr) and t.dtype == torch.float32, "lse/delta must be fp32 [rd][ud][Hl][bs][Lr]")
    hkv = Hkl * ud if hkv is None else int(hkv)
    _need(hkv > 0 and heads_per_rank(hkv, ud) == Hkl, "k/v heads per rank do not match hkv and ud")
    nseq, cu = _packed(cu_seqlens, Lr * rd, q.device)
    d = UspAttnDesc(bs, Lr * rd, Hl * ud, hkv, hd, rd, ud, _dtype_code(q), int(bool(causal)),
                    float(scale) if scale is not None else 0.0, USP_MODE_FUSED, 0, _split_code(split), 0, nseq, cu)
    _abi.check("usp_attn_bwd", _abi.load().usp_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(lse),
                                                       _ptr(delta), _ptr(dq), _ptr(dk), _ptr(dv), d, _stream(stream)))
    return dq, dk, dv


def usp_backward_workspace_size(q, k, ud: int, rd: int, head_chunk: Optional[int] = None, causal: bool = True) -> int:
    """Workspace bytes usp_backward needs for these shapes."""
    d = _forward_desc(q, k, ud, rd, causal, None)
    n = _abi.load().usp_backward_workspace_size(d, int(head_chunk or 0))
    _need(n > 0, "invalid backward shapes")
    return int(n)


def usp_backward(q, k, v, out, lse, dout, dq, dk, dv, ud: int, rd: int, causal: bool = True,
                 scale: Optional[float] = None, head_chunk: Optional[int] = None,
                 workspace: Optional[torch.Tensor] = None, split="zigzag", cu_seqlens=None, stream=None):
    """The whole backward on device buffers in one C call (natural order in and out): dq, dk, dv of
    the forward's out for the upstream gradient dout, given the forward's out and lse."""
    _dev(q, k, v, out, lse, dout, dq, dk, dv)
    _check_natural(q, k, v, out, lse)
    _need(dout.shape == q.shape and dq.shape == q.shape and dk.shape == k.shape and dv.shape == k.shape,
          "gradient shapes must match their inputs")
    for t in (dout, dq, dk, dv):
        _need(t.dtype == q.dtype and t.is_contiguous(), "gradients must be contiguous and of q's dtype")
    d = _forward_desc(q, k, ud, rd, causal, scale, split, cu_seqlens)
    n = usp_backward_workspace_size(q, k, ud, rd, head_chunk, causal=causal)
    if workspace is None:
        workspace = torch.empty(n, dtype=torch.uint8, device=q.device)
    _need(workspace.numel() >= n and workspace.is_cuda, "workspace too small")
    _abi.check("usp_backward", _abi.load().usp_backward(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), d,
        int(head_chunk or 0), _ptr(workspace), workspace.numel(), _stream(stream)))
    return dq, dk, dv


class UspAttentionFunction(torch.autograd.Function):
    """usp_forward / usp_backward as one differentiable op: out = USP-Attention(q, k, v) in natural
    order, with gradients for q, k and v (lse is saved for the backward, not differentiated)."""

    @staticmethod
    def forward(ctx, q, k, v, ud, rd, causal=True, scale=None, head_chunk=None, split="zigzag", cu_seqlens=None):
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        out = torch.empty_like(q)
        lse = torch.empty(q.shape[:3], device=q.device, dtype=torch.float32)
        usp_forward(q, k, v, out, lse, ud, rd, causal=causal, scale=scale, head_chunk=head_chunk, split=split,
                    cu_seqlens=cu_seqlens)
        ctx.save_for_backward(q, k, v, out, lse)
        ctx.cfg = (ud, rd, causal, scale, head_chunk, split, cu_seqlens)
        return out

    @staticmethod
    def backward(ctx, dout):
        q, k, v, out, lse = ctx.saved_tensors
        ud, rd, causal, scale, head_chunk, split, cu_seqlens = ctx.cfg
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        usp_backward(q, k, v, out, lse, dout.contiguous(), dq, dk, dv, ud, rd, causal=causal, scale=scale,
                     head_chunk=head_chunk, split=split, cu_seqlens=cu_seqlens)
        return dq, dk, dv, None, None, None, None, None, None, None


class UspAttention:
    """Callable form of :func:`usp_attention` with the grid fixed at construction, in the spirit of
    the pages' ``LongContextAttention(ring_impl_type="zigzag")`` (one device, virtual ranks)."""

    def __init__(self, ulysses_degree: int, ring_degree: int, causal: bool = True, scale: Optional[float] = None,
                 head_chunk: Optional[int] = None):
        self.ud, self.rd = int(ulysses_degree), int(ring_degree)
        self.causal, self.scale, self.head_chunk = causal, scale, head_chunk

    def __call__(self, q, k, v, natural_output: bool = True):
        return usp_attention(q, k, v, self.ud, self.rd, causal=self.causal, scale=self.scale,
                             head_chunk=self.head_chunk, natural_output=natural_output)


def default_scale(hd: int) -> float:
    return 1.0 / math.sqrt(hd)
