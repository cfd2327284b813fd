"""USP-Attention forward oracle -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct CPU reference (fp64) for the zigzag Ulysses x Ring forward path.
Only ``tests/``, the package's ``smoke()`` check and ``bench.py``'s CPU-baseline leg may import it.
It shares no code with the CUDA path, and the CUDA path never imports it.

Sources (page title, then the section / algorithm / figure / equation):
  * "USP: 统一序列并行方法用于长上下文生成式AI" (xllm-io paper review), section 三 技术架构:
    Algorithm 1 (USP-Attention), Algorithm 2 (load-balanced sequence split), the AllToAll4D shape
    change (bs, L/N, hc, hd) -> (hc/N, bs, L, hd), the 2 x 4 process grid.
  * "Context Parallel 与 Ulysses" (charliedreemur), section 先弄清楚 (ring attention, the online
    softmax LSE merge), Fig. 1 (ring schedule at cp = 4), Fig. 2 (zigzag balance), section 推导 /
    关键公式 (per-GPU forward communication volumes) and the hand-worked example table.

Every function is pinned by ``tests/test_oracle.py`` to something other than itself (closed forms,
the pages' printed numbers under ``tests/golden/``, library routines for the special cases, brute
force on tiny inputs). Functions without such a pin would say "parity unpinned"; none is.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "usp_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

_DT = {"f32": 0, "bf16": 1, "f64": 2}


# ----------------------------------------------------------------------------------------------
# building / loading the C core
# ----------------------------------------------------------------------------------------------
def build(force: bool = False) -> str:
    """Compile usp_oracle.c with gcc (-O2, OpenMP, no fast-math) into oracle/liboracle.so."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
    lib.oracle_attn_direct.argtypes = [vp, vp, vp, i32, i64, i64, i32, i32, i32, dbl, i32, vp, i64, vp, vp]
    lib.oracle_attn_direct.restype = i32
    lib.oracle_attn_direct_seg.argtypes = [vp, vp, vp, i32, i64, i64, i32, i32, i32, dbl, i32, vp, vp, vp, i64, vp,
                                           vp]
    lib.oracle_attn_direct_seg.restype = i32
    lib.oracle_attn_block_seg.argtypes = [vp, vp, vp, i64, vp, vp, vp, vp, i64, i32, i32, i32, dbl, i32, vp, vp]
    lib.oracle_attn_block_seg.restype = i32
    lib.oracle_attn_block.argtypes = [vp, vp, i64, vp, vp, vp, i64, i32, i32, i32, dbl, i32, vp, vp]
    lib.oracle_attn_block.restype = i32
    lib.oracle_attn_bwd_direct.argtypes = [vp, vp, vp, vp, i32, i64, i64, i32, i32, i32, dbl, i32, vp, i64, vp,
                                           i64, vp, vp]
    lib.oracle_attn_bwd_direct.restype = i32
    lib.oracle_attn_block_bwd.argtypes = [vp, vp, vp, vp, vp, i64, vp, vp, vp, i64, i32, i32, i32, dbl, i32, vp,
                                          vp, vp]
    lib.oracle_attn_block_bwd.restype = i32
    lib.oracle_attn_bwd_direct_seg.argtypes = [vp, vp, vp, vp, i32, i64, i64, i32, i32, i32, dbl, i32, vp, vp, vp,
                                               i64, vp, i64, vp, vp]
    lib.oracle_attn_bwd_direct_seg.restype = i32
    lib.oracle_attn_block_bwd_seg.argtypes = [vp, vp, vp, vp, vp, vp, i64, vp, vp, vp, vp, i64, i32, i32, i32, dbl,
                                              i32, vp, vp, vp]
    lib.oracle_attn_block_bwd_seg.restype = i32
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = i32
    _lib = lib
    return lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def _raw(x):
    """numpy view of the raw bytes of a CPU tensor/array plus the oracle dtype code."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().contiguous().cpu()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), _DT["bf16"]
            if x.dtype == torch.float32:
                return x.numpy(), _DT["f32"]
            if x.dtype == torch.float64:
                return x.numpy(), _DT["f64"]
            raise TypeError(f"unsupported dtype {x.dtype}")
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, _DT["f32"]
    if x.dtype == np.float64:
        return x, _DT["f64"]
    if x.dtype == np.uint16:
        return x, _DT["bf16"]
    raise TypeError(f"unsupported dtype {x.dtype}")


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


# ----------------------------------------------------------------------------------------------
# attention (C core)
# ----------------------------------------------------------------------------------------------
def seg_bounds(cu_seqlens, L):
    """Packed sequences: for every position, the first and one-past-last position of its sample and
    the sample's index. cu_seqlens = [0, l_0, l_0 + l_1, ..., L] (the samples' cumulative lengths)."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    if cu.ndim != 1 or len(cu) < 2 or cu[0] != 0 or cu[-1] != L or np.any(np.diff(cu) <= 0):
        raise ValueError("cu_seqlens must rise strictly from 0 to L")
    ids = np.repeat(np.arange(len(cu) - 1), np.diff(cu))
    return cu[ids], cu[ids + 1], ids


def attn_direct(q, k, v, scale=None, causal=True, rows=None, cu_seqlens=None):
    """Direct softmax attention with row LSE for selected query rows, natural token order.

    q: (bs, L, hq, hd), k/v: (bs, L, hkv, hd); fp32, bf16 or fp64 (torch tensors or numpy).
    Returns out (bs, nrows, hq, hd) fp64 and lse (bs, nrows, hq) fp64 (natural log).
    Context-Parallel page, section 先弄清楚 (partial output and log-sum-exp); causal mask j <= i.
    cu_seqlens: packed samples (every batch element packed alike); a query sees only keys of its own
    sample (the sequence packing of the Context-Parallel page's ByteScale section).
    """
    qa, dt = _raw(q)
    ka, dk = _raw(k)
    va, dv = _raw(v)
    if not (dt == dk == dv):
        raise TypeError("q, k, v must share a dtype")
    bs, L, hq, hd = qa.shape
    hkv = ka.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(hd)
    rows = np.arange(L, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((bs, len(rows), hq, hd), dtype=np.float64)
    lse = np.empty((bs, len(rows), hq), dtype=np.float64)
    if cu_seqlens is None:
        rc = _load().oracle_attn_direct(_p(qa), _p(ka), _p(va), dt, bs, L, hq, hkv, hd, float(scale),
                                        int(bool(causal)), _p(rows), len(rows), _p(out), _p(lse))
    else:
        st, en, _ = seg_bounds(cu_seqlens, L)
        st, en = np.ascontiguousarray(st), np.ascontiguousarray(en)
        rc = _load().oracle_attn_direct_seg(_p(qa), _p(ka), _p(va), dt, bs, L, hq, hkv, hd, float(scale),
                                            int(bool(causal)), _p(st), _p(en), _p(rows), len(rows), _p(out),
                                            _p(lse))
    if rc != 0:
        raise ValueError("oracle_attn_direct: bad arguments")
    return out, lse


def attn_block(q, qpos, k, v, kpos, scale, causal=True, qseg=None, kseg=None):
    """Attention of query rows against one block of keys, masked on explicit global positions.

    q: (hq, nq, hd) fp64, k/v: (hkv, nk, hd) fp64. Returns (o (hq, nq, hd), lse (hq, nq)); rows that
    see no key get (0, -inf). One ring step of Algorithm 1 (USP review) / Fig. 1 (Context-Parallel).
    """
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    qpos = np.ascontiguousarray(qpos, dtype=np.int64)
    kpos = np.ascontiguousarray(kpos, dtype=np.int64)
    hq, nq, hd = q.shape
    hkv, nk, _ = k.shape
    o = np.empty((hq, nq, hd), dtype=np.float64)
    lse = np.empty((hq, nq), dtype=np.float64)
    if qseg is None:
        rc = _load().oracle_attn_block(_p(q), _p(qpos), nq, _p(k), _p(v), _p(kpos), nk, hq, hkv, hd,
                                       float(scale), int(bool(causal)), _p(o), _p(lse))
    else:
        qseg = np.ascontiguousarray(qseg, dtype=np.int64)
        kseg = np.ascontiguousarray(kseg, dtype=np.int64)
        rc = _load().oracle_attn_block_seg(_p(q), _p(qpos), _p(qseg), nq, _p(k), _p(v), _p(kpos), _p(kseg), nk,
                                           hq, hkv, hd, float(scale), int(bool(causal)), _p(o), _p(lse))
    if rc != 0:
        raise ValueError("oracle_attn_block: bad arguments")
    return o, lse


def attn_direct_bwd(q, k, v, dout, scale=None, causal=True, q_rows=None, kv_from=0, cu_seqlens=None):
    """Gradients of direct attention's output with respect to q, k, v for an upstream gradient dout
    (the chain rule through softmax, written out in usp_oracle.c), natural token order, fp64.

    q, dout: (bs, L, hq, hd), k/v: (bs, L, hkv, hd), one dtype (fp32, bf16 or fp64).
    q_rows: query rows whose dq is returned (default all); kv_from: dk, dv are returned for key rows
    [kv_from, L) (default all; L for none). Returns dq (bs, len(q_rows), hq, hd),
    dk, dv (bs, L - kv_from, hkv, hd). cu_seqlens: packed samples (as attn_direct).
    """
    qa, dt = _raw(q)
    ka, dk_ = _raw(k)
    va, dv_ = _raw(v)
    ga, dg = _raw(dout)
    if not (dt == dk_ == dv_ == dg):
        raise TypeError("q, k, v, dout must share a dtype")
    bs, L, hq, hd = qa.shape
    hkv = ka.shape[2]
    if ga.shape != qa.shape:
        raise ValueError("dout must have q's shape")
    if scale is None:
        scale = 1.0 / math.sqrt(hd)
    rows = np.arange(L, dtype=np.int64) if q_rows is None else np.ascontiguousarray(q_rows, dtype=np.int64)
    nkv = L - int(kv_from)
    dq = np.zeros((bs, len(rows), hq, hd), dtype=np.float64)
    dk = np.zeros((bs, nkv, hkv, hd), dtype=np.float64)
    dv = np.zeros((bs, nkv, hkv, hd), dtype=np.float64)
    if cu_seqlens is None:
        rc = _load().oracle_attn_bwd_direct(_p(qa), _p(ka), _p(va), _p(ga), dt, bs, L, hq, hkv, hd, float(scale),
                                            int(bool(causal)), _p(rows), len(rows), _p(dq), int(kv_from), _p(dk),
                                            _p(dv))
    else:
        st, en, _ = seg_bounds(cu_seqlens, L)
        st, en = np.ascontiguousarray(st), np.ascontiguousarray(en)
        rc = _load().oracle_attn_bwd_direct_seg(_p(qa), _p(ka), _p(va), _p(ga), dt, bs, L, hq, hkv, hd,
                                                float(scale), int(bool(causal)), _p(st), _p(en), _p(rows),
                                                len(rows), _p(dq), int(kv_from), _p(dk), _p(dv))
    if rc != 0:
        raise ValueError("oracle_attn_bwd_direct: bad arguments")
    return dq, dk, dv


def attn_block_bwd(q, dout, qpos, lse, D, k, v, kpos, scale, causal, dq_acc, dk_acc, dv_acc, qseg=None, kseg=None):
    """One ring step's share of the backward, accumulated in place: dq_acc (hq, nq, hd) += the keys'
    contribution, dk_acc / dv_acc (hkv, nk, hd) += the queries' contribution, using the rows' final
    lse and D = <dout, out> (all fp64, head-sharded block layout as attn_block)."""
    arrs = [np.ascontiguousarray(a, dtype=np.float64) for a in (q, dout, lse, D, k, v)]
    q, dout, lse, D, k, v = arrs
    qpos = np.ascontiguousarray(qpos, dtype=np.int64)
    kpos = np.ascontiguousarray(kpos, dtype=np.int64)
    for a in (dq_acc, dk_acc, dv_acc):
        assert a.dtype == np.float64 and a.flags.c_contiguous
    hq, nq, hd = q.shape
    hkv, nk, _ = k.shape
    if qseg is None:
        rc = _load().oracle_attn_block_bwd(_p(q), _p(dout), _p(qpos), _p(lse), _p(D), nq, _p(k), _p(v), _p(kpos),
                                           nk, hq, hkv, hd, float(scale), int(bool(causal)), _p(dq_acc), _p(dk_acc),
                                           _p(dv_acc))
    else:
        qseg = np.ascontiguousarray(qseg, dtype=np.int64)
        kseg = np.ascontiguousarray(kseg, dtype=np.int64)
        rc = _load().oracle_attn_block_bwd_seg(_p(q), _p(dout), _p(qpos), _p(qseg), _p(lse), _p(D), nq, _p(k), _p(v),
                                               _p(kpos), _p(kseg), nk, hq, hkv, hd, float(scale), int(bool(causal)),
                                               _p(dq_acc), _p(dk_acc), _p(dv_acc))
    if rc != 0:
        raise ValueError("oracle_attn_block_bwd: bad arguments")


# ----------------------------------------------------------------------------------------------
# LSE merge (Context-Parallel page, section 先弄清楚, online-softmax merge equation)
# ----------------------------------------------------------------------------------------------
def lse_merge(o1, l1, o2, l2):
    """lse = log(e^l1 + e^l2), o = e^(l1-lse) o1 + e^(l2-lse) o2, in fp64.

    The log is evaluated as m + log(e^(l1-m) + e^(l2-m)) with m = max(l1, l2) (the same quantity).
    lse = -inf marks an empty partial: it contributes weight 0; two empty partials give (0, -inf).
    o*: (..., hd), l*: (...).
    """
    o1 = np.asarray(o1, dtype=np.float64)
    o2 = np.asarray(o2, dtype=np.float64)
    l1 = np.asarray(l1, dtype=np.float64)
    l2 = np.asarray(l2, dtype=np.float64)
    e1_empty = np.isneginf(l1)
    e2_empty = np.isneginf(l2)
    both = e1_empty & e2_empty
    m = np.where(both, 0.0, np.maximum(l1, l2))
    with np.errstate(invalid="ignore", over="ignore"):
        a1 = np.where(e1_empty, 0.0, np.exp(np.where(e1_empty, 0.0, l1 - m)))
        a2 = np.where(e2_empty, 0.0, np.exp(np.where(e2_empty, 0.0, l2 - m)))
        lse = np.where(both, -np.inf, m + np.log(np.where(both, 1.0, a1 + a2)))
        w1 = np.where(e1_empty, 0.0, np.exp(np.where(e1_empty, 0.0, l1 - lse)))
        w2 = np.where(e2_empty, 0.0, np.exp(np.where(e2_empty, 0.0, l2 - lse)))
    o = w1[..., None] * o1 + w2[..., None] * o2
    return o, lse


# ----------------------------------------------------------------------------------------------
# index maps (USP review, Algorithm 2 and AllToAll4D; applied as explicit gathers)
# ----------------------------------------------------------------------------------------------
def zig(r, p, c, rd):
    """Global token position of ring-local row p on ring rank r.

    Algorithm 2: the sequence is cut into 2*rd chunks of length c; rank r keeps chunk r followed by
    chunk 2*rd - r - 1. Local row p < c is in the first kept chunk, p >= c in the second.
    """
    r = np.asarray(r, dtype=np.int64)
    p = np.asarray(p, dtype=np.int64)
    return np.where(p < c, r * c + p, (2 * rd - 1 - r) * c + (p - c))


SPLITS = ("zigzag", "basic", "stripe")


def split_pos(split, r, p, L, rd):
    """Global token position of ring-local row p on ring rank r under a sequence split.

    zigzag: Algorithm 2 (chunks r and 2*rd - r - 1 of 2*rd equal chunks), see zig();
    basic:  the contiguous split of the plain ring (the USP review's "basic-ring" column, Tables 3-4;
            the Context-Parallel page's sequential split of section 为什么要一头一尾配对): rank r holds
            tokens [r L/rd, (r+1) L/rd);
    stripe: the round-robin split of Striped Attention (USP review, section 七 related work; the YunChang
            page's ring_impl_type "stripe"): rank r holds tokens r, r + rd, r + 2 rd, ...
    """
    r = np.asarray(r, dtype=np.int64)
    p = np.asarray(p, dtype=np.int64)
    if split == "zigzag":
        return zig(r, p, L // (2 * rd), rd)
    if split == "basic":
        return r * (L // rd) + p
    if split == "stripe":
        return p * rd + r
    raise ValueError(f"unknown split {split}")


def _dims(L, rd, ud):
    if L % (2 * rd) or (L // rd) % ud:
        raise ValueError("L must split into 2*rd chunks and L/rd into ud parts")
    return L // (2 * rd), L // rd, L // (rd * ud)


def extract_local(x, rd, ud, h0=0, H=None, split="zigzag"):
    """a1: natural (bs, L, Ht, ...) -> local [rd][ud][bs][Lu][H][...] for every virtual rank.

    Slot (r, u, b, j, h) holds token zig(r, u*Lu + j) of head h0 + h: Algorithm 2 steps 4-6
    (chunk into 2*rd, keep chunks r and 2*rd-r-1, then the u-th of ud equal parts). Other splits put
    token split_pos(split, r, u*Lu + j) there.
    """
    x = np.asarray(x)
    bs, L, Ht = x.shape[:3]
    H = Ht - h0 if H is None else H
    c, _, Lu = _dims(L, rd, ud)
    R = np.arange(rd).reshape(rd, 1, 1, 1, 1)
    U = np.arange(ud).reshape(1, ud, 1, 1, 1)
    B = np.arange(bs).reshape(1, 1, bs, 1, 1)
    J = np.arange(Lu).reshape(1, 1, 1, Lu, 1)
    Hh = np.arange(H).reshape(1, 1, 1, 1, H)
    return x[B, split_pos(split, R, U * Lu + J, L, rd), h0 + Hh]


def extract_inverse(loc, L, rd, ud, split="zigzag"):
    """a7: local [rd][ud][bs][Lu][H][...] -> natural (bs, L, H, ...), the inverse of a1."""
    loc = np.asarray(loc)
    _, _, bs, Lu, H = loc.shape[:5]
    c, _, Lu2 = _dims(L, rd, ud)
    assert Lu == Lu2
    g = np.arange(L)
    if split == "zigzag":
        a = g // c
        first = a < rd
        r = np.where(first, a, 2 * rd - 1 - a)
        p = np.where(first, g % c, c + g % c)
    elif split == "basic":
        r, p = g // (L // rd), g % (L // rd)
    elif split == "stripe":
        r, p = g % rd, g // rd
    else:
        raise ValueError(f"unknown split {split}")
    u, j = p // Lu, p % Lu
    B = np.arange(bs).reshape(bs, 1, 1)
    Hh = np.arange(H).reshape(1, 1, H)
    return loc[r.reshape(1, L, 1), u.reshape(1, L, 1), B, j.reshape(1, L, 1), Hh]


def a2a_fwd(loc, ud):
    """a2: AllToAll4D inside every Ulysses group, sequence-sharded -> head-sharded.

    in  [rd][ud][bs][Lu][H][...]  (rank (r,u) holds Lu tokens of all H heads, shape (bs, L/N, hc, hd))
    out [rd][ud][H/ud][bs][Lr][...] (rank (r,u') holds H/ud heads of all Lr = ud*Lu ring-local
    tokens, shape (hc/N, bs, L, hd)); out[r,u',h',b,u*Lu+j] = in[r,u,b,j,u'*(H/ud)+h'].
    Gathered pieces are concatenated by source Ulysses rank ascending, which restores the ring-local
    order of Algorithm 2 step 6.

    Fewer heads than Ulysses ranks (K/V of GQA/MQA with hkv < ud; the USP review's section 三 gives
    the all-to-all the job of handling K/V head counts that differ from Q's): with ud % H == 0,
    each rank receives the one head its query heads read, head u' // (ud/H), so every head is
    replicated on ud/H ranks and out is [rd][ud][1][bs][Lr][...]: out[r,u',0,b,u*Lu+j] =
    in[r,u,b,j,u'//(ud/H)].
    """
    loc = np.asarray(loc)
    rd, ud2, bs, Lu, H = loc.shape[:5]
    assert ud2 == ud
    Lr = ud * Lu
    R = np.arange(rd).reshape(rd, 1, 1, 1, 1)
    Uo = np.arange(ud).reshape(1, ud, 1, 1, 1)
    B = np.arange(bs).reshape(1, 1, 1, bs, 1)
    P = np.arange(Lr).reshape(1, 1, 1, 1, Lr)
    if H % ud == 0:
        Hl = H // ud
        Ho = np.arange(Hl).reshape(1, 1, Hl, 1, 1)
        return loc[R, P // Lu, B, P % Lu, Uo * Hl + Ho]
    assert ud % H == 0, "head count must divide by ud or divide ud"
    rep = ud // H
    return loc[R, P // Lu, B, P % Lu, Uo // rep]


def a2a_inv(hs, ud):
    """a5: the inverse AllToAll4D (Algorithm 1 step 5, scatter and gather indices swapped).

    in [rd][ud][Hl][bs][Lr][...] -> out [rd][ud][bs][Lu][H = ud*Hl][...];
    out[r,u,b,j,h] = in[r, h // Hl, h % Hl, b, u*Lu + j].
    """
    hs = np.asarray(hs)
    rd, ud2, Hl, bs, Lr = hs.shape[:5]
    assert ud2 == ud and Lr % ud == 0
    Lu, H = Lr // ud, Hl * ud
    R = np.arange(rd).reshape(rd, 1, 1, 1, 1)
    U = np.arange(ud).reshape(1, ud, 1, 1, 1)
    B = np.arange(bs).reshape(1, 1, bs, 1, 1)
    J = np.arange(Lu).reshape(1, 1, 1, Lu, 1)
    Hh = np.arange(H).reshape(1, 1, 1, 1, H)
    return hs[R, Hh // Hl, Hh % Hl, B, U * Lu + J]


def a2a_inv_sum(hs, ud, H):
    """The adjoint of a2a_fwd for a tensor of H heads: a5 when ud divides H; when H < ud (replicated
    heads) every head's gradient is the sum of its ud/H replicas:
    out[r,u,b,j,h] = sum over u' with u' // (ud/H) == h of hs[r,u',0,b,u*Lu+j]."""
    hs = np.asarray(hs)
    if H % ud == 0:
        return a2a_inv(hs, ud)
    assert ud % H == 0 and hs.shape[2] == 1
    rd, _, _, bs, Lr = hs.shape[:5]
    Lu, rep = Lr // ud, ud // H
    out = np.zeros((rd, ud, bs, Lu, H) + hs.shape[5:], dtype=hs.dtype)
    for h in range(H):
        for up in range(h * rep, (h + 1) * rep):
            for u in range(ud):
                out[:, u, :, :, h] += hs[:, up, 0, :, u * Lu:(u + 1) * Lu]
    return out


# ----------------------------------------------------------------------------------------------
# the ring schedule and the literal virtual-rank pipeline
# ----------------------------------------------------------------------------------------------
def ring_source(r, t, rd):
    """KV block held by ring rank r at step t (0-based): (r - t) mod rd (Context-Parallel Fig. 1)."""
    return (r - t) % rd


def ring_schedule(cp):
    """Table [step][gpu] -> index of the KV block that gpu works on at that step (Fig. 1)."""
    return [[ring_source(r, t, cp) for r in range(cp)] for t in range(cp)]


def literal_pipeline(q, k, v, rd, ud, scale=None, causal=True, split="zigzag", cu_seqlens=None):
    """USP-Attention forward, run rank by rank over the virtual ud x rd grid, in fp64.

    Algorithm 2 split (a1), AllToAll4D on Q, K, V (a2), for every ring rank the ring loop in Fig. 1
    order with one masked block per step and the LSE merge folding the partials (a3, a4), the inverse
    AllToAll4D on O and on lse (a5) and the inverse split (a7).
    q: (bs, L, hq, hd), k/v: (bs, L, hkv, hd) numpy or torch (any float dtype; widened to fp64).
    Returns out (bs, L, hq, hd) and lse (bs, L, hq) in natural order.
    cu_seqlens: packed samples; the split is applied to the packed sequence as to one sequence, and
    every block keeps a key only for queries of the same sample.
    """
    q, k, v = (np.asarray(_to_f64(x)) for x in (q, k, v))
    bs, L, hq, hd = q.shape
    hkv = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(hd)
    c, Lr, _ = _dims(L, rd, ud)
    if hq % ud or hq % hkv or (hkv % ud and ud % hkv):
        raise ValueError("hq must divide by ud and by hkv; hkv must divide by ud or divide ud")
    Q = a2a_fwd(extract_local(q, rd, ud, split=split), ud)          # [rd][ud][hq/ud][bs][Lr][hd]
    K = a2a_fwd(extract_local(k, rd, ud, split=split), ud)          # [rd][ud][max(hkv/ud,1)][bs][Lr][hd]
    V = a2a_fwd(extract_local(v, rd, ud, split=split), ud)
    pos = [split_pos(split, r, np.arange(Lr), L, rd) for r in range(rd)]
    seg = None if cu_seqlens is None else seg_bounds(cu_seqlens, L)[2]
    sg = (lambda r: None) if seg is None else (lambda r: seg[pos[r]])  # noqa: E731
    O = np.zeros_like(Q)
    LSE = np.full(Q.shape[:5], -np.inf)
    for r in range(rd):
        for u in range(ud):
            for b in range(bs):
                o_acc = np.zeros((hq // ud, Lr, hd))
                l_acc = np.full((hq // ud, Lr), -np.inf)
                for t in range(rd):
                    s = ring_source(r, t, rd)
                    o_t, l_t = attn_block(Q[r, u, :, b], pos[r], K[s, u, :, b], V[s, u, :, b], pos[s],
                                          scale, causal, sg(r), sg(s))
                    o_acc, l_acc = lse_merge(o_acc, l_acc, o_t, l_t)
                O[r, u, :, b] = o_acc
                LSE[r, u, :, b] = l_acc
    out = extract_inverse(a2a_inv(O, ud), L, rd, ud, split=split)
    lse = extract_inverse(a2a_inv(LSE[..., None], ud), L, rd, ud, split=split)[..., 0]
    return out, lse


def literal_pipeline_bwd(q, k, v, dout, rd, ud, scale=None, causal=True, split="zigzag", cu_seqlens=None):
    """USP-Attention backward, run rank by rank over the virtual ud x rd grid, in fp64.

    The forward's layout changes are applied to q, k, v, the upstream gradient dout, and the
    forward's out and lse (Algorithm 2 split, AllToAll4D). For every ring rank r, the ring runs in
    Fig. 1 order (step t: KV block of rank (r - t) mod rd): each step adds the block's share of dq
    to rank r and of dk, dv to the block's owner -- in a multi-GPU ring those two partials travel
    with the KV block and are home after rd steps. The inverse all-to-all (the replica sum for
    replicated K/V) and the inverse split return dq, dk, dv in natural order.
    """
    q, k, v, dout = (np.asarray(_to_f64(x)) for x in (q, k, v, dout))
    bs, L, hq, hd = q.shape
    hkv = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(hd)
    c, Lr, _ = _dims(L, rd, ud)
    if hq % ud or hq % hkv or (hkv % ud and ud % hkv):
        raise ValueError("hq must divide by ud and by hkv; hkv must divide by ud or divide ud")
    o_nat, l_nat = attn_direct(q, k, v, scale=scale, causal=causal, cu_seqlens=cu_seqlens)
    D_nat = np.einsum("blhd,blhd->blh", dout, o_nat)
    hs = lambda x: a2a_fwd(extract_local(x, rd, ud, split=split), ud)  # noqa: E731
    Q, K, V, dO = hs(q), hs(k), hs(v), hs(dout)
    LSE, DD = hs(l_nat[..., None])[..., 0], hs(D_nat[..., None])[..., 0]
    pos = [split_pos(split, r, np.arange(Lr), L, rd) for r in range(rd)]
    seg = None if cu_seqlens is None else seg_bounds(cu_seqlens, L)[2]
    sg = (lambda r: None) if seg is None else (lambda r: seg[pos[r]])  # noqa: E731
    dQ, dK, dV = np.zeros(Q.shape), np.zeros(K.shape), np.zeros(V.shape)
    for r in range(rd):
        for u in range(ud):
            for b in range(bs):
                dq_r = np.zeros(Q[r, u, :, b].shape)
                for t in range(rd):
                    s = ring_source(r, t, rd)
                    dk_s = np.zeros(K[s, u, :, b].shape)
                    dv_s = np.zeros(V[s, u, :, b].shape)
                    attn_block_bwd(Q[r, u, :, b], dO[r, u, :, b], pos[r], LSE[r, u, :, b], DD[r, u, :, b],
                                   K[s, u, :, b], V[s, u, :, b], pos[s], scale, causal, dq_r, dk_s, dv_s,
                                   sg(r), sg(s))
                    dK[s, u, :, b] += dk_s
                    dV[s, u, :, b] += dv_s
                dQ[r, u, :, b] = dq_r
    dq = extract_inverse(a2a_inv(dQ, ud), L, rd, ud, split=split)
    dk = extract_inverse(a2a_inv_sum(dK, ud, hkv), L, rd, ud, split=split)
    dv = extract_inverse(a2a_inv_sum(dV, ud, hkv), L, rd, ud, split=split)
    return dq, dk, dv


def _to_f64(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().cpu().to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


# ----------------------------------------------------------------------------------------------
# causal work balance (Context-Parallel page Fig. 2 and section 为什么要一头一尾配对)
# ----------------------------------------------------------------------------------------------
def pair_class(qpos, kpos):
    """Causal class of a (query block, key block) pair from its global positions:
    1 = every pair visible, 0 = none visible (skipped), 0.5 = partly visible (a diagonal block)."""
    qpos = np.asarray(qpos)
    kpos = np.asarray(kpos)
    if kpos.max() <= qpos.min():
        return 1.0
    if kpos.min() > qpos.max():
        return 0.0
    return 0.5


def zigzag_rank_work(cp, c=4):
    """Per ring rank, the computed c x c small blocks (diagonal = 1/2) under the zigzag split."""
    work = []
    for r in range(cp):
        qp = zig(r, np.arange(2 * c), c, cp)
        total = 0.0
        for qa in (qp[:c], qp[c:]):
            for b in range(2 * cp):
                total += pair_class(qa, np.arange(b * c, (b + 1) * c))
        work.append(total)
    return work


def zigzag_chunk_work(cp, c=4):
    """Computed small blocks of each of the 2*cp chunks of queries, and which rank holds it."""
    out = []
    for a in range(2 * cp):
        qa = np.arange(a * c, (a + 1) * c)
        w = sum(pair_class(qa, np.arange(b * c, (b + 1) * c)) for b in range(2 * cp))
        owner = [r for r in range(cp) if np.any(zig(r, np.arange(2 * c), c, cp) == a * c)][0]
        out.append((a, owner, w))
    return out


def contiguous_rank_work(cp, c=4):
    """Per rank, computed big blocks (2c x 2c, diagonal = 1/2) when rank r holds tokens
    [2c r, 2c (r+1)) in order (the basic ring split)."""
    B = 2 * c
    return [sum(pair_class(np.arange(r * B, (r + 1) * B), np.arange(b * B, (b + 1) * B))
                for b in range(cp)) for r in range(cp)]


def split_rank_pairs(split, L, rd):
    """Exact causal (query, key) pair count of each ring rank's queries under a split."""
    Lr = L // rd
    return [visible_pairs(split_pos(split, r, np.arange(Lr), L, rd)) for r in range(rd)]


def visible_pairs(positions):
    """Brute-force count of (query, key) pairs with key position <= query position, for one rank's
    query positions against the whole sequence (keys 0..p for a query at position p)."""
    return int(sum(int(p) + 1 for p in np.asarray(positions)))


# ----------------------------------------------------------------------------------------------
# per-GPU forward communication volumes (Context-Parallel page, section 推导 / 关键公式)
# ----------------------------------------------------------------------------------------------
def comm_ring_elems(s, h_kv, cp):
    """Ring: receive cp-1 KV blocks of 2 (s/cp) h_kv elements: V_ring = 2 s h_kv (cp-1)/cp."""
    return 2 * s * h_kv * (cp - 1) / cp


def comm_ulysses_elems(s, h, h_kv, cp):
    """Ulysses: all-to-all on Q, K, V and O, each rank sends (cp-1)/cp of its local data:
    V_Ulysses = (s/cp)(2h + 2h_kv)(cp-1)/cp."""
    return (s / cp) * (2 * h + 2 * h_kv) * (cp - 1) / cp


def counted_ring_elems(s, heads_kv, hd, cp):
    """Count, from the virtual ring schedule (ud=1, rd=cp), the K and V elements one rank uses that
    live on another rank: the blocks it holds at steps t >= 1."""
    Lr = s // cp
    r = 0
    n = 0
    for t in range(cp):
        if ring_source(r, t, cp) != r:
            n += 2 * Lr * heads_kv * hd
    return n


def counted_ulysses_elems(s, heads, heads_kv, hd, cp):
    """Count, through the a2a index maps themselves (ud=cp, rd=1, bs=1), the elements that rank 0
    receives from other ranks: Q, K, V in the forward all-to-all and O in the inverse one. Every
    slot of a label tensor holds the rank it lives on; after the map, rank 0's slots whose label is
    not 0 came over the network."""
    Lu = s // cp

    def fwd(H):
        lab = np.broadcast_to(np.arange(cp, dtype=np.int16).reshape(1, cp, 1, 1, 1), (1, cp, 1, Lu, H))
        got = a2a_fwd(lab, cp)                    # [1][cp][H/cp][1][s]
        return int(np.count_nonzero(got[0, 0] != 0)) * hd

    def inv(H):
        lab = np.broadcast_to(np.arange(cp, dtype=np.int16).reshape(1, cp, 1, 1, 1), (1, cp, H // cp, 1, s))
        got = a2a_inv(lab, cp)                    # [1][cp][1][Lu][H]
        return int(np.count_nonzero(got[0, 0] != 0)) * hd

    return fwd(heads) + 2 * fwd(heads_kv) + inv(heads)
