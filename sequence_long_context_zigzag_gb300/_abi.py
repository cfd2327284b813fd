"""ctypes view of the C ABI in include/usp.h (argument marshalling only; no computation here)."""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libusp.so")

USP_OK = 0
USP_ERR_INVALID_ARG = -1
USP_ERR_SHAPE = -2
USP_ERR_DTYPE = -3
USP_ERR_ALIGN = -4
USP_ERR_UNSUPPORTED = -5
USP_ERR_CUDA = -6
USP_ERR_TIMEOUT = -7

USP_F32 = 0
USP_BF16 = 1

USP_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024

USP_SPLIT_ZIGZAG = 0
USP_SPLIT_BASIC = 1
USP_SPLIT_STRIPE = 2
SPLITS = {"zigzag": USP_SPLIT_ZIGZAG, "basic": USP_SPLIT_BASIC, "stripe": USP_SPLIT_STRIPE}

USP_MODE_FUSED = 0
USP_MODE_STEP = 1
USP_MODE_ACCUM = 2


class UspDims(ctypes.Structure):
    _fields_ = [("bs", ctypes.c_int64), ("L", ctypes.c_int64), ("H", ctypes.c_int32), ("hd", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("rd", ctypes.c_int32), ("ud", ctypes.c_int32),
                ("H_total", ctypes.c_int32), ("h0", ctypes.c_int32), ("split", ctypes.c_int32)]


class UspAttnDesc(ctypes.Structure):
    _fields_ = [("bs", ctypes.c_int64), ("L", ctypes.c_int64), ("hq", ctypes.c_int32), ("hkv", ctypes.c_int32),
                ("hd", ctypes.c_int32), ("rd", ctypes.c_int32), ("ud", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("causal", ctypes.c_int32), ("scale", ctypes.c_float), ("mode", ctypes.c_int32),
                ("step", ctypes.c_int32), ("split", ctypes.c_int32), ("ring_rank_only", ctypes.c_int32),
                ("nseq", ctypes.c_int32), ("cu_seqlens", ctypes.c_void_p)]


class UspError(RuntimeError):
    def __init__(self, fn, status, text):
        super().__init__(f"{fn} failed: {text} (status {status})")
        self.status = status


_lib = None


def load():
    """Load libusp.so (building it with nvcc first if it is absent). Raises if it cannot be loaded:
    there is no fallback implementation."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        from . import build as _build
        _build.build()
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.usp_extract_local.argtypes = [vp, vp, UspDims, ctypes.c_int, ctypes.c_int, vp]
    lib.usp_extract_local.restype = ctypes.c_int
    lib.usp_a2a4d.argtypes = [vp, vp, UspDims, ctypes.c_int, vp]
    lib.usp_a2a4d.restype = ctypes.c_int
    lib.usp_extract_a2a.argtypes = [ctypes.c_int, ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(UspDims),
                                    ctypes.c_int, vp]
    lib.usp_extract_a2a.restype = ctypes.c_int
    lib.usp_a2a4d_multi.argtypes = [ctypes.c_int, ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(UspDims),
                                    ctypes.c_int, vp]
    lib.usp_a2a4d_multi.restype = ctypes.c_int
    lib.usp_forward.argtypes = [vp, vp, vp, vp, vp, UspAttnDesc, ctypes.c_int, vp, ctypes.c_size_t, vp]
    lib.usp_forward.restype = ctypes.c_int
    lib.usp_forward_host.argtypes = [vp, vp, vp, vp, vp, UspAttnDesc, ctypes.c_int, vp, ctypes.c_size_t, vp]
    lib.usp_forward_host.restype = ctypes.c_int
    lib.usp_forward_noalloc.argtypes = [vp, vp, vp, vp, vp, UspAttnDesc, ctypes.c_int, vp]
    lib.usp_forward_noalloc.restype = ctypes.c_int
    lib.usp_forward_workspace_size.argtypes = [UspAttnDesc, ctypes.c_int, ctypes.c_int]
    lib.usp_forward_workspace_size.restype = ctypes.c_size_t
    lib.usp_attn_fwd.argtypes = [vp, vp, vp, vp, vp, UspAttnDesc, vp]
    lib.usp_attn_fwd.restype = ctypes.c_int
    lib.usp_attn_bwd_delta.argtypes = [vp, vp, vp, i64, i32, i32, vp]
    lib.usp_attn_bwd_delta.restype = ctypes.c_int
    lib.usp_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, UspAttnDesc, vp]
    lib.usp_attn_bwd.restype = ctypes.c_int
    lib.usp_backward.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, UspAttnDesc, ctypes.c_int, vp, ctypes.c_size_t,
                                 vp]
    lib.usp_backward.restype = ctypes.c_int
    lib.usp_backward_workspace_size.argtypes = [UspAttnDesc, ctypes.c_int]
    lib.usp_backward_workspace_size.restype = ctypes.c_size_t
    lib.usp_lse_merge.argtypes = [vp, vp, vp, vp, i64, i32, i32, vp]
    lib.usp_lse_merge.restype = ctypes.c_int
    lib.usp_check.argtypes = [vp]
    lib.usp_check.restype = ctypes.c_int
    lib.usp_selftest_timeout.argtypes = [i64, vp]
    lib.usp_selftest_timeout.restype = ctypes.c_int
    lib.usp_strerror.argtypes = [ctypes.c_int]
    lib.usp_strerror.restype = ctypes.c_char_p
    lib.usp_version.argtypes = []
    lib.usp_version.restype = ctypes.c_int
    _lib = lib
    return lib


def strerror(status: int) -> str:
    return load().usp_strerror(int(status)).decode()


def check(fn: str, status: int) -> None:
    if status != USP_OK:
        raise UspError(fn, status, strerror(status))
