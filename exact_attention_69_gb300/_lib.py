"""ctypes binding of libattn.so (declared in include/attn.h): argument
marshalling only; every step of the attention forward runs in the library's
sm_103a kernels.

The library is built in place by ``exact_attention_69_gb300.build`` (or
``__graft_entry__.build()``). If it is missing, every call raises: there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libattn.so")

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_MISALIGNED = 3
ATTN_ERR_CUDA = 4
ATTN_ERR_TIMEOUT = 5

ATTN_MASK_NONE = 0
ATTN_MASK_CAUSAL = 1
ATTN_MASK_NA2D = 2
ATTN_MASK_NA3D = 3
ATTN_MASK_CAUSAL_BR = 4


class AttnParamsEx(ctypes.Structure):
    """Mirror of ``attn_params_ex`` (checked against attn_params_size())."""

    _fields_ = [
        ("q", ctypes.c_void_p),
        ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p),
        ("o", ctypes.c_void_p),
        ("lse", ctypes.c_void_p),
        ("B", ctypes.c_int),
        ("H", ctypes.c_int),
        ("Nq", ctypes.c_int),
        ("Nk", ctypes.c_int),
        ("d", ctypes.c_int),
        ("scale", ctypes.c_float),
        ("mask_kind", ctypes.c_int),
        ("window", ctypes.c_int),
        ("dilation", ctypes.c_int),
        ("wrap", ctypes.c_int),
        ("grid_h", ctypes.c_int),
        ("grid_w", ctypes.c_int),
        ("q_stride", ctypes.c_int64 * 3),
        ("k_stride", ctypes.c_int64 * 3),
        ("v_stride", ctypes.c_int64 * 3),
        ("o_stride", ctypes.c_int64 * 3),
        ("stream", ctypes.c_void_p),
        ("num_ctas", ctypes.c_int),
        ("timeout_ns", ctypes.c_uint64),
        ("inject", ctypes.c_int),
        ("ev_start", ctypes.c_void_p),
        ("ev_stop", ctypes.c_void_p),
        ("schedule", ctypes.c_int),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_uint64),
        ("window_w", ctypes.c_int),
        ("grid_d", ctypes.c_int),
        ("window_d", ctypes.c_int),
        ("wrap_d", ctypes.c_int),
    ]


class AttnBwdParams(ctypes.Structure):
    """Mirror of ``attn_bwd_params``."""

    _fields_ = [
        ("q", ctypes.c_void_p),
        ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p),
        ("o", ctypes.c_void_p),
        ("dout", ctypes.c_void_p),
        ("lse", ctypes.c_void_p),
        ("dq", ctypes.c_void_p),
        ("dk", ctypes.c_void_p),
        ("dv", ctypes.c_void_p),
        ("B", ctypes.c_int),
        ("H", ctypes.c_int),
        ("Nq", ctypes.c_int),
        ("Nk", ctypes.c_int),
        ("d", ctypes.c_int),
        ("scale", ctypes.c_float),
        ("mask_kind", ctypes.c_int),
        ("stream", ctypes.c_void_p),
        ("timeout_ns", ctypes.c_uint64),
        ("window", ctypes.c_int),
        ("window_w", ctypes.c_int),
        ("dilation", ctypes.c_int),
        ("wrap", ctypes.c_int),
        ("grid_h", ctypes.c_int),
        ("grid_w", ctypes.c_int),
        ("grid_d", ctypes.c_int),
        ("window_d", ctypes.c_int),
        ("wrap_d", ctypes.c_int),
    ]


class AttnTuneResult(ctypes.Structure):
    """Mirror of ``attn_tune_result``."""

    _fields_ = [
        ("schedule", ctypes.c_int),
        ("num_ctas", ctypes.c_int),
        ("us", ctypes.c_float),
        ("n_tried", ctypes.c_int),
    ]


class AttnError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(message)
        self.code = code


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load libattn.so once and declare the C signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise ImportError(
                f"{path} is missing: build it with exact_attention_69_gb300.build.build() "
                "(nvcc, sm_103a); there is no fallback implementation")
        lib = ctypes.CDLL(path)
        vp, i = ctypes.c_void_p, ctypes.c_int
        lib.attn_params_init.argtypes = [ctypes.POINTER(AttnParamsEx)]
        lib.attn_params_init.restype = None
        lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, ctypes.c_float, i, i, i, i]
        lib.attn_fwd.restype = i
        lib.attn_fwd_ex.argtypes = [ctypes.POINTER(AttnParamsEx)]
        lib.attn_fwd_ex.restype = i
        lib.attn_set_stream.argtypes = [vp]
        lib.attn_set_stream.restype = i
        lib.attn_get_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
        lib.attn_get_device_status.restype = i
        lib.attn_error_string.argtypes = [i]
        lib.attn_error_string.restype = ctypes.c_char_p
        lib.attn_last_error.argtypes = []
        lib.attn_last_error.restype = ctypes.c_char_p
        lib.attn_device_sm_count.argtypes = []
        lib.attn_device_sm_count.restype = i
        lib.attn_shutdown.argtypes = []
        lib.attn_shutdown.restype = None
        lib.attn_abi_version.argtypes = []
        lib.attn_abi_version.restype = i
        lib.attn_params_size.argtypes = []
        lib.attn_params_size.restype = i
        lib.attn_bwd_params_init.argtypes = [ctypes.POINTER(AttnBwdParams)]
        lib.attn_bwd_params_init.restype = None
        lib.attn_bwd.argtypes = [ctypes.POINTER(AttnBwdParams)]
        lib.attn_bwd.restype = i
        lib.attn_workspace_bytes.argtypes = [ctypes.POINTER(AttnParamsEx)]
        lib.attn_workspace_bytes.restype = ctypes.c_int64
        lib.attn_fwd_noalloc.argtypes = [ctypes.POINTER(AttnParamsEx)]
        lib.attn_fwd_noalloc.restype = i
        size = lib.attn_params_size()
        if size != ctypes.sizeof(AttnParamsEx):
            raise ImportError(f"attn_params_ex layout mismatch: library {size} bytes, "
                              f"binding {ctypes.sizeof(AttnParamsEx)} bytes")
        _lib = lib
        return lib


def check(code: int, what: str = "attn") -> None:
    """Raise AttnError for a non-zero status, with the library's message."""
    if code == ATTN_OK:
        return
    lib = load()
    msg = lib.attn_last_error().decode(errors="replace")
    name = lib.attn_error_string(code).decode(errors="replace")
    raise AttnError(code, f"{what}: {name}: {msg}")


def params() -> AttnParamsEx:
    p = AttnParamsEx()
    load().attn_params_init(ctypes.byref(p))
    return p


def fwd_ex(p: AttnParamsEx) -> int:
    return load().attn_fwd_ex(ctypes.byref(p))


def bwd_params() -> AttnBwdParams:
    p = AttnBwdParams()
    load().attn_bwd_params_init(ctypes.byref(p))
    return p


def bwd(p: AttnBwdParams) -> int:
    return load().attn_bwd(ctypes.byref(p))


def device_status():
    """(code, [code, role, tile, cta]) of the current device; clears it."""
    detail = (ctypes.c_uint32 * 4)()
    code = load().attn_get_device_status(detail)
    return code, list(detail)
