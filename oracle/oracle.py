"""ctypes front end of the fp64 C oracle -- TEST INFRASTRUCTURE ONLY.

Builds ``liboracle.so`` from ``attn_oracle.c`` with gcc (OpenMP) on first use
and evaluates exact attention row by row in fp64. See ``attn_oracle.c`` for the
definition and its sources.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

MASK_NONE = 0
MASK_CAUSAL = 1
MASK_NA2D = 2
MASK_NA3D = 3
MASK_CAUSAL_BR = 4
MASK_CODES = {"none": MASK_NONE, "causal": MASK_CAUSAL, "clamp": MASK_NA2D, "wrap": MASK_NA2D,
              "causal_br": MASK_CAUSAL_BR}

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_default = None


def library_path() -> str:
    return _LIB


def compile_oracle(src: str, out: str) -> str:
    """gcc -O2 -fopenmp, portable flags (no -march), into a shared library."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(SOURCE):
        return _LIB
    return compile_oracle(SOURCE, _LIB)


def _dptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _mask_args(mask_kind, window, wrap, grid, Nq):
    """The C oracle's mask arguments (mask code, window_h, window_w, wrap_h, wrap_w,
    grid_h, grid_w, window_d, wrap_d, grid_d).

    mask_kind: a code, or "none" | "causal" | "causal_br" | "clamp" | "wrap"; a neighbourhood mask
    on a 3-entry grid (depth, rows, columns) is NA3D, else NA2D. window: k for every
    axis, or one odd size per grid axis. wrap: a bool for every axis, or one per grid
    axis; the mask name "wrap" wraps every axis unless wrap says otherwise. NA2D
    without a grid needs a square token count."""
    code = MASK_CODES[mask_kind] if isinstance(mask_kind, str) else int(mask_kind)
    if code == MASK_NA2D and grid is not None and len(grid) == 3:
        code = MASK_NA3D
    if code not in (MASK_NA2D, MASK_NA3D):
        return code, 0, 0, 0, 0, 0, 0, 0, 0, 0
    nax = 3 if code == MASK_NA3D else 2
    if grid is None:
        if nax == 3:
            raise ValueError("NA3D needs an explicit (depth, rows, columns) grid")
        g = int(round(Nq ** 0.5))
        if g * g != Nq:
            raise ValueError("NA2D without explicit grid needs a square token count")
        grid = (g, g)
    if len(grid) != nax:
        raise ValueError(f"grid {grid} does not match the mask's {nax} axes")
    win = [int(x) for x in window] if isinstance(window, (tuple, list)) else [int(window)] * nax
    if isinstance(wrap, (tuple, list)):
        wr = [int(bool(x)) for x in wrap]
    else:
        wr = [int(bool(wrap) or mask_kind == "wrap")] * nax
    if len(win) != nax or len(wr) != nax:
        raise ValueError("window and wrap need one entry per grid axis")
    g = [int(x) for x in grid]
    if nax == 2:
        return code, win[0], win[1], wr[0], wr[1], g[0], g[1], 0, 0, 0
    return code, win[1], win[2], wr[1], wr[2], g[1], g[2], win[0], wr[0], g[0]


class Oracle:
    """One loaded copy of the oracle library (the default one, or a test build)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        lib.oracle_attn_rows.restype = ctypes.c_int
        lib.oracle_attn_rows.argtypes = [
            dp, dp, dp, dp, dp,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_double, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.POINTER(ctypes.c_int64), ctypes.c_int64, ctypes.c_int,
        ]
        lib.oracle_attn_bwd.restype = ctypes.c_int
        lib.oracle_attn_bwd.argtypes = [dp] * 7 + [ctypes.c_int] * 5 + [ctypes.c_double] + \
            [ctypes.c_int] * 12
        lib.oracle_max_threads.restype = ctypes.c_int
        lib.oracle_allowed.restype = ctypes.c_int
        lib.oracle_allowed.argtypes = [ctypes.c_int] * 15
        self._lib = lib
        self.path = path

    def attention_rows(self, q, k, v, rows=None, *, scale, mask_kind=MASK_NONE, window=0,
                       dilation=1, wrap=False, grid=None, nthreads=0):
        """Exact attention in fp64 for the given flat rows of [B, H, Nq].

        q: [B, H, Nq, d]; k, v: [B, H, Nk, d] (anything numpy reads as float64).
        rows: None for every row, else flat indices b*H*Nq + h*Nq + i.
        Returns (o, lse): o [B,H,Nq,d] / lse [B,H,Nq] for rows=None, else
        o [len(rows), d] / lse [len(rows)].
        grid: (rows, columns) for NA2D, (depth, rows, columns) for NA3D; window and
        wrap: one value for every axis or one per grid axis (see _mask_args).
        """
        q = np.ascontiguousarray(np.asarray(q, dtype=np.float64))
        k = np.ascontiguousarray(np.asarray(k, dtype=np.float64))
        v = np.ascontiguousarray(np.asarray(v, dtype=np.float64))
        B, H, Nq, d = q.shape
        Nk = k.shape[2]
        assert k.shape == (B, H, Nk, d) and v.shape == (B, H, Nk, d)
        m = _mask_args(mask_kind, window, wrap, grid, Nq)
        if rows is None:
            o = np.empty((B, H, Nq, d), dtype=np.float64)
            lse = np.empty((B, H, Nq), dtype=np.float64)
            rp, n = None, 0
        else:
            rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
            n = rows.size
            o = np.empty((n, d), dtype=np.float64)
            lse = np.empty((n,), dtype=np.float64)
            rp = rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
        rc = self._lib.oracle_attn_rows(
            _dptr(q), _dptr(k), _dptr(v), _dptr(o), _dptr(lse),
            B, H, Nq, Nk, d, float(scale), m[0], m[1], m[2], int(dilation),
            *m[3:], rp, n, int(nthreads),
        )
        if rc != 0:
            raise ValueError(f"oracle rejected the problem (code {rc})")
        return o, lse

    def attention_bwd(self, q, k, v, dout, *, scale, mask_kind=MASK_NONE, window=0, dilation=1,
                      wrap=False, grid=None, nthreads=0):
        """Gradients (dq, dk, dv) in fp64 of a loss whose gradient at the output O is
        dout [B, H, Nq, d]; q [B, H, Nq, d], k and v [B, H, Nk, d]. Mask arguments as
        attention_rows."""
        q, k, v, dout = (np.ascontiguousarray(np.asarray(t, dtype=np.float64))
                         for t in (q, k, v, dout))
        B, H, Nq, d = q.shape
        Nk = k.shape[2]
        assert k.shape == (B, H, Nk, d) and v.shape == (B, H, Nk, d) and dout.shape == q.shape
        m = _mask_args(mask_kind, window, wrap, grid, Nq)
        dq = np.empty_like(q)
        dk = np.empty_like(k)
        dv = np.empty_like(v)
        rc = self._lib.oracle_attn_bwd(_dptr(q), _dptr(k), _dptr(v), _dptr(dout), _dptr(dq),
                                       _dptr(dk), _dptr(dv), B, H, Nq, Nk, d, float(scale),
                                       m[0], m[1], m[2], int(dilation), *m[3:],
                                       int(nthreads))
        if rc != 0:
            raise ValueError(f"oracle rejected the problem (code {rc})")
        return dq, dk, dv

    def attention(self, q, k, v, **kw):
        """Every row; see attention_rows."""
        return self.attention_rows(q, k, v, None, **kw)

    def allowed(self, i, j, *, Nq, Nk, mask_kind, window=0, dilation=1, wrap=False, grid=None):
        """The oracle's allowed-set predicate for one (query, key) pair."""
        m = _mask_args(mask_kind, window, wrap, grid, Nq)
        r = self._lib.oracle_allowed(int(i), int(j), int(Nq), int(Nk), m[0], m[1], m[2],
                                     int(dilation), *m[3:])
        if r < 0:
            raise ValueError("bad arguments")
        return bool(r)

    def max_threads(self) -> int:
        return int(self._lib.oracle_max_threads())


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
        return _default


def attention_rows(*a, **kw):
    return default().attention_rows(*a, **kw)


def attention_bwd(*a, **kw):
    return default().attention_bwd(*a, **kw)


def attention(*a, **kw):
    return default().attention(*a, **kw)


def allowed(*a, **kw):
    return default().allowed(*a, **kw)


def max_threads() -> int:
    return default().max_threads()
