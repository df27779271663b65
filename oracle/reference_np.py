"""Dense numpy twin of the oracle, for tiny shapes -- TEST INFRASTRUCTURE ONLY.

Written separately from ``attn_oracle.c`` so that each can catch the other's
mistakes: here the neighbourhood mask is built from explicit window coordinate
sets (the keys a query sees, listed), not from a membership predicate, and the
softmax is the textbook ``exp(s - max(s)) / sum`` applied to one row at a time.

Sources: "Fused Self Attention" (NKI tutorial), "Background" (S = Q K^T,
R = softmax(S) V); "Profiling in PyTorch" part 3, "Deconstructing Naive
Attention" (scale, masked_fill(-inf), softmax, matmul); NATTEN issue #142
(neighbourhood windows, wrap mode, logsumexp output).
"""
from __future__ import annotations

import numpy as np


def _window_coords_clamp(c: int, G: int, k: int, dil: int) -> set:
    """Coordinates seen by query coordinate c on an axis of length G.

    The positions sharing c's residue modulo dil form a sequence; the window is
    k consecutive members of that sequence, centred on c where possible and
    pushed inward at the ends so that it always holds k members.
    """
    members = list(range(c % dil, G, dil))
    pos = members.index(c)
    lo = pos - k // 2
    lo = max(lo, 0)
    lo = min(lo, len(members) - k)
    return set(members[lo:lo + k])


def _window_coords_wrap(c: int, G: int, k: int, dil: int) -> set:
    """Circular window: k members spaced dil apart, centred on c, modulo G."""
    return {(c + dil * t) % G for t in range(-(k // 2), k // 2 + 1)}


def mask_matrix(Nq: int, Nk: int, mask: str, window=0, dilation: int = 1,
                grid=None, wrap_axes=None) -> np.ndarray:
    """Boolean [Nq, Nk] allowed-set matrix. mask: none | causal | clamp | wrap.

    window: k, or (k_rows, k_cols); wrap_axes: None (both axes wrap for "wrap",
    neither for "clamp") or (rows, cols) booleans.
    """
    if mask == "none":
        return np.ones((Nq, Nk), dtype=bool)
    if mask == "causal":
        m = np.zeros((Nq, Nk), dtype=bool)
        for i in range(Nq):
            m[i, : min(i + 1, Nk)] = True
        return m
    gh, gw = grid
    assert gh * gw == Nq == Nk
    kh, kw = (window, window) if np.isscalar(window) else (window[0], window[1])
    wh, ww = (mask == "wrap",) * 2 if wrap_axes is None else wrap_axes
    fn_h = _window_coords_wrap if wh else _window_coords_clamp
    fn_w = _window_coords_wrap if ww else _window_coords_clamp
    m = np.zeros((Nq, Nk), dtype=bool)
    for qy in range(gh):
        rows = fn_h(qy, gh, kh, dilation)
        for qx in range(gw):
            cols = fn_w(qx, gw, kw, dilation)
            i = qy * gw + qx
            for ky in rows:
                for kx in cols:
                    m[i, ky * gw + kx] = True
    return m


def attention(q, k, v, scale: float, allowed: np.ndarray):
    """q [Nq,d], k/v [Nk,d] float64; allowed [Nq,Nk] bool -> (o [Nq,d], lse [Nq])."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    Nq, d = q.shape
    o = np.zeros((Nq, v.shape[1]), dtype=np.float64)
    lse = np.full((Nq,), -np.inf, dtype=np.float64)
    for i in range(Nq):
        idx = np.nonzero(allowed[i])[0]
        if idx.size == 0:
            continue
        s = scale * (k[idx] @ q[i])
        e = np.exp(s - s.max())
        o[i] = (e / e.sum()) @ v[idx]
        lse[i] = s.max() + np.log(e.sum())
    return o, lse
