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
    """Boolean [Nq, Nk] allowed-set matrix. mask: none | causal | causal_br | clamp | wrap.

    grid: (rows, cols), or (depth, rows, cols) for a volume, tokens row-major with
    the first axis slowest; window: k for every axis, or one size per axis;
    wrap_axes: None (every axis wraps for "wrap", none for "clamp") or one boolean
    per axis.
    """
    if mask == "none":
        return np.ones((Nq, Nk), dtype=bool)
    if mask in ("causal", "causal_br"):
        # top-left: query i sees keys 0..i; bottom-right: keys 0..i + (Nk - Nq)
        shift = 0 if mask == "causal" else Nk - Nq
        m = np.zeros((Nq, Nk), dtype=bool)
        for i in range(Nq):
            m[i, : max(0, min(i + 1 + shift, Nk))] = True
        return m
    grid = tuple(int(g) for g in grid)
    nax = len(grid)
    assert int(np.prod(grid)) == Nq == Nk
    ks = (window,) * nax if np.isscalar(window) else tuple(window)
    wraps = (mask == "wrap",) * nax if wrap_axes is None else tuple(wrap_axes)
    assert len(ks) == nax and len(wraps) == nax
    m = np.zeros((Nq, Nk), dtype=bool)
    for i, qc in enumerate(np.ndindex(*grid)):
        sets = [sorted((_window_coords_wrap if wraps[a] else _window_coords_clamp)(
            qc[a], grid[a], ks[a], dilation)) for a in range(nax)]
        for kc in np.ndindex(*(len(x) for x in sets)):
            coord = tuple(sets[a][kc[a]] for a in range(nax))
            m[i, np.ravel_multi_index(coord, grid)] = True
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
