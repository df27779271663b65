"""Checks that pin the fp64 oracle to facts outside itself.

Each check takes an ``Oracle`` instance and raises AssertionError on failure,
so the same checks run against the shipped oracle (test_oracle_pins.py) and
against copies with a planted mistake (test_oracle_mutants.py), which must
each fail at least one of them.

What pins what:
  golden_wrap_example     NATTEN issue #142 worked example (values printed on the page)
  golden_clamp_by_hand    the shifted-window reading, spelled out by hand on 5x5/k=3
  window_sets_by_hand     literal key sets of a few queries (clamp, wrap, dilation 2)
  constant_v              a convex combination of equal rows returns that row
  zero_qk_means           Q=K=0: the mean of V over the allowed set, LSE = ln |A(i)|
  single_key              N=1: o = v_0, lse = scale q.k
  numpy_twin              independent dense numpy statement on tiny shapes
  sdpa_fp64               torch scaled_dot_product_attention (math) in fp64, none/causal/mask
  invariants              key shift, linearity in V, key permutation, causal prefix
  wrap_equals_pad_clamp   circular pad + clamped NA + crop == wrap NA (issue #142's recipe)
  one_axis_wrap_pad_clamp the same recipe along one axis == wrap along that axis only
  axis_windows_by_hand    literal key sets for a rectangular window and one-axis wrap
  one_d_closed_form       a 1 x N grid is 1-D neighbourhood attention: closed-form windows
  na3d_windows_by_hand    literal key sets on a volume (clamp, wrap on some axes, dilation 2)
  na3d_closed_form        NA3D allowed set == the product of per-axis closed-form windows
                          (interval / circular distance / residue class), depth slowest
  na3d_flat_is_na2d       a volume one slice deep with window 1 along depth == NA2D
  na3d_wrap_pad_clamp     issue #142's recipe in 3-D: circular pad of the wrapped axes,
                          clamped NA3D, crop == NA3D wrapping those axes
  causal_bottom_right     bottom-right causal: == top-left when Nq == Nk; row i == unmasked
                          attention over the first i + (Nk - Nq) + 1 keys; rows that see
                          no key give O = 0, LSE = -inf; torch SDPA with tril(Nk - Nq)
  bwd_autograd_fp64       backward: torch autograd through an explicit fp64 forward
  bwd_finite_differences  backward: central differences of sum(dO * O) along random directions
  bwd_invariants          backward: a common shift of all keys leaves O unchanged (sum_j dK_j
                          = 0); a common shift of V moves every o_i by it (sum_j dV_j =
                          sum_i dO_i)
"""
from __future__ import annotations

import math

import numpy as np

from oracle import reference_np as twin

RNG = np.random.default_rng(1234)


def _rand(*shape, rng=None):
    rng = rng or RNG
    return rng.standard_normal(shape)


def golden_wrap_example(orc, printed):
    q = np.ones((1, 1, 25, 8))
    k = np.ones((1, 1, 25, 8))
    v = np.zeros((1, 1, 25, 8))
    v[0, 0, 0, :] = 1.0
    o, lse = orc.attention(q, k, v, scale=1 / math.sqrt(8), mask_kind="wrap", window=3)
    x = o[0, 0, :, 0].reshape(5, 5)
    assert np.array_equal(np.round(x, 4), np.asarray(printed)), x
    exact = np.where(np.asarray(printed) > 0, 1.0 / 9.0, 0.0)
    assert np.max(np.abs(x - exact)) < 1e-15
    # every query sees exactly 9 keys of score 8/sqrt(8)
    assert np.allclose(lse, math.sqrt(8) + math.log(9), atol=1e-13, rtol=0)


def golden_clamp_by_hand(orc, expected):
    q = np.ones((1, 1, 25, 8))
    k = np.ones((1, 1, 25, 8))
    v = np.zeros((1, 1, 25, 8))
    v[0, 0, 0, :] = 1.0
    o, _ = orc.attention(q, k, v, scale=1 / math.sqrt(8), mask_kind="clamp", window=3)
    x = o[0, 0, :, 0].reshape(5, 5)
    assert np.max(np.abs(x - np.asarray(expected))) < 1e-15, x


def window_sets_by_hand(orc):
    def keys(i, mask, window, grid, dilation=1):
        n = grid[0] * grid[1]
        return {j for j in range(n)
                if orc.allowed(i, j, Nq=n, Nk=n, mask_kind=mask, window=window,
                               dilation=dilation, grid=grid)}

    def tok(y, x, w):
        return y * w + x

    g = (5, 5)
    # clamp, k=3: corner (0,0) -> rows {0,1,2} x cols {0,1,2}; (4,4) -> {2,3,4}^2; (2,1) -> {1,2,3} x {0,1,2}
    assert keys(tok(0, 0, 5), "clamp", 3, g) == {tok(y, x, 5) for y in (0, 1, 2) for x in (0, 1, 2)}
    assert keys(tok(4, 4, 5), "clamp", 3, g) == {tok(y, x, 5) for y in (2, 3, 4) for x in (2, 3, 4)}
    assert keys(tok(2, 1, 5), "clamp", 3, g) == {tok(y, x, 5) for y in (1, 2, 3) for x in (0, 1, 2)}
    # wrap, k=3: corner (0,0) -> rows {4,0,1} x cols {4,0,1}
    assert keys(tok(0, 0, 5), "wrap", 3, g) == {tok(y, x, 5) for y in (4, 0, 1) for x in (4, 0, 1)}
    # rectangular grid 3 x 7, clamp k=3 at (0,6): rows {0,1,2} x cols {4,5,6}
    assert keys(tok(0, 6, 7), "clamp", 3, (3, 7)) == {tok(y, x, 7) for y in (0, 1, 2) for x in (4, 5, 6)}
    # dilation 2 on an 8 x 8 grid, k=3, clamp: query (1,6) -> rows with residue 1: 1,3,5
    # (1 is the first member, so the window starts there) x cols with residue 0: 2,4,6
    # (6 is the last member of {0,2,4,6}, window pushed inward to {2,4,6})
    assert keys(tok(1, 6, 8), "clamp", 3, (8, 8), 2) == {tok(y, x, 8) for y in (1, 3, 5) for x in (2, 4, 6)}
    # dilation 2, wrap, 8 x 8, k=3: query (0,0) -> {6,0,2} x {6,0,2}
    assert keys(tok(0, 0, 8), "wrap", 3, (8, 8), 2) == {tok(y, x, 8) for y in (6, 0, 2) for x in (6, 0, 2)}


CASES = [
    dict(mask_kind="none", Nq=37, Nk=37),
    dict(mask_kind="none", Nq=19, Nk=41),
    dict(mask_kind="causal", Nq=37, Nk=37),
    dict(mask_kind="causal", Nq=41, Nk=23),
    dict(mask_kind="clamp", Nq=49, Nk=49, window=3, grid=(7, 7)),
    dict(mask_kind="wrap", Nq=49, Nk=49, window=5, grid=(7, 7)),
    dict(mask_kind="clamp", Nq=48, Nk=48, window=3, grid=(6, 8)),
    dict(mask_kind="wrap", Nq=48, Nk=48, window=3, grid=(6, 8)),
    dict(mask_kind="clamp", Nq=64, Nk=64, window=3, grid=(8, 8), dilation=2),
    dict(mask_kind="wrap", Nq=64, Nk=64, window=3, grid=(8, 8), dilation=2),
    dict(mask_kind="clamp", Nq=54, Nk=54, window=(3, 5), grid=(6, 9)),
    dict(mask_kind="clamp", Nq=54, Nk=54, window=(5, 3), grid=(6, 9), wrap=(True, False)),
    dict(mask_kind="clamp", Nq=54, Nk=54, window=(3, 3), grid=(6, 9), wrap=(False, True), dilation=2),
    dict(mask_kind="clamp", Nq=15, Nk=15, window=(1, 5), grid=(1, 15)),
    dict(mask_kind="causal_br", Nq=23, Nk=41),
    dict(mask_kind="clamp", Nq=60, Nk=60, window=3, grid=(3, 4, 5)),
    dict(mask_kind="wrap", Nq=64, Nk=64, window=3, grid=(4, 4, 4)),
    dict(mask_kind="clamp", Nq=90, Nk=90, window=(3, 5, 3), grid=(3, 6, 5), wrap=(True, False, True)),
    dict(mask_kind="clamp", Nq=180, Nk=180, window=(1, 3, 3), grid=(5, 6, 6), wrap=(False, True, False),
         dilation=2),
]


def _kw(case):
    kw = dict(mask_kind=case["mask_kind"])
    for name in ("window", "grid", "dilation", "wrap"):
        if name in case:
            kw[name] = case[name]
    return kw


def _twin_mask(case):
    return twin.mask_matrix(case["Nq"], case["Nk"], case["mask_kind"], case.get("window", 0),
                            case.get("dilation", 1), case.get("grid"), case.get("wrap"))


def constant_v(orc):
    rng = np.random.default_rng(7)
    for case in CASES:
        Nq, Nk, d = case["Nq"], case["Nk"], 6
        q = _rand(2, 1, Nq, d, rng=rng)
        k = _rand(2, 1, Nk, d, rng=rng)
        c = rng.standard_normal(d)
        v = np.broadcast_to(c, (2, 1, Nk, d)).copy()
        o, _ = orc.attention(q, k, v, scale=0.7, **_kw(case))
        assert np.max(np.abs(o - c)) < 1e-13, case


def zero_qk_means(orc):
    rng = np.random.default_rng(8)
    for case in CASES:
        Nq, Nk, d = case["Nq"], case["Nk"], 5
        q = np.zeros((1, 1, Nq, d))
        k = np.zeros((1, 1, Nk, d))
        v = _rand(1, 1, Nk, d, rng=rng)
        o, lse = orc.attention(q, k, v, scale=1.3, **_kw(case))
        m = case["mask_kind"]
        if m == "none":
            exp_o = np.broadcast_to(v[0, 0].mean(axis=0), (Nq, d))
            exp_n = np.full(Nq, Nk)
        elif m in ("causal", "causal_br"):
            shift = 0 if m == "causal" else Nk - Nq
            cnt = np.minimum(np.arange(Nq) + 1 + shift, Nk)
            csum = np.cumsum(v[0, 0], axis=0)
            exp_o = csum[cnt - 1] / cnt[:, None]
            exp_n = cnt
        else:
            kk = case["window"]
            nax = len(case["grid"])
            ks = (kk,) * nax if np.isscalar(kk) else kk
            exp_n = np.full(Nq, int(np.prod(ks)))  # every query sees a full window on each axis
            allowed = _twin_mask(case)
            exp_o = np.stack([v[0, 0][allowed[i]].mean(axis=0) for i in range(Nq)])
        assert np.max(np.abs(o[0, 0] - exp_o)) < 1e-13, case
        assert np.max(np.abs(lse[0, 0] - np.log(exp_n))) < 1e-13, case


def single_key(orc):
    rng = np.random.default_rng(9)
    q = _rand(1, 2, 1, 8, rng=rng)
    k = _rand(1, 2, 1, 8, rng=rng)
    v = _rand(1, 2, 1, 8, rng=rng)
    for mask in ("none", "causal"):
        o, lse = orc.attention(q, k, v, scale=0.37, mask_kind=mask)
        assert np.max(np.abs(o - v)) < 1e-15
        exp = 0.37 * np.einsum("bhid,bhid->bhi", q, k)
        assert np.max(np.abs(lse - exp)) < 1e-14


def numpy_twin(orc):
    rng = np.random.default_rng(10)
    for case in CASES:
        for d in (1, 4, 8):
            Nq, Nk = case["Nq"], case["Nk"]
            q = _rand(1, 2, Nq, d, rng=rng)
            k = _rand(1, 2, Nk, d, rng=rng)
            v = _rand(1, 2, Nk, d, rng=rng)
            scale = 0.5 / math.sqrt(d)
            o, lse = orc.attention(q, k, v, scale=scale, **_kw(case))
            allowed = _twin_mask(case)
            for h in range(2):
                to, tl = twin.attention(q[0, h], k[0, h], v[0, h], scale, allowed)
                assert np.max(np.abs(o[0, h] - to)) < 1e-12, (case, d)
                assert np.max(np.abs(lse[0, h] - tl)) < 1e-12, (case, d)


def sdpa_fp64(orc):
    import torch
    import torch.nn.functional as F

    rng = np.random.default_rng(11)
    for case in CASES:
        Nq, Nk, d = case["Nq"], case["Nk"], 8
        q = _rand(2, 3, Nq, d, rng=rng)
        k = _rand(2, 3, Nk, d, rng=rng)
        v = _rand(2, 3, Nk, d, rng=rng)
        scale = 1 / math.sqrt(d)
        o, _ = orc.attention(q, k, v, scale=scale, **_kw(case))
        tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
        m = case["mask_kind"]
        if m == "none":
            ref = F.scaled_dot_product_attention(tq, tk, tv, scale=scale)
        elif m == "causal":
            # explicit top-left lower-triangular boolean mask (True = attend)
            tri = torch.ones(Nq, Nk, dtype=torch.bool).tril()
            ref = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=tri, scale=scale)
        else:
            am = torch.from_numpy(_twin_mask(case))
            ref = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=am, scale=scale)
        assert np.max(np.abs(o - ref.numpy())) < 1e-12, case


def invariants(orc):
    rng = np.random.default_rng(12)
    d = 6
    for case in CASES:
        Nq, Nk = case["Nq"], case["Nk"]
        kw = _kw(case)
        q = _rand(1, 1, Nq, d, rng=rng)
        k = _rand(1, 1, Nk, d, rng=rng)
        v = _rand(1, 1, Nk, d, rng=rng)
        v2 = _rand(1, 1, Nk, d, rng=rng)
        s = 0.8
        o, lse = orc.attention(q, k, v, scale=s, **kw)
        # shifting every key by u leaves o alone and shifts lse_i by s * q_i . u
        u = rng.standard_normal(d)
        o_u, lse_u = orc.attention(q, k + u, v, scale=s, **kw)
        assert np.max(np.abs(o_u - o)) < 1e-12, case
        assert np.max(np.abs(lse_u - lse - s * (q[0, 0] @ u))) < 1e-12, case
        # linear in V
        o2, _ = orc.attention(q, k, v2, scale=s, **kw)
        o3, _ = orc.attention(q, k, 2.0 * v - 3.0 * v2, scale=s, **kw)
        assert np.max(np.abs(o3 - (2.0 * o - 3.0 * o2))) < 1e-12, case
    # NONE is invariant under a joint permutation of the keys and values
    Nq, Nk = 17, 29
    q = _rand(1, 1, Nq, d, rng=rng)
    k = _rand(1, 1, Nk, d, rng=rng)
    v = _rand(1, 1, Nk, d, rng=rng)
    perm = rng.permutation(Nk)
    o, lse = orc.attention(q, k, v, scale=0.9, mask_kind="none")
    op, lp = orc.attention(q, k[:, :, perm], v[:, :, perm], scale=0.9, mask_kind="none")
    assert np.max(np.abs(op - o)) < 1e-12 and np.max(np.abs(lp - lse)) < 1e-12
    # causal row i == unmasked attention of query i over the first i+1 keys
    N = 23
    q = _rand(1, 1, N, d, rng=rng)
    k = _rand(1, 1, N, d, rng=rng)
    v = _rand(1, 1, N, d, rng=rng)
    oc, lc = orc.attention(q, k, v, scale=0.6, mask_kind="causal")
    for i in (0, 1, 11, N - 1):
        on, ln = orc.attention(q[:, :, i:i + 1], k[:, :, :i + 1], v[:, :, :i + 1], scale=0.6,
                               mask_kind="none")
        assert np.max(np.abs(on[0, 0, 0] - oc[0, 0, i])) < 1e-12
        assert abs(ln[0, 0, 0] - lc[0, 0, i]) < 1e-12
    # scale -> 0 gives the plain mean over the allowed set
    o0, l0 = orc.attention(q, k, v, scale=0.0, mask_kind="none")
    assert np.max(np.abs(o0[0, 0] - v[0, 0].mean(axis=0))) < 1e-13
    assert np.max(np.abs(l0 - math.log(N))) < 1e-13


def wrap_equals_pad_clamp(orc):
    """Issue #142's recipe: circularly pad Q, K, V by (k//2)*dilation, run clamped
    NA on the padded grid, crop. It must equal the wrap mode on random inputs."""
    rng = np.random.default_rng(13)
    for (gh, gw, win, dil) in ((7, 7, 3, 1), (6, 9, 5, 1), (9, 8, 3, 2), (5, 5, 5, 1)):
        d = 4
        x = [rng.standard_normal((gh, gw, d)) for _ in range(3)]
        p = (win // 2) * dil
        padded = [np.pad(t, ((p, p), (p, p), (0, 0)), mode="wrap") for t in x]
        PH, PW = gh + 2 * p, gw + 2 * p

        def flat(t, h, w):
            return t.reshape(1, 1, h * w, d)

        ow, lw = orc.attention(*(flat(t, gh, gw) for t in x), scale=0.7, mask_kind="wrap",
                               window=win, dilation=dil, grid=(gh, gw))
        oc, lc = orc.attention(*(flat(t, PH, PW) for t in padded), scale=0.7, mask_kind="clamp",
                               window=win, dilation=dil, grid=(PH, PW))
        oc = oc.reshape(PH, PW, d)[p:p + gh, p:p + gw].reshape(1, 1, gh * gw, d)
        lc = lc.reshape(PH, PW)[p:p + gh, p:p + gw].reshape(1, 1, gh * gw)
        assert np.max(np.abs(oc - ow)) < 1e-12, (gh, gw, win, dil)
        assert np.max(np.abs(lc - lw)) < 1e-12, (gh, gw, win, dil)


def one_axis_wrap_pad_clamp(orc):
    """Issue #142's recipe along one axis only: circularly pad that axis by
    (k_axis // 2) * dilation, run clamped NA on the padded grid, crop. It must
    equal NA that wraps that axis and clamps the other."""
    rng = np.random.default_rng(17)
    for (gh, gw, kh, kw, dil, axis) in ((7, 9, 3, 5, 1, 0), (7, 9, 5, 3, 1, 1), (9, 8, 3, 3, 2, 0),
                                        (6, 11, 3, 5, 2, 1), (5, 12, 1, 7, 1, 1)):
        d = 4
        x = [rng.standard_normal((gh, gw, d)) for _ in range(3)]
        ph = (kh // 2) * dil if axis == 0 else 0
        pw = (kw // 2) * dil if axis == 1 else 0
        padded = [np.pad(t, ((ph, ph), (pw, pw), (0, 0)), mode="wrap") for t in x]
        PH, PW = gh + 2 * ph, gw + 2 * pw

        def flat(t, h, w):
            return t.reshape(1, 1, h * w, d)

        ow, lw = orc.attention(*(flat(t, gh, gw) for t in x), scale=0.6, mask_kind="clamp",
                               window=(kh, kw), dilation=dil, grid=(gh, gw),
                               wrap=(axis == 0, axis == 1))
        oc, lc = orc.attention(*(flat(t, PH, PW) for t in padded), scale=0.6, mask_kind="clamp",
                               window=(kh, kw), dilation=dil, grid=(PH, PW))
        oc = oc.reshape(PH, PW, d)[ph:ph + gh, pw:pw + gw].reshape(1, 1, gh * gw, d)
        lc = lc.reshape(PH, PW)[ph:ph + gh, pw:pw + gw].reshape(1, 1, gh * gw)
        assert np.max(np.abs(oc - ow)) < 1e-12, (gh, gw, kh, kw, dil, axis)
        assert np.max(np.abs(lc - lw)) < 1e-12, (gh, gw, kh, kw, dil, axis)


def axis_windows_by_hand(orc):
    def keys(i, grid, window, wrap=False):
        n = grid[0] * grid[1]
        return {j for j in range(n)
                if orc.allowed(i, j, Nq=n, Nk=n, mask_kind="clamp", window=window, wrap=wrap,
                               grid=grid)}

    def tok(y, x, w):
        return y * w + x

    g = (5, 7)
    # window 3 rows x 5 columns, clamp: (0,0) -> rows {0,1,2} x cols {0..4};
    # (4,6) -> rows {2,3,4} x cols {2..6}; (2,3) -> rows {1,2,3} x cols {1..5}
    assert keys(tok(0, 0, 7), g, (3, 5)) == {tok(y, x, 7) for y in (0, 1, 2) for x in range(5)}
    assert keys(tok(4, 6, 7), g, (3, 5)) == {tok(y, x, 7) for y in (2, 3, 4) for x in range(2, 7)}
    assert keys(tok(2, 3, 7), g, (3, 5)) == {tok(y, x, 7) for y in (1, 2, 3) for x in range(1, 6)}
    # window 5 rows x 1 column: a column of the grid, clamped
    assert keys(tok(0, 2, 7), g, (5, 1)) == {tok(y, 2, 7) for y in range(5)}
    # rows wrap, columns clamp, window 3 x 3: (0,0) -> rows {4,0,1} x cols {0,1,2}
    assert keys(tok(0, 0, 7), g, (3, 3), (True, False)) == \
        {tok(y, x, 7) for y in (4, 0, 1) for x in (0, 1, 2)}
    # rows clamp, columns wrap, window 3 x 5: (0,6) -> rows {0,1,2} x cols {4,5,6,0,1}
    assert keys(tok(0, 6, 7), g, (3, 5), (False, True)) == \
        {tok(y, x, 7) for y in (0, 1, 2) for x in (4, 5, 6, 0, 1)}


def one_d_closed_form(orc):
    """A 1 x N grid with window (1, k): key j is allowed for query i iff it lies in
    [s, s + k), s = min(max(i - k//2, 0), N - k) (clamp), or iff its circular
    distance to i is at most k//2 (wrap)."""
    for (N, k) in ((11, 3), (16, 5), (9, 9), (13, 1)):
        for i in range(N):
            s0 = min(max(i - k // 2, 0), N - k)
            for j in range(N):
                clamp = orc.allowed(i, j, Nq=N, Nk=N, mask_kind="clamp", window=(1, k), grid=(1, N))
                wrap = orc.allowed(i, j, Nq=N, Nk=N, mask_kind="clamp", window=(1, k), grid=(1, N),
                                   wrap=(False, True))
                assert clamp == (s0 <= j < s0 + k), (N, k, i, j)
                dist = min((j - i) % N, (i - j) % N)
                assert wrap == (dist <= k // 2), (N, k, i, j)
    # dilated, clamp: the keys of i's residue class mod dl, k of them, the
    # window of positions inside that class shifted inward at its ends
    for (N, k, dl) in ((20, 3, 3), (17, 5, 2), (9, 3, 3)):
        for i in range(N):
            members = list(range(i % dl, N, dl))
            a0 = min(max(members.index(i) - k // 2, 0), len(members) - k)
            want = set(members[a0:a0 + k])
            got = {j for j in range(N)
                   if orc.allowed(i, j, Nq=N, Nk=N, mask_kind="clamp", window=(1, k),
                                  dilation=dl, grid=(1, N))}
            assert got == want, (N, k, dl, i)



def _vol_keys(orc, i, grid, window, wrap=False, dilation=1):
    n = grid[0] * grid[1] * grid[2]
    return {j for j in range(n)
            if orc.allowed(i, j, Nq=n, Nk=n, mask_kind="clamp", window=window, wrap=wrap,
                           dilation=dilation, grid=grid)}


def na3d_windows_by_hand(orc):
    def tok(t, y, x, g):
        return (t * g[1] + y) * g[2] + x

    g = (4, 5, 6)
    # clamp, window 3 on every axis: corner (0,0,0) -> {0,1,2} x {0,1,2} x {0,1,2};
    # (3,4,5) -> {1,2,3} x {2,3,4} x {3,4,5}
    assert _vol_keys(orc, tok(0, 0, 0, g), g, 3) == \
        {tok(t, y, x, g) for t in (0, 1, 2) for y in (0, 1, 2) for x in (0, 1, 2)}
    assert _vol_keys(orc, tok(3, 4, 5, g), g, 3) == \
        {tok(t, y, x, g) for t in (1, 2, 3) for y in (2, 3, 4) for x in (3, 4, 5)}
    # depth wraps, rows and columns clamp, window (3, 1, 5): (0,2,0) -> depth {3,0,1},
    # row {2}, columns {0..4}
    assert _vol_keys(orc, tok(0, 2, 0, g), g, (3, 1, 5), (True, False, False)) == \
        {tok(t, 2, x, g) for t in (3, 0, 1) for x in range(5)}
    # depth clamps, rows and columns wrap, window 3: (2,0,5) -> depth {1,2,3},
    # rows {4,0,1}, columns {4,5,0}
    assert _vol_keys(orc, tok(2, 0, 5, g), g, 3, (False, True, True)) == \
        {tok(t, y, x, g) for t in (1, 2, 3) for y in (4, 0, 1) for x in (4, 5, 0)}
    # dilation 2 on a 4 x 6 x 6 volume, window (1, 3, 3), clamp: (1,5,0) -> depth {1},
    # rows of residue 1 {1,3,5}, columns of residue 0 {0,2,4}
    g2 = (4, 6, 6)
    assert _vol_keys(orc, tok(1, 5, 0, g2), g2, (1, 3, 3), False, 2) == \
        {tok(1, y, x, g2) for y in (1, 3, 5) for x in (0, 2, 4)}


def _axis_closed_form(qc, kc, G, k, wrap, dl):
    """One axis, from closed forms: wrap -> circular distance a multiple of dl and at
    most dl*(k//2); clamp -> same residue mod dl and the class index inside the
    interval [s, s + k), s = min(max(a - k//2, 0), L - k), L the class size."""
    if wrap:
        for t in range(-(k // 2), k // 2 + 1):
            if (qc + dl * t - kc) % G == 0:
                return True
        return False
    if qc % dl != kc % dl:
        return False
    L = len(range(qc % dl, G, dl))
    s = min(max(qc // dl - k // 2, 0), L - k)
    return s <= kc // dl < s + k


def na3d_closed_form(orc):
    for (g, win, wrap, dl) in (((3, 4, 5), (3, 3, 3), (False, False, False), 1),
                               ((4, 3, 5), (3, 1, 5), (True, False, True), 1),
                               ((5, 4, 3), (5, 3, 1), (False, True, False), 1),
                               ((6, 4, 6), (3, 1, 3), (True, False, False), 2)):
        n = g[0] * g[1] * g[2]
        for i in range(n):
            qc = (i // (g[1] * g[2]), (i // g[2]) % g[1], i % g[2])
            want = set()
            for j in range(n):
                kc = (j // (g[1] * g[2]), (j // g[2]) % g[1], j % g[2])
                if all(_axis_closed_form(qc[a], kc[a], g[a], win[a], wrap[a], dl)
                       for a in range(3)):
                    want.add(j)
            assert _vol_keys(orc, i, g, win, wrap, dl) == want, (g, win, wrap, dl, i)


def na3d_flat_is_na2d(orc):
    rng = np.random.default_rng(19)
    for (gh, gw, kh, kw, wrap, dl) in ((6, 7, 3, 5, (False, True), 1), (8, 8, 3, 3, (True, True), 2),
                                       (5, 9, 5, 1, (False, False), 1)):
        n, d = gh * gw, 5
        q, k, v = (_rand(1, 2, n, d, rng=rng) for _ in range(3))
        o2, l2 = orc.attention(q, k, v, scale=0.7, mask_kind="clamp", window=(kh, kw), wrap=wrap,
                               dilation=dl, grid=(gh, gw))
        o3, l3 = orc.attention(q, k, v, scale=0.7, mask_kind="clamp", window=(1, kh, kw),
                               wrap=(False,) + wrap, dilation=dl, grid=(1, gh, gw))
        assert np.array_equal(o2, o3) and np.array_equal(l2, l3)


def na3d_wrap_pad_clamp(orc):
    rng = np.random.default_rng(23)
    for (g, win, wrap, dl) in (((5, 6, 7), (3, 3, 3), (True, True, False), 1),
                               ((6, 5, 5), (3, 5, 3), (True, False, True), 1),
                               ((8, 6, 7), (3, 1, 3), (True, False, True), 2)):
        d = 3
        x = [rng.standard_normal(g + (d,)) for _ in range(3)]
        pads = [((win[a] // 2) * dl if wrap[a] else 0) for a in range(3)]
        padded = [np.pad(t, [(p_, p_) for p_ in pads] + [(0, 0)], mode="wrap") for t in x]
        G = tuple(g[a] + 2 * pads[a] for a in range(3))
        ow, lw = orc.attention(*(t.reshape(1, 1, -1, d) for t in x), scale=0.5, mask_kind="clamp",
                               window=win, wrap=wrap, dilation=dl, grid=g)
        oc, lc = orc.attention(*(t.reshape(1, 1, -1, d) for t in padded), scale=0.5,
                               mask_kind="clamp", window=win, dilation=dl, grid=G)
        crop = tuple(slice(pads[a], pads[a] + g[a]) for a in range(3))
        oc = oc.reshape(G + (d,))[crop].reshape(1, 1, -1, d)
        lc = lc.reshape(G)[crop].reshape(1, 1, -1)
        assert np.max(np.abs(oc - ow)) < 1e-12, (g, win, wrap, dl)
        assert np.max(np.abs(lc - lw)) < 1e-12, (g, win, wrap, dl)



def causal_bottom_right(orc):
    rng = np.random.default_rng(29)
    d = 6
    # Nq == Nk: the same allowed sets as top-left
    q, k, v = (_rand(1, 2, 19, d, rng=rng) for _ in range(3))
    o1, l1 = orc.attention(q, k, v, scale=0.6, mask_kind="causal")
    o2, l2 = orc.attention(q, k, v, scale=0.6, mask_kind="causal_br")
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # Nq < Nk: row i is unmasked attention of query i over keys 0 .. i + Nk - Nq
    Nq, Nk = 9, 25
    q = _rand(1, 1, Nq, d, rng=rng)
    k, v = (_rand(1, 1, Nk, d, rng=rng) for _ in range(2))
    o, lse = orc.attention(q, k, v, scale=0.7, mask_kind="causal_br")
    for i in range(Nq):
        n = i + Nk - Nq + 1
        on, ln = orc.attention(q[:, :, i:i + 1], k[:, :, :n], v[:, :, :n], scale=0.7, mask_kind="none")
        assert np.max(np.abs(on[0, 0, 0] - o[0, 0, i])) < 1e-12 and abs(ln[0, 0, 0] - lse[0, 0, i]) < 1e-12
    # Nq > Nk: the first Nq - Nk rows see no key; the others see keys 0 .. i - (Nq - Nk)
    Nq, Nk = 20, 7
    q = _rand(1, 1, Nq, d, rng=rng)
    k, v = (_rand(1, 1, Nk, d, rng=rng) for _ in range(2))
    o, lse = orc.attention(q, k, v, scale=0.7, mask_kind="causal_br")
    for i in range(Nq):
        n = i - (Nq - Nk) + 1
        if n <= 0:
            assert np.all(o[0, 0, i] == 0.0) and lse[0, 0, i] == -np.inf, i
        else:
            on, ln = orc.attention(q[:, :, i:i + 1], k[:, :, :n], v[:, :, :n], scale=0.7,
                                   mask_kind="none")
            assert np.max(np.abs(on[0, 0, 0] - o[0, 0, i])) < 1e-12, i
    # torch SDPA (fp64, math) with the explicit bottom-right mask, Nq < Nk
    import torch
    import torch.nn.functional as F
    Nq, Nk = 13, 30
    q = _rand(2, 2, Nq, 8, rng=rng)
    k, v = (_rand(2, 2, Nk, 8, rng=rng) for _ in range(2))
    o, _ = orc.attention(q, k, v, scale=0.35, mask_kind="causal_br")
    am = torch.ones(Nq, Nk, dtype=torch.bool).tril(diagonal=Nk - Nq)
    ref = F.scaled_dot_product_attention(*(torch.from_numpy(x) for x in (q, k, v)), attn_mask=am,
                                         scale=0.35)
    assert np.max(np.abs(o - ref.numpy())) < 1e-12


BWD_CASES = [
    dict(mask_kind="none", Nq=13, Nk=21),
    dict(mask_kind="causal", Nq=17, Nk=17),
    dict(mask_kind="causal", Nq=9, Nk=20),
    dict(mask_kind="causal_br", Nq=9, Nk=20),
    dict(mask_kind="clamp", Nq=30, Nk=30, window=(3, 5), grid=(5, 6)),
    dict(mask_kind="wrap", Nq=36, Nk=36, window=3, grid=(6, 6), dilation=2),
    dict(mask_kind="clamp", Nq=48, Nk=48, window=(3, 3, 1), grid=(3, 4, 4), wrap=(True, False, True)),
    dict(mask_kind="clamp", Nq=72, Nk=72, window=(1, 3, 3), grid=(2, 6, 6), wrap=(False, True, False),
         dilation=2),
]


def _bwd_inputs(case, rng, d=6):
    B, H = 1, 2
    shapes = [(B, H, case["Nq"], d), (B, H, case["Nk"], d), (B, H, case["Nk"], d),
              (B, H, case["Nq"], d)]
    return [rng.standard_normal(sh) for sh in shapes]


def bwd_autograd_fp64(orc):
    import torch
    rng = np.random.default_rng(21)
    for case in BWD_CASES:
        q, k, v, g = _bwd_inputs(case, rng)
        dq, dk, dv = orc.attention_bwd(q, k, v, g, scale=0.45, **_kw(case))
        t = [torch.tensor(x, requires_grad=True) for x in (q, k, v)]
        allowed = torch.from_numpy(_twin_mask(case))
        sc = (0.45 * t[0] @ t[1].transpose(-1, -2)).masked_fill(~allowed, float("-inf"))
        o = torch.softmax(sc, dim=-1) @ t[2]
        (o * torch.from_numpy(g)).sum().backward()
        for name, ref, got in (("dq", t[0].grad, dq), ("dk", t[1].grad, dk), ("dv", t[2].grad, dv)):
            err = np.max(np.abs(ref.numpy() - got))
            assert err < 1e-12, (case, name, err)


def bwd_finite_differences(orc):
    rng = np.random.default_rng(22)
    h = 1e-5
    for case in BWD_CASES:
        q, k, v, g = _bwd_inputs(case, rng)
        grads = orc.attention_bwd(q, k, v, g, scale=0.45, **_kw(case))
        for which in range(3):
            e = rng.standard_normal(grads[which].shape)

            def loss(eps):
                x = [q, k, v]
                x[which] = x[which] + eps * e
                o, _ = orc.attention(*x, scale=0.45, **_kw(case))
                return float(np.sum(o * g))

            fd = (loss(h) - loss(-h)) / (2 * h)
            an = float(np.sum(grads[which] * e))
            assert abs(fd - an) < 1e-7 * max(1.0, abs(an)), (case, which, fd, an)


def bwd_invariants(orc):
    rng = np.random.default_rng(23)
    for case in BWD_CASES:
        q, k, v, g = _bwd_inputs(case, rng)
        dq, dk, dv = orc.attention_bwd(q, k, v, g, scale=0.45, **_kw(case))
        # every query row has a non-empty allowed set in these cases
        assert np.max(np.abs(dk.sum(axis=2))) < 1e-12, case
        assert np.max(np.abs(dv.sum(axis=2) - g.sum(axis=2))) < 1e-12, case


def row_subset_matches_full(orc):
    rng = np.random.default_rng(14)
    q = _rand(2, 2, 33, 8, rng=rng)
    k = _rand(2, 2, 33, 8, rng=rng)
    v = _rand(2, 2, 33, 8, rng=rng)
    o, lse = orc.attention(q, k, v, scale=0.4, mask_kind="causal")
    rows = np.array([0, 5, 32, 33, 70, 131])
    os_, ls = orc.attention_rows(q, k, v, rows, scale=0.4, mask_kind="causal")
    assert np.array_equal(os_, o.reshape(-1, 8)[rows])
    assert np.array_equal(ls, lse.reshape(-1)[rows])


def all_checks(goldens):
    """(name, callable(orc)) for every check, goldens = (wrap_printed, clamp_by_hand)."""
    wrap_printed, clamp_by_hand = goldens
    return [
        ("golden_wrap_example", lambda o: golden_wrap_example(o, wrap_printed)),
        ("golden_clamp_by_hand", lambda o: golden_clamp_by_hand(o, clamp_by_hand)),
        ("window_sets_by_hand", window_sets_by_hand),
        ("constant_v", constant_v),
        ("zero_qk_means", zero_qk_means),
        ("single_key", single_key),
        ("numpy_twin", numpy_twin),
        ("sdpa_fp64", sdpa_fp64),
        ("invariants", invariants),
        ("wrap_equals_pad_clamp", wrap_equals_pad_clamp),
        ("one_axis_wrap_pad_clamp", one_axis_wrap_pad_clamp),
        ("axis_windows_by_hand", axis_windows_by_hand),
        ("one_d_closed_form", one_d_closed_form),
        ("na3d_windows_by_hand", na3d_windows_by_hand),
        ("na3d_closed_form", na3d_closed_form),
        ("na3d_flat_is_na2d", na3d_flat_is_na2d),
        ("na3d_wrap_pad_clamp", na3d_wrap_pad_clamp),
        ("causal_bottom_right", causal_bottom_right),
        ("bwd_autograd_fp64", bwd_autograd_fp64),
        ("bwd_finite_differences", bwd_finite_differences),
        ("bwd_invariants", bwd_invariants),
        ("row_subset_matches_full", row_subset_matches_full),
    ]
