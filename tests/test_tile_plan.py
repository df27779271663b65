"""Host build of the kernel's tile planning against the oracle's masks (CPU).

For every Q tile (128 query rows) and K/V tile (128 keys) the kernel decides:
skip (no allowed pair), unmasked (every pair allowed) or masked. Checked here
against the allowed-set matrix of the numpy oracle twin: a skipped tile holds
no allowed pair and an unmasked one holds only allowed pairs; with dilation 1
a visited tile also holds at least one (no wasted tiles), while dilated
neighbourhoods may visit a few fully masked tiles (a superset test).
"""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

from oracle import reference_np as twin

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KIND = {"none": 0, "causal": 1, "clamp": 2, "wrap": 2}


@pytest.fixture(scope="module")
def plan(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    out = str(tmp_path_factory.mktemp("plan") / "tile_plan.so")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O1", "-std=c++17",
                    "-shared", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(ROOT, "exact_attention_69_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "host", "tile_plan.cu"), "-o", out], check=True)
    lib = ctypes.CDLL(out)
    lib.tile_class_host.argtypes = [ctypes.c_int] * 12
    lib.tile_class_host.restype = ctypes.c_int
    lib.decode_task_host.argtypes = [ctypes.c_int] * 6 + [ctypes.POINTER(ctypes.c_int)]
    lib.na_bits_host.argtypes = [ctypes.c_int] * 10 + [ctypes.POINTER(ctypes.c_uint)]
    lib.tile_class3_host.argtypes = [ctypes.c_int] * 11
    lib.tile_class3_host.restype = ctypes.c_int
    lib.na3_bits_host.argtypes = [ctypes.c_int] * 11 + [ctypes.POINTER(ctypes.c_uint)]
    lib.na_key_bits_host.argtypes = [ctypes.c_int] * 11 + [ctypes.POINTER(ctypes.c_uint)]
    lib.band_host.argtypes = [ctypes.c_int] * 10 + [ctypes.POINTER(ctypes.c_int)]
    lib.twin_host.argtypes = [ctypes.c_int] * 11
    lib.twin_host.restype = ctypes.c_int
    return lib


CASES = [
    ("none", 300, 300, None, 0), ("none", 129, 1000, None, 0), ("none", 1, 1, None, 0),
    ("causal", 700, 700, None, 0), ("causal", 300, 1000, None, 0), ("causal", 1000, 300, None, 0),
    ("causal", 2048, 2048, None, 0),
    ("clamp", 4096, 4096, (64, 64), 7), ("wrap", 4096, 4096, (64, 64), 7),
    ("clamp", 25, 25, (5, 5), 3), ("wrap", 25, 25, (5, 5), 3),
    ("clamp", 400, 400, (20, 20), 5), ("wrap", 400, 400, (20, 20), 5),
    ("clamp", 1200, 1200, (24, 50), 7), ("wrap", 1200, 1200, (24, 50), 7),
    ("clamp", 4800, 4800, (30, 160), 9), ("wrap", 4800, 4800, (30, 160), 9),
    ("wrap", 1521, 1521, (39, 39), 39), ("clamp", 1521, 1521, (39, 39), 1),
]


DILATED = [
    ("clamp", 4096, 4096, (64, 64), 7, 2), ("wrap", 4096, 4096, (64, 64), 7, 3),
    ("clamp", 400, 400, (20, 20), 3, 4), ("wrap", 400, 400, (20, 20), 5, 4),
    ("clamp", 1200, 1200, (24, 50), 3, 7), ("wrap", 1200, 1200, (24, 50), 5, 4),
    ("clamp", 64, 64, (8, 8), 3, 2), ("wrap", 64, 64, (8, 8), 3, 2),
]

# per-axis windows and wrap: (grid, (k_rows, k_cols), (wrap_rows, wrap_cols), dilation)
AXES = [
    ((64, 64), (7, 3), (True, False), 1), ((64, 64), (3, 9), (False, True), 1),
    ((20, 60), (5, 11), (False, False), 1), ((20, 60), (1, 9), (True, True), 1),
    ((1, 4096), (1, 31), (False, False), 1), ((1, 4096), (1, 31), (False, True), 1),
    ((1, 700), (1, 9), (False, False), 3), ((48, 40), (5, 3), (True, False), 4),
    ((30, 160), (9, 5), (False, True), 2), ((13, 29), (3, 7), (True, False), 1),
]


def _na_args(mask, window, wrap_axes):
    kh, kw = (window, window) if isinstance(window, int) else window
    if wrap_axes is None:
        wrap_axes = (mask == "wrap", mask == "wrap")
    return kh, kw, int(wrap_axes[0]), int(wrap_axes[1])


@pytest.mark.parametrize("mask,Nq,Nk,grid,window,dilation,wrap_axes",
                         [c + (1, None) for c in CASES] + [c + (None,) for c in DILATED] +
                         [("clamp", g[0] * g[1], g[0] * g[1], g, win, dil, wr)
                          for (g, win, wr, dil) in AXES])
def test_tile_classes_match_oracle_mask(plan, mask, Nq, Nk, grid, window, dilation, wrap_axes):
    allowed = twin.mask_matrix(Nq, Nk, mask, window, dilation, grid, wrap_axes)
    kh, kw, wh, ww = _na_args(mask, window, wrap_axes)
    gh, gw = grid if grid else (0, 0)
    n_kv = -(-Nk // 128)
    visited = wasted = 0
    for q0 in range(0, Nq, 128):
        rows = allowed[q0:min(q0 + 128, Nq)]
        for j in range(n_kv):
            block = rows[:, j * 128:min(j * 128 + 128, Nk)]
            c = plan.tile_class_host(KIND[mask], q0, j, Nq, Nk, gh, gw, kh, kw, dilation, wh, ww)
            assert c in (0, 1, 2)
            if c == 0:
                assert not block.any(), (q0, j)
            else:
                visited += 1
                wasted += not block.any()
            if dilation == 1:
                assert (c != 0) == bool(block.any()), (q0, j, c)
            if c == 1:
                assert block.all() and block.shape[1] == 128, (q0, j)
    assert wasted <= visited // 2 + 1, (visited, wasted)


@pytest.mark.parametrize("q_tiles", [1, 2])
@pytest.mark.parametrize("mask", ["none", "causal"])
def test_tasks_cover_every_q_tile_once(plan, mask, q_tiles):
    """Tasks of one Q tile or of a pair: every 128-row Q tile of every head is
    in exactly one task (a pair's second tile only if it starts below Nq)."""
    B, H, Nq = 3, 5, 1000
    span = 128 * q_tiles
    n_tasks = -(-Nq // span)
    seen = set()
    out = (ctypes.c_int * 4)()
    for t in range(B * H * n_tasks):
        plan.decode_task_host(KIND[mask], t, B, H, Nq, q_tiles, out)
        tiles = [out[2]] + ([out[2] + 128] if out[3] else [])
        for q0 in tiles:
            key = (out[0], out[1], q0)
            assert key not in seen
            seen.add(key)
    assert seen == {(b, h, 128 * i) for b in range(B) for h in range(H) for i in range(-(-Nq // 128))}
    if mask == "causal":  # longest tasks (largest row offset) come first
        plan.decode_task_host(1, 0, B, H, Nq, q_tiles, out)
        assert out[2] == span * (n_tasks - 1)


@pytest.mark.parametrize("mode,gh,gw,window,dilation", [
    ("clamp", 64, 64, 7, 1), ("wrap", 64, 64, 7, 1), ("clamp", 5, 5, 3, 1), ("wrap", 5, 5, 3, 1),
    ("clamp", 13, 29, 7, 1), ("wrap", 13, 29, 7, 1), ("wrap", 24, 50, 9, 1),
    ("clamp", 30, 160, 9, 1), ("wrap", 39, 39, 39, 1), ("clamp", 12, 20, 1, 1),
    ("clamp", 8, 8, 3, 2), ("wrap", 8, 8, 3, 2), ("clamp", 20, 20, 5, 3), ("wrap", 20, 20, 5, 4),
    ("clamp", 13, 29, 3, 4), ("wrap", 13, 29, 3, 4), ("clamp", 64, 64, 7, 2), ("wrap", 64, 64, 7, 9),
    ("wrap", 21, 21, 7, 3), ("clamp", 21, 35, 3, 7)] +
    [("axes", g[0], g[1], (win, wr), dil) for (g, win, wr, dil) in AXES])
def test_in_tile_mask_bits_match_oracle_mask(plan, mode, gh, gw, window, dilation):
    """The kernel's in-tile neighbourhood mask, bit for bit, against the oracle
    twin's allowed-set matrix, for every query and every K/V tile."""
    N = gh * gw
    if mode == "axes":
        (window, wrap_axes), mode = window, "clamp"
    else:
        wrap_axes = None
    allowed = twin.mask_matrix(N, N, mode, window, dilation, (gh, gw), wrap_axes)
    kh, kw, wh, ww = _na_args(mode, window, wrap_axes)
    out = (ctypes.c_uint * 4)()
    rng = np.random.default_rng(0)
    queries = range(N) if N <= 1600 else rng.choice(N, 400, replace=False)
    for q in queries:
        for k0 in range(0, N, 128):
            plan.na_bits_host(int(q), k0, N, gh, gw, kh, kw, dilation, wh, ww, out)
            bits = np.array([(out[i >> 5] >> (i & 31)) & 1 for i in range(128)], dtype=bool)
            ref = np.zeros(128, dtype=bool)
            n = min(128, N - k0)
            ref[:n] = allowed[q, k0:k0 + n]
            assert np.array_equal(bits, ref), (q, k0)


# volumes: (grid (depth, rows, cols), window per axis, wrap per axis, dilation)
VOLUMES = [
    ((16, 16, 16), (5, 5, 5), (True, True, False), 1), ((16, 16, 16), (5, 5, 5), (False, False, False), 1),
    ((20, 15, 18), (5, 3, 7), (False, True, True), 1), ((8, 8, 8), (3, 3, 3), (True, True, True), 2),
    ((6, 10, 30), (1, 3, 9), (False, False, True), 3), ((12, 1, 40), (3, 1, 5), (True, False, False), 1),
    ((4, 20, 3), (3, 7, 3), (False, True, False), 1), ((9, 9, 9), (9, 9, 9), (True, False, True), 1),
]


def _wrap_bits(wrap):
    return (1 if wrap[2] else 0) | (2 if wrap[1] else 0) | (4 if wrap[0] else 0)


@pytest.mark.parametrize("grid,window,wrap,dilation", VOLUMES)
def test_volume_tile_classes_and_bits_match_oracle_mask(plan, grid, window, wrap, dilation):
    N = grid[0] * grid[1] * grid[2]
    allowed = twin.mask_matrix(N, N, "clamp", window, dilation, grid, wrap)
    args = (N,) + tuple(grid) + tuple(window) + (dilation, _wrap_bits(wrap))
    n_kv = -(-N // 128)
    visited = wasted = 0
    for q0 in range(0, N, 128):
        rows = allowed[q0:min(q0 + 128, N)]
        for j in range(n_kv):
            block = rows[:, j * 128:min(j * 128 + 128, N)]
            c = plan.tile_class3_host(q0, j, *args)
            assert c in (0, 2), (q0, j, c)
            if c == 0:
                assert not block.any(), (q0, j)
            else:
                visited += 1
                wasted += not block.any()
            if dilation == 1:
                assert (c != 0) == bool(block.any()), (q0, j, c)
    assert wasted <= visited // 2 + 1, (visited, wasted)
    out = (ctypes.c_uint * 4)()
    rng = np.random.default_rng(1)
    queries = range(N) if N <= 1000 else rng.choice(N, 300, replace=False)
    for q in queries:
        for k0 in range(0, N, 128):
            plan.na3_bits_host(int(q), k0, *args, out)
            bits = np.array([(out[i >> 5] >> (i & 31)) & 1 for i in range(128)], dtype=bool)
            ref = np.zeros(128, dtype=bool)
            n = min(128, N - k0)
            ref[:n] = allowed[q, k0:k0 + n]
            assert np.array_equal(bits, ref), (q, k0)


KEY_BITS = [((8, 8), (3, 3), (False, False), 1), ((8, 8), (3, 3), (True, True), 1),
            ((13, 29), (5, 7), (False, True), 1), ((20, 12), (3, 5), (True, False), 2),
            ((24, 50), (5, 5), (False, False), 4), ((1, 700), (1, 9), (False, True), 3),
            ((6, 10, 12), (3, 5, 3), (True, False, True), 1), ((8, 8, 8), (3, 3, 3), (False, True, False), 2),
            ((64, 64), (7, 7), (False, False), 1), ((64, 64), (7, 7), (True, True), 1),
            ((20, 12), (5, 3), (True, False), 1), ((1, 700), (1, 9), (False, False), 1),
            ((39, 39), (39, 39), (True, True), 1), ((5, 5), (5, 5), (False, False), 1),
            ((7, 30), (7, 1), (False, True), 1), ((30, 7), (1, 7), (True, False), 1),
            ((16, 16, 16), (5, 5, 5), (True, True, False), 1), ((5, 9, 7), (5, 3, 7), (False, True, True), 1),
            ((12, 1, 40), (3, 1, 5), (True, False, False), 1), ((3, 5, 7), (3, 5, 7), (False, False, False), 1)]


@pytest.mark.parametrize("grid,window,wrap,dilation", KEY_BITS)
def test_backward_key_bits_match_transposed_oracle_mask(plan, grid, window, wrap, dilation):
    """The dK/dV kernel's per-key mask (which queries of a 128-query tile hold
    the key in their window) equals the oracle twin's column, bit for bit."""
    N = int(np.prod(grid))
    allowed = twin.mask_matrix(N, N, "clamp", window, dilation, grid, wrap)
    if len(grid) == 3:
        g3, w3, bits_w = grid, window, _wrap_bits(wrap)
    else:
        g3, w3 = (0,) + tuple(grid), (1,) + tuple(window)
        bits_w = (1 if wrap[1] else 0) | (2 if wrap[0] else 0)
    out = (ctypes.c_uint * 4)()
    rng = np.random.default_rng(2)
    keys = range(N) if N <= 800 else rng.choice(N, 250, replace=False)
    for kk in keys:
        for q0 in range(0, N, 128):
            plan.na_key_bits_host(q0, int(kk), N, *g3, *w3, dilation, bits_w, out)
            bits = np.array([(out[i >> 5] >> (i & 31)) & 1 for i in range(128)], dtype=bool)
            ref = np.zeros(128, dtype=bool)
            n = min(128, N - q0)
            ref[:n] = allowed[q0:q0 + n, kk]
            assert np.array_equal(bits, ref), (kk, q0)


BANDS = [((64, 64), (7, 7), (False, False), 1), ((64, 64), (7, 7), (True, True), 1),
         ((13, 29), (5, 7), (False, True), 1), ((20, 12), (3, 5), (True, False), 2),
         ((24, 50), (5, 5), (False, False), 4), ((1, 700), (1, 9), (False, True), 3),
         ((1, 4096), (1, 63), (False, False), 1), ((39, 39), (39, 39), (True, True), 1),
         ((5, 5), (3, 3), (True, True), 1),
         ((16, 16, 16), (5, 5, 5), (True, True, False), 1), ((6, 10, 30), (1, 3, 9), (False, False, True), 3),
         ((12, 1, 40), (3, 1, 5), (True, False, False), 1), ((1, 20, 20), (1, 5, 5), (False, True, True), 1),
         ((1, 1, 300), (1, 1, 7), (False, False, True), 2), ((9, 9, 9), (9, 9, 9), (True, False, True), 1)]


def _band_tiles(out):
    return set(range(out[0], out[1])) | set(range(out[2], out[3]))


@pytest.mark.parametrize("grid,window,wrap,dilation", BANDS)
def test_band_holds_every_meeting_tile_both_ways(plan, grid, window, wrap, dilation):
    """The candidate band of a tile (the tiles the kernels visit) holds every tile
    of the other side that shares an allowed pair with it: K/V tiles of a Q tile
    (forward, dQ) and Q tiles of a K/V tile (dK/dV)."""
    N = int(np.prod(grid))
    allowed = twin.mask_matrix(N, N, "clamp", window, dilation, grid, wrap)
    if len(grid) == 3:
        g3, w3, bits_w = grid, window, _wrap_bits(wrap)
    else:
        g3, w3 = (0,) + tuple(grid), (1,) + tuple(window)
        bits_w = (1 if wrap[1] else 0) | (2 if wrap[0] else 0)
    n_t = -(-N // 128)
    pad = np.zeros((n_t * 128, n_t * 128), dtype=bool)
    pad[:N, :N] = allowed
    meets = pad.reshape(n_t, 128, n_t, 128).any(axis=(1, 3))  # [q tile, k tile]
    out = (ctypes.c_int * 4)()
    total = 0
    for t in range(n_t):
        plan.band_host(t * 128, N, *g3, *w3, dilation, bits_w, out)
        band = _band_tiles(out)
        # the second interval may share a tile with the first; iteration skips it
        assert out[0] < out[1] and (out[2] == out[3] or out[0] <= out[2]), list(out)
        assert set(np.nonzero(meets[t])[0]) <= band, (t, list(out))
        assert set(np.nonzero(meets[:, t])[0]) <= band, (t, list(out))
        total += len(band)
    # a band is a narrow superset: no more than the meeting tiles plus a margin
    assert total <= meets.sum() + 4 * n_t, (total, int(meets.sum()))


# The host's twin decision (both softmax warpgroups on one Q tile, its K/V tiles
# in turn) for the twin configurations of the GPU tests and the 64 x 64 grid
# with window 7 of the neighbourhood workloads: twins from 8 active K/V tiles a
# Q tile on (a task from the middle of head 0), counted with the kernel's own
# band and tile tests. The GPU tests read the same flags from ATTN_LOG.
TWIN_DECISIONS = [  # (grid, window, dilation, wrap (per axis), twin)
    ((40, 40), 39, 1, (False, False), 1),
    ((48, 48), 21, 1, (True, False), 1),
    ((32, 32), 9, 2, (False, True), 1),
    ((16, 16, 16), 5, 1, (True, True, False), 1),
    ((12, 14, 10), (7, 7, 3), 1, (False, True, False), 1),
    ((16, 16, 24), 3, 2, (False, False, False), 1),
    ((64, 64), 7, 1, (False, False), 0),
    ((64, 64), 7, 1, (True, True), 0),
]


@pytest.mark.parametrize("grid,window,dilation,wrap,twin_on", TWIN_DECISIONS)
def test_twin_decision(plan, grid, window, dilation, wrap, twin_on):
    N = int(np.prod(grid))
    win = window if isinstance(window, tuple) else (window,) * len(grid)
    if len(grid) == 3:
        g3, w3, bits = grid, win, _wrap_bits(wrap)
    else:
        g3, w3 = (0,) + tuple(grid), (1,) + tuple(win)
        bits = (1 if wrap[1] else 0) | (2 if wrap[0] else 0)
    assert plan.twin_host(1, 2, N, *g3, *w3, dilation, bits) == twin_on
    # the count is of one task's tiles: the decision does not depend on B or H
    assert plan.twin_host(3, 5, N, *g3, *w3, dilation, bits) == twin_on


def _dealt(rnd, cta, G):
    """Causal tasks dealt back and forth: the task of a CTA's round `rnd`."""
    return rnd * G + (G - 1 - cta if rnd & 1 else cta)


@pytest.mark.parametrize("n_tasks,G", [(512, 152), (1, 152), (151, 152), (152, 152), (153, 152),
                                       (305, 152), (1000, 7), (6, 1), (77, 3)])
def test_causal_tasks_dealt_back_and_forth_cover_every_task_once(n_tasks, G):
    """Each CTA takes its round-r task until the first one past n_tasks (the
    kernel stops there): every task is taken once, by one CTA."""
    seen = []
    for c in range(G):
        r = 0
        while _dealt(r, c, G) < n_tasks:
            seen.append(_dealt(r, c, G))
            r += 1
        # once past the end, every later round is too
        assert all(_dealt(rr, c, G) >= n_tasks for rr in range(r, r + 4))
    assert sorted(seen) == list(range(n_tasks))


def test_causal_deal_evens_out_the_lm_shape(plan):
    """B4 H16 N2048 causal over 152 CTAs: a task (a pair of Q tiles) takes as
    many K/V tile steps as its second tile sees; longest first. Dealt back and
    forth, no CTA holds more than 32 steps against 38 for a round robin (the
    mean is 30.3)."""
    B, H, N, G = 4, 16, 2048, 152
    n_tasks = B * H * (N // 256)
    out = (ctypes.c_int * 4)()
    steps = []
    for t in range(n_tasks):
        plan.decode_task_host(1, t, B, H, N, 2, out)
        steps.append((out[2] + 256) // 128)  # K/V tiles of the pair's second Q tile
    assert steps == sorted(steps, reverse=True)
    load_rr = [sum(steps[t] for t in range(c, n_tasks, G)) for c in range(G)]
    load_snake = [0] * G
    for c in range(G):
        r = 0
        while _dealt(r, c, G) < n_tasks:
            load_snake[c] += steps[_dealt(r, c, G)]
            r += 1
    assert max(load_rr) == 38 and max(load_snake) == 32
    assert sum(load_snake) == sum(load_rr) == sum(steps)
