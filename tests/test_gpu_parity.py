"""GPU parity: the sm_103a kernels through the C ABI against the fp64 oracle.

Tolerances: every bf16 output element |o - ref| <= 1e-2 + 1e-2 |ref|, every
log-sum-exp |lse - ref| <= 1e-3. Inputs are the seeded bf16 tensors of
seeded_inputs; the oracle reads the same bf16 values in fp64.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from seeded_inputs import WORKLOADS, make_qkv, make_workload, to_f64

pytestmark = pytest.mark.gpu

ATOL, RTOL, LSE_TOL = 1e-2, 1e-2, 1e-3


@pytest.fixture(scope="module")
def E():
    from exact_attention_69_gb300 import build
    build.build()
    import exact_attention_69_gb300 as E
    return E


def _status_ok(E):
    torch.cuda.synchronize()
    code, detail = E.device_status()
    assert code == 0, f"device status {code} {detail}"


def check(o, lse, ref_o, ref_lse, rows=None):
    o = o.float().cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy().astype(np.float64)
    d = o.shape[-1]
    if rows is not None:
        o = o.reshape(-1, d)[rows]
        lse = lse.reshape(-1)[rows]
    err = np.abs(o - ref_o)
    bad = err > ATOL + RTOL * np.abs(ref_o)
    assert not bad.any(), (f"{int(bad.sum())} of {bad.size} O elements out of tolerance; "
                           f"max err {err.max():.3e}")
    both_inf = np.isneginf(lse) & np.isneginf(ref_lse)
    with np.errstate(invalid="ignore"):  # -inf - -inf in the rows that see no key
        lerr = np.where(both_inf, 0.0, np.abs(lse - ref_lse))
    assert lerr.max() <= LSE_TOL, f"LSE max err {lerr.max():.3e}"
    return float(err.max()), float(lerr.max())


def run(E, B, H, Nq, Nk, d, mask="none", window=0, grid=None, sigma=1.0, seed=1, rows=None,
        num_ctas=0, scale=None, dilation=1, wrap_axes=None):
    q, k, v = make_qkv(B, H, Nq, Nk, d, sigma, seed)
    scale = scale if scale is not None else 1.0 / math.sqrt(d)
    o, lse = E.attn_fwd(q.cuda(), k.cuda(), v.cuda(), scale=scale, mask=mask, window=window,
                        dilation=dilation, grid=grid, num_ctas=num_ctas, wrap_axes=wrap_axes)
    _status_ok(E)
    ref_o, ref_lse = oracle.attention_rows(to_f64(q), to_f64(k), to_f64(v), rows, scale=scale,
                                           mask_kind=mask, window=window, dilation=dilation,
                                           grid=grid,
                                           wrap=wrap_axes if wrap_axes is not None else False)
    return check(o, lse, ref_o, ref_lse, rows)


SMALL_N = [1, 7, 127, 128, 129, 255, 256, 257, 300, 513]


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("mask", ["none", "causal"])
@pytest.mark.parametrize("N", SMALL_N)
def test_small_square(E, d, mask, N):
    run(E, 1, 2, N, N, d, mask, seed=N * 7 + d)


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("mask", ["none", "causal"])
@pytest.mark.parametrize("Nq,Nk", [(100, 300), (300, 100), (256, 1), (1, 700), (129, 1025)])
def test_small_rectangular(E, d, mask, Nq, Nk):
    run(E, 2, 1, Nq, Nk, d, mask, seed=Nq + Nk + d)


NA_GRIDS = [(5, 5, 3), (8, 8, 3), (16, 16, 5), (20, 12, 5), (13, 29, 7), (64, 64, 7), (40, 40, 39)]


@pytest.mark.parametrize("mode", ["clamp", "wrap"])
@pytest.mark.parametrize("gh,gw,win", NA_GRIDS)
@pytest.mark.parametrize("d", [32, 64, 128])
def test_neighbourhood(E, mode, gh, gw, win, d):
    run(E, 1, 2, gh * gw, gh * gw, d, mode, window=win, grid=(gh, gw), seed=gh * gw + win)


# dilated neighbourhoods: (grid_h, grid_w, window, dilation), window * dilation <= each side
NA_DILATED = [(8, 8, 3, 2), (16, 16, 5, 3), (20, 12, 3, 4), (13, 29, 3, 4), (24, 50, 5, 4),
              (64, 64, 7, 2), (64, 64, 7, 9), (21, 21, 7, 3)]


@pytest.mark.parametrize("mode", ["clamp", "wrap"])
@pytest.mark.parametrize("gh,gw,win,dil", NA_DILATED)
@pytest.mark.parametrize("d", [32, 64])
def test_neighbourhood_dilated(E, mode, gh, gw, win, dil, d):
    run(E, 1, 2, gh * gw, gh * gw, d, mode, window=win, dilation=dil, grid=(gh, gw),
        seed=gh * gw + 31 * win + dil)


# per-axis windows and wrap: (grid, (k_rows, k_cols), (wrap_rows, wrap_cols), dilation)
NA_AXES = [((16, 24), (3, 7), (True, False), 1), ((20, 20), (5, 3), (False, True), 1),
           ((32, 64), (7, 5), (True, True), 1), ((48, 40), (5, 3), (True, False), 4),
           ((13, 29), (1, 9), (False, True), 2), ((1, 1000), (1, 15), (False, False), 1),
           ((1, 1000), (1, 15), (False, True), 1), ((1, 777), (1, 9), (False, False), 3),
           ((1, 4096), (1, 63), (False, False), 1)]


@pytest.mark.parametrize("grid,win,wrap_axes,dil", NA_AXES)
@pytest.mark.parametrize("d", [32, 64])
def test_neighbourhood_per_axis(E, grid, win, wrap_axes, dil, d):
    N = grid[0] * grid[1]
    run(E, 1, 2, N, N, d, "clamp", window=win, dilation=dil, grid=grid, wrap_axes=wrap_axes,
        seed=N + 7 * win[0] + 13 * win[1] + dil)


def test_na2d_heads_last_per_axis_modes(E):
    B, X, Y, H, d = 1, 12, 20, 2, 32
    q, k, v = (torch.randn(B, X, Y, H, d, generator=torch.Generator().manual_seed(s)).to(
        torch.bfloat16) for s in (1, 2, 3))
    o = E.na2d(q.cuda(), k.cuda(), v.cuda(), (5, 3), mode=("wrap", "clamp"))
    _status_ok(E)
    to_bhnd = lambda t: t.float().permute(0, 3, 1, 2, 4).reshape(B, H, X * Y, d)
    ref_o, _ = oracle.attention_rows(to_bhnd(q).numpy(), to_bhnd(k).numpy(), to_bhnd(v).numpy(),
                                     None, scale=1 / math.sqrt(d), mask_kind="clamp",
                                     window=(5, 3), wrap=(True, False), grid=(X, Y))
    got = to_bhnd(o.cpu()).numpy()
    err = np.abs(got - ref_o)
    assert (err <= ATOL + RTOL * np.abs(ref_o)).all(), float(err.max())


# Volumes (NA3D): (grid (depth, rows, cols), window per axis, wrap per axis, dilation).
# The first is the NATTEN issue requester's setting: ~16 patches a side, window 5,
# two wrapped axes.
NA3 = [((16, 16, 16), (5, 5, 5), (True, True, False), 1), ((8, 8, 8), (3, 3, 3), (True, True, True), 1),
       ((20, 15, 18), (5, 3, 7), (False, True, True), 1), ((6, 10, 30), (1, 3, 9), (False, False, True), 3),
       ((12, 1, 40), (3, 1, 5), (True, False, False), 1), ((9, 9, 9), (9, 9, 9), (True, False, True), 1),
       ((4, 20, 3), (3, 7, 3), (False, True, False), 1), ((8, 8, 8), (3, 3, 3), (False, False, False), 2),
       ((3, 5, 7), (3, 5, 7), (False, False, False), 1)]


@pytest.mark.parametrize("grid,win,wrap_axes,dil", NA3)
@pytest.mark.parametrize("d", [32, 64, 128])
def test_neighbourhood_3d(E, grid, win, wrap_axes, dil, d):
    n = grid[0] * grid[1] * grid[2]
    run(E, 1, 2, n, n, d, "clamp", window=win, dilation=dil, grid=grid, wrap_axes=wrap_axes,
        seed=n + d + dil)


def test_neighbourhood_3d_mask_name_and_persistent(E):
    run(E, 2, 1, 4096, 4096, 64, "wrap", window=5, grid=(16, 16, 16), seed=91)
    run(E, 1, 3, 1000, 1000, 32, "clamp", window=(3, 5, 3), grid=(10, 10, 10), num_ctas=2, seed=92)


def test_na3d_heads_last(E):
    B, X, Y, Z, H, d = 1, 6, 8, 10, 2, 64
    q, k, v = (torch.randn(B, X, Y, Z, H, d, generator=torch.Generator().manual_seed(s)).to(
        torch.bfloat16) for s in (4, 5, 6))
    o, lse = E.na3d(q.cuda(), k.cuda(), v.cuda(), (3, 5, 3), mode=("wrap", "clamp", "wrap"),
                    return_lse=True)
    _status_ok(E)
    n = X * Y * Z
    to_bhnd = lambda t: t.float().permute(0, 4, 1, 2, 3, 5).reshape(B, H, n, d)
    ref_o, ref_lse = oracle.attention_rows(to_bhnd(q).numpy(), to_bhnd(k).numpy(),
                                           to_bhnd(v).numpy(), None, scale=1 / math.sqrt(d),
                                           mask_kind="clamp", window=(3, 5, 3),
                                           wrap=(True, False, True), grid=(X, Y, Z))
    assert o.shape == q.shape
    o_bhnd = o.permute(0, 4, 1, 2, 3, 5).reshape(B, H, n, d)
    check(o_bhnd, lse, ref_o, ref_lse)


def test_neighbourhood_dilated_d128_and_persistent(E):
    run(E, 2, 1, 1024, 1024, 128, "wrap", window=5, dilation=3, grid=(32, 32), seed=77)
    run(E, 1, 3, 1024, 1024, 32, "clamp", window=5, dilation=2, grid=(32, 32), num_ctas=2,
        seed=78)


def test_issue142_wrap_example_on_gpu(E):
    """NATTEN issue #142: 5x5 grid, kernel 3, wrap, q = k = ones, v one-hot top-left."""
    q = torch.ones(1, 1, 25, 32, dtype=torch.bfloat16, device="cuda")
    k = torch.ones_like(q)
    v = torch.zeros_like(q)
    v[0, 0, 0, :] = 1
    o = E.attn_fwd(q, k, v, mask="wrap", window=3, return_lse=False)
    _status_ok(E)
    x = o[0, 0, :, 0].float().cpu().reshape(5, 5).numpy()
    expect = np.zeros((5, 5))
    for i in (0, 1, 4):
        for j in (0, 1, 4):
            expect[i, j] = 1 / 9
    assert np.max(np.abs(x - expect)) <= ATOL + RTOL * np.abs(expect).max()


@pytest.mark.parametrize("num_ctas", [1, 3, 7])
@pytest.mark.parametrize("mask", ["none", "causal"])
def test_persistent_small_grid(E, num_ctas, mask):
    """Several tasks per CTA: the barrier phases must carry across tasks."""
    run(E, 2, 3, 700, 700, 64, mask, num_ctas=num_ctas, seed=num_ctas)


def test_persistent_small_grid_na(E):
    run(E, 1, 3, 1024, 1024, 32, "wrap", window=5, grid=(32, 32), num_ctas=2, seed=5)


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_workloads_all_rows(E, name):
    """The full-size workloads in the launch configuration the benchmark times
    (default schedule, every SM), every output row compared with the oracle.
    The fp64 oracle runs on all host cores; the longest (16384 keys, d 128,
    eight heads, about 1.1 TFLOP in fp64) takes tens of seconds."""
    w = WORKLOADS[name]
    q, k, v = make_workload(w)
    o, lse = E.attn_fwd(q.cuda(), k.cuda(), v.cuda(), scale=w.scale, mask=w.mask,
                        window=w.window, grid=w.grid, wrap_axes=w.wrap_axes)
    _status_ok(E)
    ref_o, ref_lse = oracle.attention(to_f64(q), to_f64(k), to_f64(v), scale=w.scale,
                                      mask_kind=w.mask, window=w.window, grid=w.grid,
                                      wrap=w.wrap_axes if w.wrap_axes is not None else False)
    check(o, lse, ref_o, ref_lse)


def test_heads_last_layout_na2d(E):
    """NATTEN's [B, X, Y, heads, d] layout through strides, no permute."""
    B, X, Y, H, d = 2, 12, 20, 3, 64
    g = torch.Generator().manual_seed(3)
    q, k, v = (torch.randn(B, X, Y, H, d, generator=g).bfloat16() for _ in range(3))
    o = E.na2d(q.cuda(), k.cuda(), v.cuda(), 5, mode="wrap")
    _status_ok(E)
    perm = lambda t: t.permute(0, 3, 1, 2, 4).reshape(B, H, X * Y, d)
    ref_o, _ = oracle.attention(to_f64(perm(q)), to_f64(perm(k)), to_f64(perm(v)),
                                scale=1 / math.sqrt(d), mask_kind="wrap", window=5, grid=(X, Y))
    got = perm(o.cpu()).float().numpy()
    err = np.abs(got - ref_o)
    assert (err <= ATOL + RTOL * np.abs(ref_o)).all(), err.max()


def test_strided_inputs(E):
    """q, k, v as strided views (a slice of a wider tensor)."""
    B, H, N, d = 1, 2, 300, 64
    g = torch.Generator().manual_seed(4)
    big = torch.randn(B, H, N, 3 * d, generator=g).bfloat16()
    q, k, v = big[..., :d], big[..., d:2 * d], big[..., 2 * d:]
    bigc = big.cuda()
    o, lse = E.attn_fwd(bigc[..., :d], bigc[..., d:2 * d], bigc[..., 2 * d:], mask="causal")
    _status_ok(E)
    ref_o, ref_lse = oracle.attention(to_f64(q.contiguous()), to_f64(k.contiguous()),
                                      to_f64(v.contiguous()), scale=1 / math.sqrt(d),
                                      mask_kind="causal")
    check(o, lse, ref_o, ref_lse)


def test_outputs_stay_in_bounds(E):
    """Guard bands around O and LSE are untouched (ragged Nq)."""
    B, H, N, d = 1, 2, 300, 128
    q, k, v = make_qkv(B, H, N, N, d, 1.0, 9)
    guard = 4096
    o_buf = torch.full((B * H * N * d + 2 * guard,), 7.0, dtype=torch.bfloat16, device="cuda")
    l_buf = torch.full((B * H * N + 2 * guard,), 7.0, dtype=torch.float32, device="cuda")
    o = o_buf[guard:guard + B * H * N * d].view(B, H, N, d)
    lse = l_buf[guard:guard + B * H * N].view(B, H, N)
    E.attn_fwd(q.cuda(), k.cuda(), v.cuda(), out=o, lse=lse)
    _status_ok(E)
    assert bool((o_buf[:guard] == 7).all()) and bool((o_buf[-guard:] == 7).all())
    assert bool((l_buf[:guard] == 7).all()) and bool((l_buf[-guard:] == 7).all())


def test_no_lse(E):
    q, k, v = make_qkv(1, 1, 200, 200, 64, 1.0, 10)
    o = E.attn_fwd(q.cuda(), k.cuda(), v.cuda(), return_lse=False)
    _status_ok(E)
    ref_o, _ = oracle.attention(to_f64(q), to_f64(k), to_f64(v), scale=0.125)
    err = np.abs(o.float().cpu().numpy() - ref_o)
    assert (err <= ATOL + RTOL * np.abs(ref_o)).all()


def test_host_tensors_roundtrip(E):
    """CPU tensors in, CPU tensors out (the end-to-end path)."""
    q, k, v = make_qkv(1, 2, 333, 333, 64, 1.0, 11)
    o, lse = E.attn_fwd(q, k, v, mask="causal")
    assert o.device.type == "cpu" and lse.device.type == "cpu"
    ref_o, ref_lse = oracle.attention(to_f64(q), to_f64(k), to_f64(v), scale=0.125,
                                      mask_kind="causal")
    check(o, lse, ref_o, ref_lse)


def test_bounded_wait_reports_timeout(E):
    """The loader withholds one K tile: the MMA issuer's wait runs out after the
    bound, the kernel returns, and the host reads ATTN_ERR_TIMEOUT. The context
    stays usable: a normal call afterwards is correct."""
    q, k, v = make_qkv(1, 1, 256, 1024, 64, 1.0, 12)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    E.attn_fwd(qc, kc, vc, timeout_ns=20_000_000, inject=1, num_ctas=1)
    torch.cuda.synchronize()
    code, detail = E.device_status()
    assert code == 5 and detail[0] == 5, (code, detail)
    assert E.device_status()[0] == 0  # reading cleared it
    o, lse = E.attn_fwd(qc, kc, vc)
    _status_ok(E)
    ref_o, ref_lse = oracle.attention(to_f64(q), to_f64(k), to_f64(v), scale=0.125)
    check(o, lse, ref_o, ref_lse)


@pytest.mark.parametrize("num_ctas", [2, 3, 5, 13, 0])
@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("N", [300, 1000])
def test_split_schedule(E, num_ctas, d, N):
    """Equal shares of K/V tiles per CTA: tasks cut between CTAs are merged by
    their last part (ragged Nk included: 300 and 1000 are not multiples of 128)."""
    q, k, v = make_qkv(1, 3, N, N, d, 1.0, 20 + num_ctas + d)
    o, lse = E.attn_fwd(q.cuda(), k.cuda(), v.cuda(), num_ctas=num_ctas, schedule=2)
    _status_ok(E)
    ref_o, ref_lse = oracle.attention(to_f64(q), to_f64(k), to_f64(v), scale=1 / math.sqrt(d))
    check(o, lse, ref_o, ref_lse)


def test_split_many_parts_per_task(E):
    """One head, two Q pairs over many CTAs: every task is cut into ~10 parts."""
    q, k, v = make_qkv(1, 1, 512, 4096, 64, 1.0, 31)
    o, lse = E.attn_fwd(q.cuda(), k.cuda(), v.cuda(), num_ctas=20, schedule=2)
    _status_ok(E)
    ref_o, ref_lse = oracle.attention(to_f64(q), to_f64(k), to_f64(v), scale=0.125)
    check(o, lse, ref_o, ref_lse)


def test_split_repeated_calls_reuse_workspace(E):
    """Consecutive calls share the library's workspace; per-call tags keep the
    arrival counts of one call from leaking into the next."""
    q, k, v = (t.cuda() for t in make_qkv(2, 2, 700, 700, 64, 1.0, 32))
    ref = None
    for _ in range(5):
        o, lse = E.attn_fwd(q, k, v, num_ctas=7, schedule=2)
        _status_ok(E)
        if ref is None:
            ref = (o.clone(), lse.clone())
        else:
            assert torch.equal(o, ref[0]) and torch.equal(lse, ref[1])
    ref_o, ref_lse = oracle.attention(to_f64(q.cpu()), to_f64(k.cpu()), to_f64(v.cpu()),
                                      scale=0.125)
    check(ref[0], ref[1], ref_o, ref_lse)


def test_split_caller_workspace(E):
    q, k, v = (t.cuda() for t in make_qkv(1, 2, 777, 900, 128, 1.0, 33))
    nbytes = E.workspace_bytes(1, 2, 777, 900, 128, num_ctas=5, schedule=2)
    assert nbytes > 0
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        o, lse = E.attn_fwd(q, k, v, num_ctas=5, schedule=2, workspace=ws)
        _status_ok(E)
    ref_o, ref_lse = oracle.attention(to_f64(q.cpu()), to_f64(k.cpu()), to_f64(v.cpu()),
                                      scale=1 / math.sqrt(128))
    check(o, lse, ref_o, ref_lse)


def test_split_and_whole_schedules_agree(E):
    q, k, v = (t.cuda() for t in make_qkv(2, 5, 4096, 4096, 64, 0.5, 34))
    o1, l1 = E.attn_fwd(q, k, v, schedule=1)
    o2, l2 = E.attn_fwd(q, k, v, schedule=2)
    _status_ok(E)
    assert (o1.float() - o2.float()).abs().max().item() <= 1e-2
    assert (l1 - l2).abs().max().item() <= 1e-3


def test_split_many_parts_bitwise_repeatable(E):
    """One head of 4096 queries on the default schedule cuts every task into
    several parts; whichever part merges, the merge sums the parts in CTA order,
    so repeated calls give identical bits."""
    q, k, v = (t.cuda() for t in make_qkv(1, 1, 4096, 4096, 64, 1.0, 33))
    first = E.attn_fwd(q, k, v)
    _status_ok(E)
    for _ in range(4):
        o, lse = E.attn_fwd(q, k, v)
        _status_ok(E)
        assert torch.equal(o, first[0]) and torch.equal(lse, first[1])
    rows = np.arange(0, 4096, 37)
    ref_o, ref_lse = oracle.attention_rows(to_f64(q.cpu()), to_f64(k.cpu()), to_f64(v.cpu()), rows,
                                           scale=0.125)
    check(first[0], first[1], ref_o, ref_lse, rows)


@pytest.mark.parametrize("mask,shape", [("none", (1, 1, 4096, 64)), ("none", (2, 5, 4096, 64)),
                                        ("causal", (2, 4, 1024, 128))])
def test_tuned_schedule_is_valid_and_exact(E, mask, shape):
    B, H, N, d = shape
    q, k, v = (t.cuda() for t in make_qkv(B, H, N, N, d, 1.0, 41))
    best = E.tune(q, k, v, mask=mask, iters=3)
    _status_ok(E)
    assert best["schedule"] in (1, 2) and best["us"] > 0 and best["n_tried"] >= 1
    if mask != "none":
        assert best["schedule"] == 1 and best["n_tried"] == 1
    assert 0 <= best["num_ctas"] <= E.sm_count()
    o, lse = E.attn_fwd(q, k, v, mask=mask, schedule=best["schedule"], num_ctas=best["num_ctas"])
    _status_ok(E)
    rows = np.arange(0, B * H * N, 97)
    ref_o, ref_lse = oracle.attention_rows(to_f64(q.cpu()), to_f64(k.cpu()), to_f64(v.cpu()), rows,
                                           scale=1.0 / math.sqrt(d), mask_kind=mask)
    check(o, lse, ref_o, ref_lse, rows)



@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("Nq,Nk", [(100, 300), (300, 100), (1, 700), (700, 1), (129, 1025), (1000, 260)])
def test_causal_bottom_right(E, d, Nq, Nk):
    """Query i sees keys 0 .. i + Nk - Nq; with Nq > Nk the first rows see none
    (O = 0, LSE = -inf)."""
    run(E, 2, 1, Nq, Nk, d, "causal_br", seed=Nq * 3 + Nk + d)


@pytest.mark.parametrize("num_ctas,d", [(3, 64), (5, 128), (0, 32)])
def test_causal_bottom_right_many_empty_tasks_per_cta(E, num_ctas, d):
    """Nq much larger than Nk: most Q tiles have no key at all, and each CTA
    takes several of those tasks in a row (few CTAs for many tasks). Every
    task, even one without a K/V tile, must hand its Q buffer back so that the
    next task's Q can be loaded."""
    run(E, 2, 3, 3000, 100, d, "causal_br", seed=3100 + d, num_ctas=num_ctas)


def test_causal_bottom_right_equals_top_left_when_square(E):
    q, k, v = (t.cuda() for t in make_qkv(1, 3, 777, 777, 64, 1.0, 51))
    a = E.attn_fwd(q, k, v, mask="causal")
    b = E.attn_fwd(q, k, v, mask="causal_br")
    _status_ok(E)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


# Twin tasks: neighbourhood launches with one Q tile per task and K/V chains of
# 8 tiles or more give both softmax warpgroups the same queries, the K/V tiles
# in turn, and merge the two halves in the CTA. (B, H, grid, window, dilation,
# wrap axes, d, CTAs; 0 = one per SM). One Q tile per task needs fewer Q-tile
# pairs than CTAs; with fewer CTAs than single-tile tasks, some CTAs run two
# twin tasks in a row (the exchange's phases carry over).
TWIN = [
    (1, 2, (40, 40), 39, 1, None, 64, 0),                     # every key in every window
    (1, 3, (48, 48), 21, 1, (True, False), 32, 40),      # 27 pairs, 54 tasks
    (2, 1, (32, 32), 9, 2, (False, True), 128, 12),      # 8 pairs, 16 tasks
    (1, 2, (16, 16, 16), 5, 1, (True, True, False), 32, 0),   # the NATTEN-issue volume
    (1, 1, (12, 14, 10), (7, 7, 3), 1, (False, True, False), 64, 10),  # 7 pairs
    (1, 2, (16, 16, 24), 3, 2, (False, False, False), 128, 64),  # 48 pairs
]


@pytest.mark.parametrize("B,H,grid,win,dil,wrap_axes,d,num_ctas", TWIN)
def test_twin_tasks_match_the_oracle(E, B, H, grid, win, dil, wrap_axes, d, num_ctas):
    n = math.prod(grid)
    run(E, B, H, n, n, d, "clamp", window=win, dilation=dil, grid=grid, wrap_axes=wrap_axes,
        num_ctas=num_ctas, seed=n + d + 17 * dil)


def test_twin_decision_in_the_log():
    """ATTN_LOG's twin flag: on for every case above, off for a 64 x 64 grid
    with window 7 (5 K/V tiles a Q tile) and for launches with Q-tile pairs."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    calls = [f"E.attn_fwd(*qkv({math.prod(g)}, {d}, {B}, {H}), mask='clamp', window={w!r}, "
             f"dilation={dl}, grid={g!r}, wrap_axes={wa!r}, num_ctas={nc})"
             for B, H, g, w, dl, wa, d, nc in TWIN]
    calls += ["E.attn_fwd(*qkv(4096, 32, 1, 4), mask='clamp', window=7, grid=(64, 64))",
              "E.attn_fwd(*qkv(4096, 32, 8, 16), mask='clamp', window=7, grid=(64, 64))"]
    code = ("import torch, exact_attention_69_gb300 as E; from seeded_inputs import make_qkv\n"
            "def qkv(n, d, B, H): return [t.cuda() for t in make_qkv(B, H, n, n, d, 1.0, 3)]\n"
            + "\n".join(calls) + "\ntorch.cuda.synchronize()\n")
    env = dict(os.environ, ATTN_LOG="1", PYTHONPATH=root)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       cwd=root, timeout=600)
    assert r.returncode == 0, r.stderr
    flags = [ln.rsplit("twin=", 1)[1].strip() for ln in r.stderr.splitlines()
             if ln.startswith("attn_fwd:")]
    assert flags == ["1"] * len(TWIN) + ["0", "0"], r.stderr
