"""GPU backward pass (attn_bwd) against the fp64 oracle's backward.

Inputs are seeded bf16 tensors; the oracle takes the same bf16 values in fp64.
Tolerance, from the arithmetic: the kernels round P (for dV) and dS (for dQ
and dK) to bf16, relative 2^-9, before their products and sums, which run in
fp32 over up to N terms of mixed sign; the gradients are then rounded to bf16.
Per element: |err| <= 2e-2 |ref| + 1e-2 g, where g is the larger of max|ref| of
that gradient and a tenth of the largest max|ref| of the three (a gradient can
vanish exactly, e.g. dQ with a single key, while its terms do not).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from seeded_inputs import make_qkv, to_f64

pytestmark = pytest.mark.gpu

RTOL, ATOL_FRAC = 2e-2, 1e-2


@pytest.fixture(scope="module")
def E():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import exact_attention_69_gb300 as E
    return E


def _grad_check(name, got, ref, scale_all):
    got = got.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    lim = RTOL * np.abs(ref) + ATOL_FRAC * max(np.abs(ref).max(), 0.1 * scale_all, 1e-30)
    bad = err > lim
    assert not bad.any(), (f"{name}: {int(bad.sum())} of {bad.size} elements out of tolerance; "
                           f"max err {err.max():.3e}, max |ref| {np.abs(ref).max():.3e}")


def run_bwd(E, B, H, Nq, Nk, d, mask, seed, window=0, dilation=1, grid=None, wrap_axes=None):
    q, k, v = make_qkv(B, H, Nq, Nk, d, 1.0, seed)
    g = torch.Generator().manual_seed(seed + 1)
    dout = torch.randn(B, H, Nq, d, generator=g).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(d)
    qc, kc, vc, gc = (t.cuda() for t in (q, k, v, dout))
    na = dict(window=window, dilation=dilation, grid=grid, wrap_axes=wrap_axes)
    o, lse = E.attn_fwd(qc, kc, vc, scale=scale, mask=mask, **na)
    dq, dk, dv = E.attn_bwd(qc, kc, vc, o, lse, gc, scale=scale, mask=mask, **na)
    torch.cuda.synchronize()
    code, detail = E.device_status()
    assert code == 0, detail
    rq, rk, rv = oracle.attention_bwd(to_f64(q), to_f64(k), to_f64(v), to_f64(dout), scale=scale,
                                      mask_kind=mask, window=window, dilation=dilation, grid=grid,
                                      wrap=wrap_axes if wrap_axes is not None else False)
    scale_all = max(np.abs(r).max() for r in (rq, rk, rv))
    _grad_check("dq", dq, rq, scale_all)
    _grad_check("dk", dk, rk, scale_all)
    _grad_check("dv", dv, rv, scale_all)


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("mask", ["none", "causal"])
@pytest.mark.parametrize("N", [1, 100, 128, 129, 300])
def test_backward_square(E, d, mask, N):
    run_bwd(E, 1, 2, N, N, d, mask, seed=N * 3 + d)


@pytest.mark.parametrize("mask", ["none", "causal"])
@pytest.mark.parametrize("Nq,Nk", [(200, 333), (333, 200), (128, 1), (1, 257)])
def test_backward_rectangular(E, mask, Nq, Nk):
    run_bwd(E, 2, 1, Nq, Nk, 64, mask, seed=Nq + Nk)


@pytest.mark.parametrize("mask", ["none", "causal"])
def test_backward_longer(E, mask):
    run_bwd(E, 1, 2, 1024, 1024, 64, mask, seed=11)


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("Nq,Nk", [(200, 333), (333, 200), (128, 1), (1, 257), (300, 128)])
def test_backward_causal_bottom_right(E, d, Nq, Nk):
    """Rows that see no key (Nq > Nk) have zero gradients and add nothing to dK, dV."""
    run_bwd(E, 2, 1, Nq, Nk, d, "causal_br", seed=Nq + 2 * Nk + d)


def test_autograd_wrapper_matches_attn_bwd(E):
    q, k, v = (t.cuda() for t in make_qkv(1, 2, 300, 300, 64, 1.0, 5))
    g = torch.randn(1, 2, 300, 64, generator=torch.Generator().manual_seed(6)).to(torch.bfloat16).cuda()
    qr, kr, vr = (t.clone().requires_grad_(True) for t in (q, k, v))
    out = E.attention(qr, kr, vr, mask="causal")
    out.backward(g)
    o, lse = E.attn_fwd(q, k, v, mask="causal")
    dq, dk, dv = E.attn_bwd(q, k, v, o, lse, g, mask="causal")
    assert torch.equal(out, o)
    for a, b in ((qr.grad, dq), (kr.grad, dk), (vr.grad, dv)):
        assert torch.equal(a, b)


# Neighbourhood attention: the dQ kernel masks each query row as the forward does;
# the dK/dV kernel needs the transposed relation (which queries hold a key in their
# window), which for wrap-around windows differs from a window centred on the key.
NA_BWD = [(8, 8, 3), (16, 16, 5), (20, 12, 5), (13, 29, 7), (40, 40, 13)]


@pytest.mark.parametrize("mode", ["clamp", "wrap"])
@pytest.mark.parametrize("gh,gw,win", NA_BWD)
@pytest.mark.parametrize("d", [32, 64, 128])
def test_backward_neighbourhood(E, mode, gh, gw, win, d):
    run_bwd(E, 1, 2, gh * gw, gh * gw, d, mode, seed=gh * gw + win + d, window=win, grid=(gh, gw))


NA_BWD_DILATED = [(16, 16, 3, 2), (20, 12, 3, 4), (24, 50, 5, 4), (21, 21, 7, 3)]


@pytest.mark.parametrize("mode", ["clamp", "wrap"])
@pytest.mark.parametrize("gh,gw,win,dil", NA_BWD_DILATED)
def test_backward_neighbourhood_dilated(E, mode, gh, gw, win, dil):
    run_bwd(E, 1, 2, gh * gw, gh * gw, 64, mode, seed=gh + gw + win * dil, window=win,
            dilation=dil, grid=(gh, gw))


NA_BWD_AXES = [((16, 24), (3, 7), (True, False), 1), ((20, 20), (5, 3), (False, True), 1),
               ((48, 40), (5, 3), (True, False), 4), ((13, 29), (1, 9), (False, True), 2),
               ((1, 1000), (1, 15), (False, True), 1), ((1, 777), (1, 9), (False, False), 3)]


@pytest.mark.parametrize("grid,win,wrap_axes,dil", NA_BWD_AXES)
def test_backward_neighbourhood_per_axis(E, grid, win, wrap_axes, dil):
    n = grid[0] * grid[1]
    run_bwd(E, 1, 2, n, n, 64, "clamp", seed=n + dil, window=win, dilation=dil, grid=grid,
            wrap_axes=wrap_axes)


NA3_BWD = [((16, 16, 16), (5, 5, 5), (True, True, False), 1, 64),
           ((8, 8, 8), (3, 3, 3), (True, True, True), 1, 32),
           ((20, 15, 18), (5, 3, 7), (False, True, True), 1, 128),
           ((6, 10, 30), (1, 3, 9), (False, False, True), 3, 64),
           ((12, 1, 40), (3, 1, 5), (True, False, False), 1, 64),
           ((8, 8, 8), (3, 3, 3), (False, False, False), 2, 64)]


@pytest.mark.parametrize("grid,win,wrap_axes,dil,d", NA3_BWD)
def test_backward_neighbourhood_3d(E, grid, win, wrap_axes, dil, d):
    n = grid[0] * grid[1] * grid[2]
    run_bwd(E, 1, 2, n, n, d, "clamp", seed=n + dil + d, window=win, dilation=dil, grid=grid,
            wrap_axes=wrap_axes)


def test_backward_neighbourhood_full_window_is_unmasked(E):
    """A window that covers the whole grid (clamp) allows every key: from the same
    O and LSE, the backward kernels give the unmasked gradients bit for bit. (The
    two forwards are separate kernels that round P at different points, so each
    is checked against the oracle elsewhere, not against the other.)"""
    q, k, v = (t.cuda() for t in make_qkv(1, 2, 15 * 15, 15 * 15, 64, 1.0, 21))
    g = torch.randn(1, 2, 225, 64, generator=torch.Generator().manual_seed(22)).to(torch.bfloat16).cuda()
    o, lse = E.attn_fwd(q, k, v, mask="clamp", window=15, grid=(15, 15))
    ref = E.attn_bwd(q, k, v, o, lse, g)
    got = E.attn_bwd(q, k, v, o, lse, g, mask="clamp", window=15, grid=(15, 15))
    for a, b in zip(got, ref):
        assert torch.equal(a, b)


def test_autograd_wrapper_neighbourhood(E):
    q, k, v = (t.cuda() for t in make_qkv(1, 2, 256, 256, 64, 1.0, 8))
    g = torch.randn(1, 2, 256, 64, generator=torch.Generator().manual_seed(9)).to(torch.bfloat16).cuda()
    na = dict(mask="wrap", window=(5, 3), grid=(16, 16), dilation=2)
    qr, kr, vr = (t.clone().requires_grad_(True) for t in (q, k, v))
    out = E.attention(qr, kr, vr, **na)
    out.backward(g)
    o, lse = E.attn_fwd(q, k, v, **na)
    dq, dk, dv = E.attn_bwd(q, k, v, o, lse, g, **na)
    assert torch.equal(out, o)
    for a, b in ((qr.grad, dq), (kr.grad, dk), (vr.grad, dv)):
        assert torch.equal(a, b)
