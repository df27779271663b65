"""GPU backward pass (attn_bwd) against the fp64 oracle's backward.

Inputs are seeded bf16 tensors; the oracle takes the same bf16 values in fp64.

Tolerance, per element, from where the kernels round (u = 2^-9, the bf16
unit roundoff):
  - the forward's O is bf16 and was formed from bf16 P: |dO_err| <= 2u (P |V|),
    so D = rowsum(dout * O) is off by at most dD = |dout| . 2u (P |V|);
  - dS = P (dP - D) is rounded to bf16 before dQ = scale dS K and
    dK = scale dS^T Q: |dS_err| <= u |dS| + P dD (+ 1e-5 P |dP - D| for the
    fp32 recomputation of P from the log-sum-exp);
  - P is rounded to bf16 before dV = P^T dout;
  - every gradient is rounded to bf16 (u |grad|).
So |dQ_err| <= scale |dS_err| |K| + u |dQ|, |dK_err| <= scale |dS_err|^T |Q| +
u |dK|, |dV_err| <= u P^T |dout| + u |dV|, each taken twice (fp32 sums over up
to N terms and second-order terms), plus a floor of 1e-6 max|grad| for fp32
noise. The magnitudes are computed in fp64 from the inputs and the explicit
mask. Simulating those rounding points in numpy on the CPU keeps every element
within the bound (worst ratio about 0.8, for dV).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import reference_np
from seeded_inputs import make_qkv, to_f64

pytestmark = pytest.mark.gpu

U = 2.0 ** -9  # bf16 unit roundoff


@pytest.fixture(scope="module")
def E():
    from exact_attention_69_gb300 import build
    build.build()
    import exact_attention_69_gb300 as E
    return E


def grad_bounds(q, k, v, dout, scale, allowed):
    """Per-element error bounds (dq, dk, dv) of one head: q [Nq, d], k/v [Nk, d],
    dout [Nq, d] fp64; allowed [Nq, Nk] bool."""
    s = np.where(allowed, scale * (q @ k.T), -np.inf)
    mx = s.max(axis=1, keepdims=True)
    mx = np.where(np.isfinite(mx), mx, 0.0)
    e = np.where(allowed, np.exp(s - mx), 0.0)
    l = e.sum(axis=1, keepdims=True)
    P = np.where(l > 0, e / np.where(l > 0, l, 1.0), 0.0)
    o = P @ v
    dP = dout @ v.T
    D = (dout * o).sum(axis=1, keepdims=True)
    dS = P * (dP - D)
    dq, dk, dv = scale * dS @ k, scale * dS.T @ q, P.T @ dout
    dD = (np.abs(dout) * (2 * U * (P @ np.abs(v)))).sum(axis=1, keepdims=True)
    dS_err = U * np.abs(dS) + P * dD + 1e-5 * P * np.abs(dP - D)
    bq = 2 * (scale * dS_err @ np.abs(k) + U * np.abs(dq))
    bk = 2 * (scale * dS_err.T @ np.abs(q) + U * np.abs(dk))
    bv = 2 * (U * (P.T @ np.abs(dout)) + U * np.abs(dv))
    return bq, bk, bv


def _grad_check(name, got, ref, bound):
    got = got.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    lim = bound + 1e-6 * max(np.abs(ref).max(), 1e-30)
    bad = err > lim
    assert not bad.any(), (f"{name}: {int(bad.sum())} of {bad.size} elements out of tolerance; "
                           f"worst err/bound {float((err / lim).max()):.2f}")


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
    allowed = reference_np.mask_matrix(Nq, Nk, mask, window=window, dilation=dilation, grid=grid,
                                       wrap_axes=wrap_axes)
    qf, kf, vf, gf = to_f64(q), to_f64(k), to_f64(v), to_f64(dout)
    bq, bk, bv = np.empty_like(rq), np.empty_like(rk), np.empty_like(rv)
    for b in range(B):
        for h in range(H):
            bq[b, h], bk[b, h], bv[b, h] = grad_bounds(qf[b, h], kf[b, h], vf[b, h], gf[b, h], scale,
                                                       allowed)
    _grad_check("dq", dq, rq, bq)
    _grad_check("dk", dk, rk, bk)
    _grad_check("dv", dv, rv, bv)


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
