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


def run_bwd(E, B, H, Nq, Nk, d, mask, seed):
    q, k, v = make_qkv(B, H, Nq, Nk, d, 1.0, seed)
    g = torch.Generator().manual_seed(seed + 1)
    dout = torch.randn(B, H, Nq, d, generator=g).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(d)
    qc, kc, vc, gc = (t.cuda() for t in (q, k, v, dout))
    o, lse = E.attn_fwd(qc, kc, vc, scale=scale, mask=mask)
    dq, dk, dv = E.attn_bwd(qc, kc, vc, o, lse, gc, scale=scale, mask=mask)
    torch.cuda.synchronize()
    code, detail = E.device_status()
    assert code == 0, detail
    rq, rk, rv = oracle.attention_bwd(to_f64(q), to_f64(k), to_f64(v), to_f64(dout), scale=scale,
                                      mask_kind=mask)
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


def test_backward_rejects_neighbourhood_masks(E):
    q, k, v = (t.cuda() for t in make_qkv(1, 1, 64, 64, 32, 1.0, 1))
    o, lse = E.attn_fwd(q, k, v, mask="clamp", window=3, grid=(8, 8))
    with pytest.raises(ValueError):
        E.attn_bwd(q, k, v, o, lse, torch.ones_like(q), mask="clamp")
