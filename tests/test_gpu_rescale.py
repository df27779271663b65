"""GPU parity for the running-maximum correction of the online softmax.

The kernel keeps each row's maximum lazily: O and the row sum are rescaled
(O <- alpha O with alpha = 2^(m_old - m_new)) only when a tile's maximum
exceeds the stale one by more than 8 (log2 units). With inputs whose scores
are N(0, 1)-sized, the maximum never grows that much after the first tile,
so the rescale would only ever run with alpha = 0. Here the scores grow along
the key sequence: the queries are non-negative and key j is shifted by
beta_j = gamma * j / Nk in every component, so q . k_j grows by
beta_j * sum(q). Each test first computes, from the very bf16 inputs, how far
a tile's maximum rises above the running maximum of the tiles before it, and
asserts that this exceeds the threshold (so the rescale path runs), then
compares O and the log-sum-exp with the fp64 oracle at the usual tolerances.

The split-schedule cases cut tasks between CTAs whose parts' maxima differ by
tens to hundreds of log2 units, so the merge's weights 2^(m_i - M) are tiny or
underflow to zero for the earlier parts.

Sources: the xformers/PhotoRoom memory-efficient attention post (a running
softmax over K/V tiles); "Fused Self Attention" (NKI tutorial), section
"Softmax implementation" (partial row maxima combined into the row maximum).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import reference_np
from seeded_inputs import make_qkv, to_f64

pytestmark = pytest.mark.gpu

ATOL, RTOL, LSE_TOL = 1e-2, 1e-2, 1e-3
LOG2E = 1.4426950408889634
TAU = 8.0  # the kernel's rescale threshold, log2 units


@pytest.fixture(scope="module")
def E():
    from exact_attention_69_gb300 import build
    build.build()
    import exact_attention_69_gb300 as E
    return E


def growing_qkv(B, H, N, d, gamma, seed):
    """Seeded bf16 q (non-negative), k shifted by gamma * j / N along the
    sequence, v as drawn."""
    q, k, v = make_qkv(B, H, N, N, d, 1.0, seed)
    q = q.abs()
    beta = gamma * torch.arange(N, dtype=torch.float32) / N
    k = (k.float() + beta[None, None, :, None]).to(torch.bfloat16)
    return q, k, v


def tile_maxima(q, k, scale, allowed):
    """[Nq, tiles] maxima (log2 units) of each 128-key tile's allowed scores of one head."""
    s = (q @ k.T) * (scale * LOG2E)
    s = np.where(allowed, s, -np.inf)
    nt = -(-k.shape[0] // 128)
    pad = np.full((s.shape[0], nt * 128), -np.inf)
    pad[:, :s.shape[1]] = s
    return pad.reshape(s.shape[0], nt, 128).max(axis=2)


def max_growth(tm):
    """Largest rise of a tile's maximum above the running maximum of the
    earlier tiles (tiles visited in increasing order), over all rows."""
    best = -np.inf
    run = tm[:, 0].copy()
    for t in range(1, tm.shape[1]):
        ok = np.isfinite(run) & np.isfinite(tm[:, t])
        if ok.any():
            best = max(best, float((tm[ok, t] - run[ok]).max()))
        run = np.fmax(run, tm[:, t])
    return best


def max_spread(tm):
    """Largest difference between two finite tile maxima of one row."""
    fin = np.where(np.isfinite(tm), tm, np.nan)
    return float(np.nanmax(np.nanmax(fin, axis=1) - np.nanmin(fin, axis=1)))


def check(o, lse, ref_o, ref_lse):
    o = o.float().cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy().astype(np.float64)
    err = np.abs(o - ref_o)
    bad = err > ATOL + RTOL * np.abs(ref_o)
    assert not bad.any(), f"{int(bad.sum())} O elements out of tolerance; max err {err.max():.3e}"
    lerr = np.abs(lse - ref_lse).max()
    assert lerr <= LSE_TOL, f"LSE max err {lerr:.3e}"


def run_case(E, B, H, N, d, gamma, seed, mask="none", window=0, grid=None, schedule=0,
             num_ctas=0, min_growth=TAU, min_spread=0.0):
    q, k, v = growing_qkv(B, H, N, d, gamma, seed)
    scale = 1.0 / math.sqrt(d)
    qf, kf, vf = to_f64(q), to_f64(k), to_f64(v)
    allowed = reference_np.mask_matrix(N, N, mask, window=window, grid=grid)
    tm = tile_maxima(qf[0, 0], kf[0, 0], scale, allowed)
    g, sp = max_growth(tm), max_spread(tm)
    assert g > min_growth, f"inputs too tame: largest growth {g:.1f} log2 units"
    assert sp > min_spread, f"inputs too tame: largest spread {sp:.1f} log2 units"
    o, lse = E.attn_fwd(q.cuda(), k.cuda(), v.cuda(), scale=scale, mask=mask, window=window,
                        grid=grid, schedule=schedule, num_ctas=num_ctas)
    torch.cuda.synchronize()
    code, detail = E.device_status()
    assert code == 0, (code, detail)
    ref_o, ref_lse = oracle.attention(qf, kf, vf, scale=scale, mask_kind=mask, window=window,
                                      grid=grid)
    check(o, lse, ref_o, ref_lse)
    return g, sp


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("mask", ["none", "causal"])
@pytest.mark.parametrize("schedule", [1, 2])
def test_rescale_dense(E, d, mask, schedule):
    """Growth of ~40-60 log2 units over 8 tiles: the maximum is renewed every
    tile or two. Schedule 1: whole tasks; 2: tasks cut over 3 CTAs (dense
    masks only), so parts with maxima tens of units apart are merged."""
    if schedule == 2 and mask != "none":
        pytest.skip("the split schedule applies to unmasked problems")
    run_case(E, 1, 2, 1024, d, 10.0 if d == 32 else 8.0, 700 + d, mask, schedule=schedule,
             num_ctas=3 if schedule == 2 else 0, min_spread=30.0)


@pytest.mark.parametrize("mode", ["clamp", "wrap"])
@pytest.mark.parametrize("d", [32, 64])
def test_rescale_neighbourhood(E, mode, d):
    """32x32 grid, window 7: each query visits 2-3 key tiles whose maxima
    differ by more than the threshold."""
    run_case(E, 1, 2, 1024, d, 40.0, 710 + d, mode, window=7, grid=(32, 32))


@pytest.mark.parametrize("num_ctas", [4, 8, 11])
def test_rescale_split_merge_underflow(E, num_ctas):
    """Maxima hundreds of log2 units apart along the sequence: in the merge of
    a cut task, 2^(m_i - M) underflows to zero for the earlier parts, and the
    result is that of the last parts alone."""
    run_case(E, 1, 2, 1024, 64, 60.0, 720 + num_ctas, schedule=2, num_ctas=num_ctas,
             min_growth=TAU, min_spread=150.0)
