"""attn_fwd_noalloc: the entry point for callers that cannot allocate device
memory (code inside an allocator or memory pool, or an embedded runtime that
owns every allocation). It keeps its scratch in a fixed array inside the
library; here it is called through the C ABI and its outputs are compared with
those of the regular entry point, on two calls in a row with different inputs
(the second call runs over whatever the first left in the shared scratch), and
with the fp64 oracle directly; a large call followed by smaller ones checks
that what one call leaves in the shared array does not leak into the next;
an injected stall checks that its bounded waits report through
attn_get_device_status.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
from seeded_inputs import make_qkv, to_f64

pytestmark = pytest.mark.gpu

ATOL, RTOL, LSE_TOL = 1e-2, 1e-2, 1e-3


@pytest.fixture(scope="module")
def lib():
    from exact_attention_69_gb300 import _lib, build
    build.build()
    return _lib


def _params(_lib, q, k, v, o, lse, **extra):
    p = _lib.params()
    p.q, p.k, p.v, p.o, p.lse = q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr()
    p.B, p.H, p.Nq, p.d = q.shape
    p.Nk = k.shape[2]
    p.scale = 1.0 / math.sqrt(q.shape[-1])
    p.mask_kind = _lib.ATTN_MASK_NONE
    p.stream = torch.cuda.current_stream().cuda_stream
    for key, val in extra.items():
        setattr(p, key, val)
    return p


def _noalloc(_lib, q, k, v, **extra):
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    p = _params(_lib, q, k, v, o, lse, **extra)
    _lib.check(_lib.load().attn_fwd_noalloc(ctypes.byref(p)), "attn_fwd_noalloc")
    return o, lse


def _close(o, lse, ref_o, ref_lse):
    o, ref_o = o.float().cpu().numpy(), ref_o.float().cpu().numpy()
    err = np.abs(o - ref_o)
    assert (err <= ATOL + RTOL * np.abs(ref_o)).all(), f"O max err {err.max():.3e}"
    lerr = np.abs(lse.cpu().numpy() - ref_lse.cpu().numpy()).max()
    assert lerr <= LSE_TOL, f"LSE max err {lerr:.3e}"


@pytest.mark.parametrize("shape", [(2, 5, 4096, 4096, 64), (1, 3, 700, 1000, 128), (1, 2, 300, 300, 32)])
def test_noalloc_matches_regular_entry_point_twice(lib, shape):
    import exact_attention_69_gb300 as E
    B, H, Nq, Nk, d = shape
    for seed in (101, 202):  # two calls in a row, different inputs
        q, k, v = (t.cuda() for t in make_qkv(B, H, Nq, Nk, d, 0.5, seed + d))
        o, lse = _noalloc(lib, q, k, v)
        ref_o, ref_lse = E.attn_fwd(q, k, v)
        torch.cuda.synchronize()
        _close(o, lse, ref_o, ref_lse)


def test_noalloc_many_parts_per_task(lib):
    """Few CTAs per task cut into many parts: the merge runs from the fixed scratch."""
    import exact_attention_69_gb300 as E
    for seed in (7, 8):
        q, k, v = (t.cuda() for t in make_qkv(1, 1, 512, 4096, 64, 1.0, seed))
        o, lse = _noalloc(lib, q, k, v, num_ctas=20)
        ref_o, ref_lse = E.attn_fwd(q, k, v)
        torch.cuda.synchronize()
        _close(o, lse, ref_o, ref_lse)


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    """A problem needing more scratch than the fixed array is refused before
    any device work (the pointers are never dereferenced)."""
    q = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    p = lib.params()
    p.q = p.k = p.v = p.o = q.data_ptr()
    p.B, p.H, p.Nq, p.Nk, p.d = 4096, 64, 65536, 128, 128
    p.scale = 0.1
    rc = lib.load().attn_fwd_noalloc(ctypes.byref(p))
    assert rc == lib.ATTN_ERR_INVALID_ARG
    assert b"bytes of scratch" in lib.load().attn_last_error()


def test_noalloc_rejects_masks(lib):
    q = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    p = lib.params()
    p.q = p.k = p.v = p.o = q.data_ptr()
    p.B, p.H, p.Nq, p.Nk, p.d = 1, 1, 256, 256, 64
    p.scale = 0.1
    p.mask_kind = lib.ATTN_MASK_CAUSAL
    assert lib.load().attn_fwd_noalloc(ctypes.byref(p)) == lib.ATTN_ERR_INVALID_ARG


def _close_oracle(o, lse, q, k, v):
    ref_o, ref_lse = oracle.attention(to_f64(q.cpu()), to_f64(k.cpu()), to_f64(v.cpu()),
                                      scale=1.0 / math.sqrt(q.shape[-1]))
    err = np.abs(o.float().cpu().numpy() - ref_o)
    assert (err <= ATOL + RTOL * np.abs(ref_o)).all(), f"O max err {err.max():.3e}"
    lerr = np.abs(lse.cpu().numpy() - ref_lse).max()
    assert lerr <= LSE_TOL, f"LSE max err {lerr:.3e}"


@pytest.mark.parametrize("shape,num_ctas", [((1, 2, 700, 900, 64), 5), ((2, 1, 513, 1025, 32), 0),
                                            ((1, 1, 300, 2000, 128), 7)])
def test_noalloc_matches_the_oracle(lib, shape, num_ctas):
    B, H, Nq, Nk, d = shape
    q, k, v = (t.cuda() for t in make_qkv(B, H, Nq, Nk, d, 1.0, 300 + Nq))
    o, lse = _noalloc(lib, q, k, v, num_ctas=num_ctas)
    torch.cuda.synchronize()
    assert lib.device_status()[0] == 0
    _close_oracle(o, lse, q, k, v)


def test_noalloc_large_then_small_calls(lib):
    """A large call (many tasks, every SM, parts and arrival words all over the
    array) followed by smaller problems with other task counts and grids: each
    call must see only its own arrivals and parts."""
    import exact_attention_69_gb300 as E
    seq = [((2, 8, 4096, 4096, 64), 0), ((1, 1, 512, 4096, 64), 20), ((1, 3, 300, 700, 64), 3),
           ((2, 8, 4096, 4096, 64), 0), ((1, 1, 256, 1024, 64), 9)]
    for i, ((B, H, Nq, Nk, d), nc) in enumerate(seq):
        q, k, v = (t.cuda() for t in make_qkv(B, H, Nq, Nk, d, 1.0, 400 + i))
        o, lse = _noalloc(lib, q, k, v, num_ctas=nc)
        ref_o, ref_lse = E.attn_fwd(q, k, v)
        torch.cuda.synchronize()
        assert lib.device_status()[0] == 0
        _close(o, lse, ref_o, ref_lse)
        if Nq * Nk <= 700 * 700:
            _close_oracle(o, lse, q, k, v)


def test_noalloc_bounded_wait_is_reported(lib):
    """The loader withholds one K tile: the MMA warp's wait runs out after the
    short bound, the kernel stops, attn_get_device_status reports the timeout
    from the fixed array's status word (and clears it), and the next call is
    correct."""
    q, k, v = (t.cuda() for t in make_qkv(1, 1, 256, 1024, 64, 1.0, 12))
    _noalloc(lib, q, k, v, num_ctas=1, timeout_ns=20_000_000, inject=1)
    torch.cuda.synchronize()
    code, detail = lib.device_status()
    assert code == lib.ATTN_ERR_TIMEOUT and detail[0] == lib.ATTN_ERR_TIMEOUT, (code, detail)
    assert lib.device_status()[0] == 0  # reading cleared it
    o, lse = _noalloc(lib, q, k, v, num_ctas=3)
    torch.cuda.synchronize()
    assert lib.device_status()[0] == 0
    _close_oracle(o, lse, q, k, v)


def test_noalloc_after_shutdown(lib):
    """attn_shutdown forgets the array's device address; the next call looks it
    up again and works."""
    q, k, v = (t.cuda() for t in make_qkv(1, 2, 400, 600, 64, 1.0, 13))
    lib.load().attn_shutdown()
    o, lse = _noalloc(lib, q, k, v, num_ctas=4)
    torch.cuda.synchronize()
    assert lib.device_status()[0] == 0
    _close_oracle(o, lse, q, k, v)
