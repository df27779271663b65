"""The C ABI on the CPU: the library loads without a GPU, exports every
function include/attn.h declares, and rejects bad arguments on the host
before touching CUDA."""
import ctypes
import os
import re

import pytest

from exact_attention_69_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from exact_attention_69_gb300 import build
    build.build()
    return _lib.load()


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert "attn_fwd" in names and "attn_fwd_ex" in names
    for n in names:
        assert hasattr(lib, n), n


def test_struct_layout_and_version(lib):
    assert lib.attn_params_size() == ctypes.sizeof(_lib.AttnParamsEx)
    assert lib.attn_abi_version() == 6


def test_error_strings(lib):
    for code in range(6):
        assert lib.attn_error_string(code)
    assert b"unknown" in lib.attn_error_string(99)


def _base():
    p = _lib.params()
    p.q = p.k = p.v = p.o = 1 << 20
    p.B, p.H, p.Nq, p.Nk, p.d, p.scale = 1, 2, 256, 256, 64, 0.125
    return p


BAD = [
    ("B0", dict(B=0), _lib.ATTN_ERR_INVALID_ARG),
    ("Nk0", dict(Nk=0), _lib.ATTN_ERR_INVALID_ARG),
    ("d48", dict(d=48), _lib.ATTN_ERR_UNSUPPORTED),
    ("d256", dict(d=256), _lib.ATTN_ERR_UNSUPPORTED),
    ("scale_nan", dict(scale=float("nan")), _lib.ATTN_ERR_INVALID_ARG),
    ("scale_neg", dict(scale=-1.0), _lib.ATTN_ERR_INVALID_ARG),
    ("mask9", dict(mask_kind=9), _lib.ATTN_ERR_INVALID_ARG),
    ("window_without_na", dict(window=3), _lib.ATTN_ERR_INVALID_ARG),
    ("wrap_without_na", dict(wrap=1), _lib.ATTN_ERR_INVALID_ARG),
    ("na_even_window", dict(mask_kind=2, window=4), _lib.ATTN_ERR_INVALID_ARG),
    ("na_nonsquare", dict(mask_kind=2, window=3, Nq=250, Nk=250), _lib.ATTN_ERR_INVALID_ARG),
    ("na_q_ne_k", dict(mask_kind=2, window=3, Nq=256, Nk=289), _lib.ATTN_ERR_INVALID_ARG),
    ("na_window_too_big", dict(mask_kind=2, window=17), _lib.ATTN_ERR_INVALID_ARG),
    ("na_bad_grid", dict(mask_kind=2, window=3, grid_h=10, grid_w=20), _lib.ATTN_ERR_INVALID_ARG),
    ("na_dilation0", dict(mask_kind=2, window=3, dilation=0), _lib.ATTN_ERR_INVALID_ARG),
    ("na_dilated_window_too_big", dict(mask_kind=2, window=3, dilation=6), _lib.ATTN_ERR_INVALID_ARG),
    ("na_wrap4", dict(mask_kind=2, window=3, wrap=4), _lib.ATTN_ERR_INVALID_ARG),
    ("na_even_window_w", dict(mask_kind=2, window=3, window_w=2), _lib.ATTN_ERR_INVALID_ARG),
    ("na_window_w_too_big", dict(mask_kind=2, window=3, window_w=17), _lib.ATTN_ERR_INVALID_ARG),
    ("window_w_without_na", dict(window_w=3), _lib.ATTN_ERR_INVALID_ARG),
    ("null_q", dict(q=None), _lib.ATTN_ERR_INVALID_ARG),
    ("misaligned_k", dict(k=(1 << 20) + 8), _lib.ATTN_ERR_MISALIGNED),
    ("misaligned_lse", dict(lse=(1 << 20) + 2), _lib.ATTN_ERR_MISALIGNED),
    ("neg_ctas", dict(num_ctas=-1), _lib.ATTN_ERR_INVALID_ARG),
    ("schedule3", dict(schedule=3), _lib.ATTN_ERR_INVALID_ARG),
    ("misaligned_ws", dict(workspace=(1 << 20) + 4), _lib.ATTN_ERR_MISALIGNED),
    ("na3_no_grid", dict(mask_kind=3, window=3), _lib.ATTN_ERR_INVALID_ARG),
    ("na3_bad_volume", dict(mask_kind=3, window=3, grid_d=4, grid_h=8, grid_w=9), _lib.ATTN_ERR_INVALID_ARG),
    ("na3_wrap_d2", dict(mask_kind=3, window=3, grid_d=4, grid_h=8, grid_w=8, wrap_d=2),
     _lib.ATTN_ERR_INVALID_ARG),
    ("na3_even_window_d", dict(mask_kind=3, window=3, grid_d=4, grid_h=8, grid_w=8, window_d=2),
     _lib.ATTN_ERR_INVALID_ARG),
    ("na3_window_d_too_big", dict(mask_kind=3, window=3, grid_d=4, grid_h=8, grid_w=8, window_d=5),
     _lib.ATTN_ERR_INVALID_ARG),
    ("na3_dilated_depth_too_big", dict(mask_kind=3, window=3, grid_d=4, grid_h=8, grid_w=8, dilation=2),
     _lib.ATTN_ERR_INVALID_ARG),
    ("na3_q_ne_k", dict(mask_kind=3, window=3, grid_d=4, grid_h=8, grid_w=8, Nk=512),
     _lib.ATTN_ERR_INVALID_ARG),
    ("grid_d_without_na3", dict(mask_kind=2, window=3, grid_d=1), _lib.ATTN_ERR_INVALID_ARG),
    ("wrap_d_without_na3", dict(wrap_d=1), _lib.ATTN_ERR_INVALID_ARG),
    ("mask5", dict(mask_kind=5), _lib.ATTN_ERR_INVALID_ARG),
    ("causal_br_window", dict(mask_kind=4, window=3), _lib.ATTN_ERR_INVALID_ARG),
]


@pytest.mark.parametrize("name,changes,code", BAD, ids=[b[0] for b in BAD])
def test_rejects_bad_arguments_on_host(lib, name, changes, code):
    p = _base()
    for k, v in changes.items():
        setattr(p, k, v)
    assert _lib.fwd_ex(p) == code
    assert lib.attn_last_error()


def test_bad_strides(lib):
    p = _base()
    p.q_stride[:] = (256 * 64 * 2, 256 * 64, 60)
    assert _lib.fwd_ex(p) == _lib.ATTN_ERR_MISALIGNED
    p.q_stride[:] = (256 * 64 * 2, 0, 64)
    assert _lib.fwd_ex(p) == _lib.ATTN_ERR_INVALID_ARG


def test_plain_entry_point_validates(lib):
    # attn_fwd with an unsupported head dimension, never reaching CUDA
    assert lib.attn_fwd(16, 16, 16, 16, None, 1, 1, 8, 8, 40, ctypes.c_float(0.1), 0, 0, 1, 0) == \
        _lib.ATTN_ERR_UNSUPPORTED


def _bwd_base():
    p = _lib.bwd_params()
    p.q = p.k = p.v = p.o = p.dout = p.lse = p.dq = p.dk = p.dv = 1 << 20
    p.B, p.H, p.Nq, p.Nk, p.d, p.scale = 1, 2, 256, 256, 64, 0.125
    return p


BWD_BAD = [
    ("B0", dict(B=0), _lib.ATTN_ERR_INVALID_ARG),
    ("d48", dict(d=48), _lib.ATTN_ERR_UNSUPPORTED),
    ("mask9", dict(mask_kind=9), _lib.ATTN_ERR_INVALID_ARG),
    ("null_dout", dict(dout=None), _lib.ATTN_ERR_INVALID_ARG),
    ("null_dk", dict(dk=None), _lib.ATTN_ERR_INVALID_ARG),
    ("misaligned_dv", dict(dv=(1 << 20) + 8), _lib.ATTN_ERR_MISALIGNED),
    ("window_without_na", dict(window=3), _lib.ATTN_ERR_INVALID_ARG),
    ("na_even_window", dict(mask_kind=2, window=4), _lib.ATTN_ERR_INVALID_ARG),
    ("na_q_ne_k", dict(mask_kind=2, window=3, Nk=289), _lib.ATTN_ERR_INVALID_ARG),
    ("na_bad_grid", dict(mask_kind=2, window=3, grid_h=10, grid_w=20), _lib.ATTN_ERR_INVALID_ARG),
    ("na_dilated_window_too_big", dict(mask_kind=2, window=3, dilation=6), _lib.ATTN_ERR_INVALID_ARG),
    ("na_wrap4", dict(mask_kind=2, window=3, wrap=4), _lib.ATTN_ERR_INVALID_ARG),
    ("na3_bad_volume", dict(mask_kind=3, window=3, grid_d=4, grid_h=8, grid_w=9), _lib.ATTN_ERR_INVALID_ARG),
    ("na3_window_d_too_big", dict(mask_kind=3, window=3, grid_d=4, grid_h=8, grid_w=8, window_d=5),
     _lib.ATTN_ERR_INVALID_ARG),
    ("window_d_without_na3", dict(window_d=3), _lib.ATTN_ERR_INVALID_ARG),
]


@pytest.mark.parametrize("name,changes,code", BWD_BAD, ids=[b[0] for b in BWD_BAD])
def test_backward_rejects_bad_arguments_on_host(lib, name, changes, code):
    p = _bwd_base()
    for k, v in changes.items():
        setattr(p, k, v)
    assert _lib.bwd(p) == code
    assert lib.attn_last_error()


def test_backward_params_init_defaults(lib):
    p = _lib.bwd_params()
    assert p.dilation == 1 and p.window == 0 and p.wrap == 0 and p.mask_kind == 0


def test_tune_rejects_bad_arguments_on_host(lib):
    res = _lib.AttnTuneResult()
    p = _base()
    assert lib.attn_tune(ctypes.byref(p), 0, ctypes.byref(res)) == _lib.ATTN_ERR_INVALID_ARG
    assert lib.attn_tune(ctypes.byref(p), 5, None) == _lib.ATTN_ERR_INVALID_ARG
    assert lib.attn_tune(None, 5, ctypes.byref(res)) == _lib.ATTN_ERR_INVALID_ARG
