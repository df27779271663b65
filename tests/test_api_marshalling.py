"""The Python layer's argument marshalling onto the C parameter blocks (CPU:
no kernel runs). Each mask name and option set must land in the ABI fields
include/attn.h defines for it."""
import pytest

from exact_attention_69_gb300 import _lib, api


def _p():
    return _lib.params()


def test_plain_masks():
    for name, code in (("none", 0), ("causal", 1), ("causal_br", 4)):
        p = _p()
        api._set_mask(p, name, 0, 1, None, None)
        assert p.mask_kind == code and p.window == 0 and p.dilation == 1 and p.wrap == 0


def test_na2d_square_and_per_axis():
    p = _p()
    api._set_mask(p, "wrap", 7, 1, None, None)
    assert (p.mask_kind, p.window, p.window_w, p.wrap, p.grid_h, p.grid_w) == (2, 7, 0, 1, 0, 0)
    p = _p()
    api._set_mask(p, "clamp", (5, 3), 2, (20, 12), (True, False))
    assert (p.mask_kind, p.window, p.window_w, p.dilation, p.wrap) == (2, 5, 3, 2, 2)
    assert (p.grid_h, p.grid_w) == (20, 12)
    p = _p()
    api._set_mask(p, "clamp", 3, 1, (8, 8), (False, True))
    assert p.wrap == 3 and p.window_w == 0


def test_na3d_fields():
    p = _p()
    api._set_mask(p, "clamp", (3, 5, 7), 1, (4, 6, 8), (True, False, True))
    assert p.mask_kind == _lib.ATTN_MASK_NA3D
    assert (p.grid_d, p.grid_h, p.grid_w) == (4, 6, 8)
    assert (p.window_d, p.window, p.window_w) == (3, 5, 7)
    assert (p.wrap_d, p.wrap) == (1, 3)  # depth wraps; of rows and columns, the columns
    p = _p()
    api._set_mask(p, "wrap", 5, 1, (16, 16, 16), None)
    assert (p.window_d, p.window, p.window_w, p.wrap_d, p.wrap) == (0, 5, 0, 1, 1)


def test_rejections():
    with pytest.raises(ValueError):
        api._set_mask(_p(), "sliding", 3, 1, None, None)
    with pytest.raises(ValueError):
        api._set_mask(_p(), "clamp", (3, 3), 1, (4, 4, 4), None)  # two windows, three axes
    with pytest.raises(ValueError):
        api._set_mask(_p(), "clamp", 3, 1, (4, 4, 4), (True, False))


def test_bwd_block_mirrors_the_forward_fields():
    p = _lib.bwd_params()
    api._set_mask(p, "clamp", (3, 5, 7), 2, (6, 10, 14), (False, True, False))
    assert p.mask_kind == 3 and (p.grid_d, p.window_d, p.wrap_d) == (6, 3, 0)
    assert (p.window, p.window_w, p.wrap, p.dilation) == (5, 7, 2, 2)
