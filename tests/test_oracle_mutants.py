"""Planted mistakes in copies of the oracle must each fail at least one pin.

Each mutant is a one-line textual change to a temporary copy of the C oracle
(the shipped source is never touched), compiled with gcc and run through the
same checks as tests/test_oracle_pins.py. A mutant that no check catches means
the pins leave that part of the oracle unpinned.
"""
import os

import pytest

import oracle
from tests import oracle_pins as pins
from tests.helpers import read_golden

GOLDENS = (read_golden("natten_issue142_wrap_5x5_k3.txt"),
           read_golden("na2d_clamp_5x5_k3_by_hand.txt"))

MUTANTS = {
    "causal_off_by_one": ("return j <= i;", "return j < i + (i == 0);"),
    "dropped_scale": ("scores[j] = p->scale * dot;", "scores[j] = dot;"),
    "lse_dropped_max": ("*lse_out = M + log(l);", "*lse_out = log(l);"),
    "v_wrong_operand": ("o_row[t] += w * vj[t];", "o_row[t] += w * qi[t % d];"),
    "key_index_transposed": ("const double* kj = kb + (int64_t)j * d;",
                             "const double* kj = kb + (int64_t)(j % (i + 1)) * d;"),
    "wrap_negative_modulo": ("if (c < 0) c += G;", ""),
    "clamp_no_upper_shift": ("if (start > len - k) start = len - k;", ""),
    "clamp_window_off_centre": ("int start = a - k / 2;", "int start = a - k / 2 + 1;"),
    "na_axis_swapped": (": axis_allowed_clamp(qx, kx, p->grid_w, p->window_w, p->dilation);",
                        ": axis_allowed_clamp(qx, kx, p->grid_h, p->window_w, p->dilation);"),
    "na_window_axes_swapped": (": axis_allowed_clamp(qy, ky, p->grid_h, p->window_h, p->dilation);",
                               ": axis_allowed_clamp(qy, ky, p->grid_h, p->window_w, p->dilation);"),
    "na_wrap_axes_swapped": ("const int row_ok = p->wrap_h ?", "const int row_ok = p->wrap_w ?"),
    "dilation_residue_ignored": ("if (kc % dl != residue) return 0;", ""),
    "softmax_sign": ("double w = exp(scores[j] - M);", "double w = exp(M - scores[j]);"),
    "causal_br_offset_off_by_one": ("return (int64_t)j <= (int64_t)i + (p->Nk - p->Nq);",
                                    "return (int64_t)j < (int64_t)i + (p->Nk - p->Nq);"),
    "causal_br_offset_reversed": ("return (int64_t)j <= (int64_t)i + (p->Nk - p->Nq);",
                                  "return (int64_t)j <= (int64_t)i + (p->Nq - p->Nk);"),
    "na3_depth_dropped": ("return axis_allowed(p->wrap_d, qt, kt, p->grid_d, p->window_d, p->dilation) &&",
                          "return 1 &&"),
    "na3_plane_stride": ("const int plane = p->grid_h * p->grid_w;",
                         "const int plane = p->grid_w * p->grid_w;"),
    "na3_depth_wrap_from_rows": ("axis_allowed(p->wrap_d, qt, kt,", "axis_allowed(p->wrap_h, qt, kt,"),
    "na3_depth_window_from_rows": ("p->grid_d, p->window_d, p->dilation)",
                                   "p->grid_d, p->window_h, p->dilation)"),
    "na3_axes_transposed": ("int kt = j / plane, ky = (j % plane) / p->grid_w, kx = j % p->grid_w;",
                            "int kx = j / plane, ky = (j % plane) / p->grid_w, kt = j % p->grid_w;"),
    "bwd_mask_transposed": ("      ok[j] = (unsigned char)allowed(p, i, j);\n      if (!ok[j]) continue;\n      double dot = 0.0;",
                            "      ok[j] = (unsigned char)allowed(p, j < p->Nq ? j : i, j < p->Nq ? i : j);\n      if (!ok[j]) continue;\n      double dot = 0.0;"),
    "bwd_dropped_d_term": ("const double dsij = pw[j] * (dp[j] - Di);", "const double dsij = pw[j] * dp[j];"),
    "bwd_dk_unscaled": ("dk[(int64_t)j * d + t] += p->scale * dsij * qi[t];",
                        "dk[(int64_t)j * d + t] += dsij * qi[t];"),
    "bwd_dv_wrong_weight": ("dv[(int64_t)j * d + t] += pw[j] * gi[t];",
                            "dv[(int64_t)j * d + t] += dp[j] * gi[t];"),
    "bwd_dp_wrong_operand": ("for (int t = 0; t < d; ++t) g += gi[t] * v[(int64_t)j * d + t];",
                             "for (int t = 0; t < d; ++t) g += gi[t] * k[(int64_t)j * d + t];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mutated = src.replace(old, new)
    path = os.path.join(tmp_path, f"mut_{name}.c")
    with open(path, "w") as f:
        f.write(mutated)
    lib = oracle.compile_oracle(path, os.path.join(tmp_path, f"libmut_{name}.so"))
    orc = oracle.Oracle(lib)
    caught = []
    for check_name, check in pins.all_checks(GOLDENS):
        try:
            check(orc)
        except (AssertionError, ValueError, IndexError):
            caught.append(check_name)
    assert caught, f"no pin catches the planted mistake {name}"
