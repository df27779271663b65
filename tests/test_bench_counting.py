"""The benchmark's FLOP counting (CPU): the allowed-pair matrix it builds for
each masked workload equals the oracle twin's mask, and the counts equal their
closed forms. Every reported TFLOP/s divides these counts by time."""
import numpy as np
import pytest

import bench
from oracle import reference_np as twin
from seeded_inputs import WORKLOADS


def test_unmasked_counts():
    for name in ("sd21_single_head", "sd21_unet_block", "long_seq"):
        w = WORKLOADS[name]
        tile, exact = bench.count_flops(w)
        assert tile == exact == 4.0 * w.B * w.H * w.Nq * w.Nk * w.d


def test_causal_counts():
    w = WORKLOADS["lm_causal"]
    tile, exact = bench.count_flops(w)
    t = w.Nq // 128
    assert tile == 4.0 * w.B * w.H * w.d * 128 * 128 * (t * (t + 1) // 2)
    assert exact == 4.0 * w.B * w.H * w.d * (w.Nq * (w.Nq + 1) // 2)


@pytest.mark.parametrize("name", ["na2d_clamp", "na2d_wrap", "na3d_wrap2"])
def test_neighbourhood_matrix_matches_the_oracle_twin(name):
    w = WORKLOADS[name]
    m = bench.allowed_pairs_matrix(w)
    ref = twin.mask_matrix(w.Nq, w.Nk, w.mask, w.window, w.dilation, w.grid, w.wrap_axes)
    assert np.array_equal(m, ref)
    per_query = w.window ** len(w.grid)
    assert (m.sum(axis=1) == per_query).all()
    _, exact = bench.count_flops(w)
    assert exact == 4.0 * w.B * w.H * w.d * w.Nq * per_query
