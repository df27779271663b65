"""The fp64 oracle against facts outside itself (CPU only)."""
import pytest

import oracle
from tests.helpers import read_golden
from tests import oracle_pins as pins

GOLDENS = (read_golden("natten_issue142_wrap_5x5_k3.txt"),
           read_golden("na2d_clamp_5x5_k3_by_hand.txt"))


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("name,check", pins.all_checks(GOLDENS), ids=lambda x: x if isinstance(x, str) else "")
def test_pin(orc, name, check):
    check(orc)


def test_twin_masks_agree_with_oracle_predicate(orc):
    """The numpy twin's window sets and the C predicate agree pair by pair."""
    from oracle import reference_np as twin
    for case in pins.CASES:
        m = twin.mask_matrix(case["Nq"], case["Nk"], case["mask_kind"], case.get("window", 0),
                             case.get("dilation", 1), case.get("grid"), case.get("wrap"))
        for i in range(case["Nq"]):
            for j in range(case["Nk"]):
                got = orc.allowed(i, j, Nq=case["Nq"], Nk=case["Nk"], mask_kind=case["mask_kind"],
                                  window=case.get("window", 0), dilation=case.get("dilation", 1),
                                  grid=case.get("grid"), wrap=case.get("wrap", False))
                assert got == bool(m[i, j]), (case, i, j)


def test_oracle_rejects_bad_problems(orc):
    import numpy as np
    z = np.zeros((1, 1, 25, 4))
    with pytest.raises(ValueError):
        orc.attention(z, z, z, scale=1.0, mask_kind="clamp", window=4)   # even window
    with pytest.raises(ValueError):
        orc.attention(z, z, z, scale=1.0, mask_kind="wrap", window=7)    # window > grid side
    with pytest.raises(ValueError):
        orc.attention(z, z, z, scale=1.0, mask_kind="clamp", window=3, grid=(4, 7))  # 28 != 25
