"""The oracle against facts other than itself (formats, closed forms, brute force)."""
import pytest

import oracle
from tests import oracle_pins


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(lib, check):
    check(lib)


def test_bad_arguments_rejected(lib):
    import numpy as np
    A = np.zeros((2, 3), np.uint16)
    B = np.zeros((4, 5), np.uint16)
    with pytest.raises(ValueError):
        oracle.gemm(oracle.BF16, A, B, lib=lib)
    with pytest.raises(ValueError):
        oracle.gemm_points(oracle.BF16, A, np.zeros((4, 3), np.uint16), [2], [0], lib=lib)
