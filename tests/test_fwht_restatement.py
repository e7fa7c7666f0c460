"""Pins of the tests' float32 restatement of the rotation (tests/fwht_f32.py):
it is the Sylvester Hadamard matrix product (scipy's) wherever float32 holds
every partial sum exactly, it inverts itself up to the factor n, and on random
data it stays within float32 rounding of the float64 product."""
import numpy as np
import pytest
from scipy.linalg import hadamard

from tests.fwht_f32 import sequential_transform_f32


@pytest.mark.parametrize("n", [2, 4, 64, 128, 256])
def test_equals_sylvester_matrix_on_exact_inputs(n):
    x = np.random.default_rng(n).integers(-1000, 1000, size=(5, n)).astype(np.float32)  # every sum exact
    want = x.astype(np.float64) @ hadamard(n).T.astype(np.float64)
    assert np.array_equal(sequential_transform_f32(x).astype(np.float64), want)


@pytest.mark.parametrize("n", [64, 128, 256])
def test_self_inverse_and_close_to_float64(n):
    x = np.random.default_rng(7 + n).standard_normal((9, n)).astype(np.float32)
    y = sequential_transform_f32(x)
    ref = x.astype(np.float64) @ hadamard(n).T.astype(np.float64)
    assert np.max(np.abs(y - ref)) <= 1e-5 * np.sqrt(n) * np.max(np.abs(ref))
    back = sequential_transform_f32(y) / n
    assert np.max(np.abs(back - x)) <= 1e-5


def test_butterfly_order_and_sign():
    # n = 4: stage h = 1 pairs (0, 1), (2, 3); stage h = 2 pairs (0, 2), (1, 3)
    x = np.array([[1.0, 2.0, 4.0, 8.0]], np.float32)
    assert sequential_transform_f32(x).tolist() == [[15.0, -5.0, -9.0, 3.0]]
