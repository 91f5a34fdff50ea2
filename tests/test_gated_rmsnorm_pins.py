"""Pins for the oracle's gated RMSNorm (CPU): closed forms and identities that
hold whatever the implementation, so that a wrong mean (a sum), a dropped eps,
a sign slip in the sigmoid, a missing or transposed weight or the wrong
reduction axis each fail one of them."""
import math

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

SIGMOID_1 = math.e / (1.0 + math.e)  # logistic(1) = e / (1 + e)


def test_two_entry_closed_form():
    # o = (3, 4): mean square 12.5, rms = 5 / sqrt(2); z = 1: silu(1) = e / (1 + e)
    y = oracle.gated_rmsnorm([[3.0, 4.0]], [[1.0, 1.0]], [1.0, 2.0], eps=0.0)
    expect = [3 * math.sqrt(2) / 5 * SIGMOID_1, 2 * 4 * math.sqrt(2) / 5 * SIGMOID_1]
    np.testing.assert_allclose(y[0], expect, rtol=1e-15)


def test_constant_row_with_eps():
    # a row of equal entries c: x / sqrt(c^2 + eps) = sign(c) |c| / sqrt(c^2 + eps)
    c, eps, d = -0.25, 0.01, 16
    z = np.full((1, d), 30.0)  # silu(30) = 30 up to e^-30
    w = np.full(d, 1.0 / 30.0)
    y = oracle.gated_rmsnorm(np.full((1, d), c), z, w, eps=eps)
    np.testing.assert_allclose(y, -0.25 / math.sqrt(0.0625 + 0.01), rtol=1e-12)


def test_unit_rms_and_direction():
    # with w = 1 / silu(z) constant the output is x / rms(x): rms 1, parallel to x
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 64)) * rng.uniform(0.1, 10.0, (5, 1))
    y = oracle.gated_rmsnorm(x, np.full_like(x, 40.0), np.full(64, 1.0 / 40.0), eps=0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=1e-12)
    ratio = y / x
    np.testing.assert_allclose(ratio, ratio[:, :1] * np.ones_like(ratio), rtol=1e-12)
    assert (ratio > 0).all()


def test_scale_invariance_rows_independent():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 32))
    z = rng.standard_normal((3, 32))
    w = rng.uniform(0.5, 1.5, 32)
    y = oracle.gated_rmsnorm(x, z, w, eps=0.0)
    s = np.array([[1e-3], [7.0], [1e4]])
    np.testing.assert_allclose(oracle.gated_rmsnorm(x * s, z, w, eps=0.0), y, rtol=1e-12)
    # rows do not mix: one row alone gives the same result
    np.testing.assert_allclose(oracle.gated_rmsnorm(x[1:2], z[1:2], w, eps=0.0), y[1:2], rtol=1e-15)


def test_silu_odd_part_identity():
    # silu(z) - silu(-z) = z, so y(z) - y(-z) = w * x / rms(x) * z
    rng = np.random.default_rng(5)
    x = rng.standard_normal((4, 16))
    z = rng.standard_normal((4, 16)) * 3
    w = rng.uniform(0.5, 1.5, 16)
    eps = 1e-6
    d = oracle.gated_rmsnorm(x, z, w, eps) - oracle.gated_rmsnorm(x, -z, w, eps)
    n = x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    np.testing.assert_allclose(d, w * n * z, rtol=1e-12, atol=1e-15)


def test_zero_gate_zero_row_and_extremes():
    x = np.zeros((1, 8))
    y = oracle.gated_rmsnorm(x, np.ones((1, 8)), np.ones(8), eps=1e-6)
    assert np.all(y == 0.0)  # a zero row stays zero (finite) when eps > 0
    rng = np.random.default_rng(6)
    x = rng.standard_normal((1, 8))
    assert np.all(oracle.gated_rmsnorm(x, np.zeros((1, 8)), np.ones(8)) == 0.0)  # silu(0) = 0
    y = oracle.gated_rmsnorm(x, np.full((1, 8), -800.0), np.ones(8))  # e^800 overflows: silu -> -0
    assert np.all(np.isfinite(y)) and np.all(np.abs(y) == 0.0)


def test_shape_errors():
    with pytest.raises(ValueError):
        oracle.gated_rmsnorm(np.ones((2, 4)), np.ones((2, 3)), np.ones(4))
    with pytest.raises(ValueError):
        oracle.gated_rmsnorm(np.ones((2, 4)), np.ones((2, 4)), np.ones(3))
