"""Pins of the oracle's RMSNorm (``oracle.rmsnorm``) to facts that do not come
from the oracle itself: closed forms of constant rows, the unit mean square of
the normalised row, invariance under power-of-two scaling, the per-column
action of the weight, the place of eps under the square root, and row
independence. A dropped 1/K, a missing square root, eps outside the root, a
weight indexed by row instead of column, or rows mixed through a wrong stride
each fail one of these.

Source: "Deploying Hunyuan 770B in INT8 on domestic accelerators", §4.1
operator table (RMSNorm runs in high precision beside the INT8 GEMMs).
"""
import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.filterwarnings("error")

ONE = np.uint16(0x3F80)   # 1.0 in BF16


def bits(v):
    return workloads.f32_to_bf16_bits(np.asarray(v, dtype=np.float32))


def test_constant_row_normalises_to_its_sign():
    # mean(c^2) = c^2, so c / sqrt(c^2) = sign(c) for every K
    for c, K in [(3.0, 8), (-0.375, 136), (96.0, 4096), (-2.0 ** -20, 24)]:
        x = bits(np.full((1, K), c))
        y = oracle.rmsnorm(x, np.full(K, ONE), 0.0)
        np.testing.assert_array_equal(y, np.full((1, K), np.sign(c)))


def test_eps_sits_under_the_square_root():
    # c / sqrt(c^2 + 3 c^2) = sign(c) / 2 exactly
    for c in (0.5, -4.0, 48.0):
        K = 40
        x = bits(np.full((1, K), c))
        y = oracle.rmsnorm(x, np.full(K, ONE), 3.0 * c * c)
        np.testing.assert_array_equal(y, np.full((1, K), np.sign(c) * 0.5))


def test_unit_weight_gives_unit_mean_square():
    rng = np.random.default_rng(5)
    for K in (8, 100, 4096):
        x = bits(rng.standard_normal((4, K)) * rng.uniform(0.01, 100.0, (4, 1)))
        y = oracle.rmsnorm(x, np.full(K, ONE), 0.0)
        np.testing.assert_allclose(np.mean(y * y, axis=1), 1.0, rtol=1e-13)


def test_power_of_two_scaling_of_a_row_changes_nothing():
    rng = np.random.default_rng(6)
    K = 512
    x32 = rng.standard_normal((3, K)).astype(np.float32)
    g = bits(rng.normal(1.0, 0.25, K))
    y = oracle.rmsnorm(bits(x32), g, 0.0)
    for e in (-30, -3, 7, 40):
        np.testing.assert_array_equal(oracle.rmsnorm(bits(x32 * np.float32(2.0 ** e)), g, 0.0), y)


def test_weight_scales_each_column():
    rng = np.random.default_rng(7)
    K = 300 - 300 % 8
    x = bits(rng.standard_normal((5, K)))
    g = bits(rng.normal(1.0, 0.25, K))
    y1 = oracle.rmsnorm(x, np.full(K, ONE), 1e-5)
    yg = oracle.rmsnorm(x, g, 1e-5)
    np.testing.assert_allclose(yg, y1 * workloads.bf16_bits_to_f32(g).astype(np.float64)[None, :],
                               rtol=1e-15, atol=0)


def test_rows_are_independent():
    rng = np.random.default_rng(8)
    K = 64
    x = bits(rng.standard_normal((6, K)) * np.arange(1, 7)[:, None])
    g = bits(rng.normal(1.0, 0.25, K))
    y = oracle.rmsnorm(x, g, 1e-6)
    perm = np.array([3, 0, 5, 1, 4, 2])
    np.testing.assert_array_equal(oracle.rmsnorm(x[perm], g, 1e-6), y[perm])
    for m in range(6):
        np.testing.assert_array_equal(oracle.rmsnorm(x[m:m + 1], g, 1e-6), y[m:m + 1])


def test_two_element_row_by_hand():
    # x = (3, 4): mean square 25 / 2; with eps = 3.5 the root is sqrt(16) = 4
    x = bits([[3.0, 4.0]])
    g = bits([2.0, -0.5])
    np.testing.assert_array_equal(oracle.rmsnorm(x, g, 3.5), [[1.5, -0.5]])


def test_zero_row_stays_zero():
    K = 16
    y = oracle.rmsnorm(np.zeros((2, K), np.uint16), np.full(K, ONE), 1e-6)
    np.testing.assert_array_equal(y, np.zeros((2, K)))
