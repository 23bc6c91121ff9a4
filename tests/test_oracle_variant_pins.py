"""Pins of the oracle's scale-format and weight-only variants (CPU only):
power-of-two (UE8M0) scales against exact rationals and their defining
inequalities; [128, 128] block scales against the per-row functions they
reduce to; the W8A16 GEMM against exact integer matmuls and numpy.

Source: "Running DeepSeek-V4-Flash-Vision on 4xA800", §一 (FP8 weights in
[128, 128] blocks with UE8M0 power-of-two scales) and §二 (MoE experts run by
a weight-only INT8 runner with 16-bit activations, "WNA16").
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads
from exact import f32_value, round_half_even


def _pow2_exponent(s):
    m, e = np.frexp(np.float64(s))
    assert m == 0.5, f"{s} is not a power of two"
    return int(e) - 1


def test_pow2_act_scales_are_the_smallest_power_of_two_above_amax_over_127():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal((40, 256)) * 10.0 ** rng.uniform(-6, 6, (40, 1))).astype(np.float32)
    x[3] = 0.0
    bits = workloads.f32_to_bf16_bits(x)
    qa, sa = oracle.quant_act_pow2(bits)
    for m in range(bits.shape[0]):
        row = [f32_value(v) for v in workloads.bf16_bits_to_f32(bits[m])]
        amax = max(abs(v) for v in row)
        e = _pow2_exponent(sa[m])
        s = Fraction(2) ** e
        if amax == 0:
            assert e == -127 and (qa[m] == 0).all()
            continue
        assert s >= amax / 127 and (e == -127 or s / 2 < amax / 127)
        want = [max(-127, min(127, round_half_even(v / s))) for v in row]   # x/s exact
        assert qa[m].tolist() == want
        assert np.abs(qa[m]).max() >= 64                                  # amax/s > 63.5


def test_weight_blocks_of_one_row_equal_the_per_row_groups():
    rng = np.random.default_rng(1)
    w = (rng.standard_normal((70, 384)) * 0.02).astype(np.float32)
    qw, sw = oracle.quant_weight_blocks(w, 1, False)
    qw_r, sw_r = oracle.quant_weight(w)
    np.testing.assert_array_equal(qw, qw_r)
    np.testing.assert_array_equal(sw, sw_r)


@pytest.mark.parametrize("pow2", [False, True])
def test_weight_128x128_blocks_share_one_scale(pow2):
    rng = np.random.default_rng(2)
    N, K = 300, 256                                   # a ragged last block of 44 rows
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    w[5, 7] = 0.5                                     # dominates block (0, 0)
    qw, sw = oracle.quant_weight_blocks(w, 128, pow2)
    assert sw.shape == (3, 2)
    for b in range(3):
        for g in range(2):
            blk = w[128 * b:128 * (b + 1), 128 * g:128 * (g + 1)]
            amax = f32_value(np.abs(blk).max())
            s = f32_value(sw[b, g])
            if pow2:
                e = _pow2_exponent(sw[b, g])
                assert s >= amax / 127 and Fraction(2) ** (e - 1) < amax / 127
            else:
                assert sw[b, g] == np.float32(np.abs(blk).max()) / np.float32(127)
            # every code of the block from the block's scale: x / s (IEEE)
            q = np.clip(np.rint((blk / sw[b, g]).astype(np.float32)), -127, 127)
            np.testing.assert_array_equal(qw[128 * b:128 * (b + 1), 128 * g:128 * (g + 1)], q)
    assert qw[5, 7] == (64 if pow2 else 127)          # 0.5 / 2^-7 with power-of-two scales


def test_gemm_blocks_reduces_to_the_per_row_gemm():
    rng = np.random.default_rng(3)
    M, N, K = 9, 200, 384
    qa = rng.integers(-127, 128, (M, K), dtype=np.int8)
    qw = rng.integers(-127, 128, (N, K), dtype=np.int8)
    sa = rng.random(M).astype(np.float32)
    sw_b = rng.random((2, K // 128)).astype(np.float32)
    y, T = oracle.gemm_blocks(qa, sa, qw, sw_b, 128)
    sw_rows = np.repeat(sw_b, 128, axis=0)[:N]
    y_r, T_r = oracle.gemm(qa, sa, qw, sw_rows)
    np.testing.assert_array_equal(y, y_r)
    np.testing.assert_array_equal(T, T_r)
    y1, _ = oracle.gemm_blocks(qa, sa, qw, sw_rows, 1)
    np.testing.assert_array_equal(y1, y_r)


def test_w8a16_gemm_is_the_integer_matmul_for_integer_activations():
    rng = np.random.default_rng(4)
    M, N, K = 7, 33, 256
    ai = rng.integers(-100, 101, (M, K))
    a = workloads.f32_to_bf16_bits(ai.astype(np.float32))       # exact in BF16
    qw = rng.integers(-127, 128, (N, K), dtype=np.int8)
    y, T = oracle.w8a16_gemm(a, qw, np.ones((N, K // 128), np.float32))
    exact = ai @ qw.astype(np.int64).T
    np.testing.assert_array_equal(y, exact.astype(np.float64))
    np.testing.assert_array_equal(T, np.abs(ai) @ np.abs(qw.astype(np.int64)).T)


@pytest.mark.parametrize("block_rows", [1, 128])
def test_w8a16_gemm_matches_numpy_group_sums(block_rows):
    rng = np.random.default_rng(5)
    M, N, K = 6, 140, 384
    a = workloads.f32_to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    af = workloads.bf16_bits_to_f32(a).astype(np.float64)
    qw = rng.integers(-127, 128, (N, K), dtype=np.int8)
    nb = (N + block_rows - 1) // block_rows
    sw = (rng.random((nb, K // 128)) * 1e-2).astype(np.float32)
    y, _ = oracle.w8a16_gemm(a, qw, sw, block_rows)
    P = np.einsum("mgk,ngk->mng", af.reshape(M, K // 128, 128),
                  qw.astype(np.float64).reshape(N, K // 128, 128))
    sw_rows = np.repeat(sw, block_rows, axis=0)[:N].astype(np.float64)
    want = np.einsum("mng,ng->mn", P, sw_rows)
    np.testing.assert_allclose(y, want, rtol=1e-13, atol=1e-13 * np.abs(want).max())
