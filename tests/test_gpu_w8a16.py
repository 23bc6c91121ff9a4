"""GPU parity of the weight-only INT8 GEMM with BF16 activations (W8A16,
through the C ABI) against the CPU oracle: integer-valued activations with
unit scales reproduce the integer matmul exactly (every partial sum is an
integer below 2^24); otherwise FP32 outputs are within 1e-5 * T of the exact
value (T = sum_g |sw| * sum_k |a * qw|) and BF16 outputs within one ulp of the
correctly rounded exact value, or that bound plus half an ulp. Covers the
narrow, 96/128-row and 256-row tiles, padded activation rows, [128, 128]
block scales and the grouped (MoE expert) form.

Source: "Running DeepSeek-V4-Flash-Vision on 4xA800", §二 (MoE experts on a
weight-only INT8 runner with 16-bit activations, "WNA16").
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import moe_gemm_gb300 as w8  # noqa: E402
from tests.test_gpu_parity import bf16_bits_of, check_bf16, to_dev_bf16  # noqa: E402

DEV = torch.device("cuda:0")
G = 128


def test_integer_activations_with_unit_scales_give_the_integer_matmul():
    rng = np.random.default_rng(30)
    M, N, K = 40, 200, 256
    ai = rng.integers(-100, 101, (M, K))
    a = to_dev_bf16(workloads.f32_to_bf16_bits(ai.astype(np.float32)))
    qw_o = rng.integers(-127, 128, (N, K), dtype=np.int8)
    y = w8.w8a16_gemm(a, torch.from_numpy(qw_o).to(DEV),
                      torch.ones((N, K // G), device=DEV), out_dtype=torch.float32)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(y.cpu().numpy().astype(np.int64),
                                  ai @ qw_o.astype(np.int64).T)


def _check(y, y_ref, T, out):
    if out == "fp32":
        yv = y.cpu().numpy().astype(np.float64)
        assert not np.isnan(yv).any()
        err = np.abs(yv - y_ref)
        assert np.all(err <= 1e-5 * T), f"worst err/T {np.max(err / np.maximum(T, 1e-300)):.3e}"
    else:
        check_bf16(bf16_bits_of(y), y_ref, T)


@pytest.mark.parametrize("M,N,K,out,block_rows,pad", [
    (1, 300, 512, "fp32", 1, 0), (8, 256, 1024, "bf16", 1, 8), (40, 520, 384, "fp32", 128, 0),
    (100, 264, 512, "bf16", 1, 0), (300, 200, 640, "fp32", 128, 16), (513, 128, 256, "bf16", 1, 0),
])
def test_dense_w8a16(M, N, K, out, block_rows, pad):
    rng = np.random.default_rng(M + N + K)
    a_bits = workloads.f32_to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    qw, sw = w8.quant_weight(torch.from_numpy(w).to(DEV), block_rows=block_rows)
    qw_o, sw_o = oracle.quant_weight_blocks(w, block_rows, False)
    np.testing.assert_array_equal(qw.cpu().numpy(), qw_o)
    big = np.zeros((M, K + pad), np.uint16)
    big[:, :K] = a_bits
    a = to_dev_bf16(big)[:, :K]                      # row stride K + pad
    dt = torch.float32 if out == "fp32" else torch.bfloat16
    y = torch.full((M, N), float("nan"), dtype=dt, device=DEV)
    w8.w8a16_gemm(a, qw, sw, out_dtype=dt, out=y, sw_block_rows=block_rows)
    torch.cuda.synchronize()
    y_ref, T = oracle.w8a16_gemm(a_bits, qw_o, sw_o, block_rows)
    _check(y, y_ref, T, out)


def test_grouped_w8a16():
    rng = np.random.default_rng(31)
    R, E, N, K = 333, 6, 256, 384
    a_bits = workloads.f32_to_bf16_bits(rng.standard_normal((R, K)).astype(np.float32))
    off = workloads.random_offsets(rng, R, E)
    ws = [(rng.standard_normal((N, K)) * 0.02).astype(np.float32) for _ in range(E)]
    q = [w8.quant_weight(torch.from_numpy(w).to(DEV)) for w in ws]
    qw = torch.stack([x for x, _ in q])
    sw = torch.stack([s for _, s in q])
    y = torch.full((R, N), float("nan"), dtype=torch.float32, device=DEV)
    w8.w8a16_grouped_gemm(to_dev_bf16(a_bits), torch.from_numpy(off).to(DEV), qw, sw,
                          out_dtype=torch.float32, out=y)
    torch.cuda.synchronize()
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            continue
        y_ref, T = oracle.w8a16_gemm(a_bits[lo:hi], qw[e].cpu().numpy(), sw[e].cpu().numpy())
        _check(y[lo:hi], y_ref, T, "fp32")
    assert w8.device_error() == 0
