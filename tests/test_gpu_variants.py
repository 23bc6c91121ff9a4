"""GPU parity of the scale-format variants (through the C ABI) against the CPU
oracle: power-of-two (UE8M0) activation and weight scales, and [128, 128]
weight block scales, on every GEMM path (CUDA-core GEMV, narrow and K-split
tensor-core tiles, 96/128-row tiles, 256-row tiles, grouped). Bars as in
test_gpu_parity.py: codes, scales and INT32 group partials bit-exact, FP32
outputs within the stated bound, BF16 within one ulp or the cancellation
clause.

Source: "Running DeepSeek-V4-Flash-Vision on 4xA800", §一 (weights in
[128, 128] blocks with power-of-two UE8M0 scales).
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
from tests.test_gpu_parity import bf16_bits_of, check_bf16, check_fp32, to_dev_bf16  # noqa: E402

DEV = torch.device("cuda:0")
G = 128


def test_quant_act_pow2_bitexact():
    rng = np.random.default_rng(20)
    x = (rng.standard_normal((64, 1024)) * 10.0 ** rng.uniform(-30, 30, (64, 1))).astype(np.float32)
    x[5] = 0.0
    x[6, :] = 1e-38                       # subnormal-range rows
    bits = workloads.f32_to_bf16_bits(x)
    qa, sa = w8.quant_act(to_dev_bf16(bits), scale_mode=w8.SCALE_POW2)
    qa_o, sa_o = oracle.quant_act_pow2(bits)
    np.testing.assert_array_equal(qa.cpu().numpy(), qa_o)
    np.testing.assert_array_equal(sa.cpu().numpy().view(np.uint32), sa_o.view(np.uint32))


@pytest.mark.parametrize("block_rows,pow2", [(1, True), (128, False), (128, True)])
def test_quant_weight_blocks_bitexact(block_rows, pow2):
    rng = np.random.default_rng(21)
    w = (rng.standard_normal((300, 512)) * 0.02).astype(np.float32)
    w[7, 3] = 3.0
    qw, sw = w8.quant_weight(torch.from_numpy(w).to(DEV), block_rows=block_rows,
                             scale_mode=w8.SCALE_POW2 if pow2 else w8.SCALE_AMAX)
    qw_o, sw_o = oracle.quant_weight_blocks(w, block_rows, pow2)
    np.testing.assert_array_equal(qw.cpu().numpy(), qw_o)
    np.testing.assert_array_equal(sw.cpu().numpy().view(np.uint32), sw_o.view(np.uint32))


def _block_problem(seed, M, N, K, pow2):
    rng = np.random.default_rng(seed)
    a_bits = workloads.f32_to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    mode = w8.SCALE_POW2 if pow2 else w8.SCALE_AMAX
    qa, sa = w8.quant_act(to_dev_bf16(a_bits), scale_mode=mode)
    qw, sw = w8.quant_weight(torch.from_numpy(w).to(DEV), block_rows=128, scale_mode=mode)
    if pow2:
        qa_o, sa_o = oracle.quant_act_pow2(a_bits)
    else:
        qa_o, sa_o = oracle.quant_act(a_bits)
    qw_o, sw_o = oracle.quant_weight_blocks(w, 128, pow2)
    np.testing.assert_array_equal(qa.cpu().numpy(), qa_o)
    np.testing.assert_array_equal(qw.cpu().numpy(), qw_o)
    np.testing.assert_array_equal(sw.cpu().numpy().view(np.uint32), sw_o.view(np.uint32))
    return a_bits, (qa, sa, qw, sw), (qa_o, sa_o, qw_o, sw_o)


@pytest.mark.parametrize("M,N,K,out,pow2", [
    (1, 300, 512, "fp32", False),      # CUDA-core GEMV
    (3, 256, 384, "bf16", True),
    (16, 520, 1024, "fp32", True),     # narrow tiles, K split
    (50, 384, 256, "bf16", False),
    (100, 264, 512, "fp32", False),    # 96/128-row tiles
    (300, 200, 640, "bf16", True),     # 256-row tiles, ragged
])
def test_gemm_with_128x128_weight_blocks(M, N, K, out, pow2):
    a_bits, (qa, sa, qw, sw), (qa_o, sa_o, qw_o, sw_o) = _block_problem(M * 3 + N, M, N, K, pow2)
    dt = torch.float32 if out == "fp32" else torch.bfloat16
    y = torch.full((M, N), float("nan"), dtype=dt, device=DEV)
    _, P = w8.gemm(qa, sa, qw, sw, out_dtype=dt, out=y, debug_partials=True, sw_block_rows=128)
    y2 = torch.full((M, N), float("nan"), dtype=dt, device=DEV)
    w8.gemm(qa, sa, qw, sw, out_dtype=dt, out=y2, sw_block_rows=128)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(P.cpu().numpy(), oracle.group_partials(qa_o, qw_o))
    assert torch.equal(y, y2)
    y_ref, T = oracle.gemm_blocks(qa_o, sa_o, qw_o, sw_o, 128)
    if out == "fp32":
        check_fp32(y.cpu().numpy(), y_ref, T, K)
    else:
        check_bf16(bf16_bits_of(y), y_ref, T)
    # the fused quantizer + GEMM call gives the same result
    y3 = torch.full((M, N), float("nan"), dtype=dt, device=DEV)
    w8.linear(to_dev_bf16(a_bits), qw, sw, out_dtype=dt, out=y3, sw_block_rows=128,
              act_scale_mode=w8.SCALE_POW2 if pow2 else w8.SCALE_AMAX)
    torch.cuda.synchronize()
    assert torch.equal(y3, y)


def test_grouped_gemm_with_128x128_weight_blocks():
    rng = np.random.default_rng(22)
    R, E, N, K = 333, 5, 256, 384
    a_bits = workloads.f32_to_bf16_bits(rng.standard_normal((R, K)).astype(np.float32))
    off = workloads.random_offsets(rng, R, E)
    ws = [(rng.standard_normal((N, K)) * 0.02).astype(np.float32) for _ in range(E)]
    qa, sa = w8.quant_act(to_dev_bf16(a_bits))
    q = [w8.quant_weight(torch.from_numpy(w).to(DEV), block_rows=128) for w in ws]
    qw = torch.stack([x for x, _ in q])
    sw = torch.stack([s for _, s in q])
    y = torch.full((R, N), float("nan"), dtype=torch.float32, device=DEV)
    _, P = w8.grouped_gemm(qa, sa, torch.from_numpy(off).to(DEV), qw, sw, out_dtype=torch.float32,
                           out=y, debug_partials=True, sw_block_rows=128)
    torch.cuda.synchronize()
    qa_o, sa_o = oracle.quant_act(a_bits)
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            continue
        qw_o, sw_o = oracle.quant_weight_blocks(ws[e], 128, False)
        np.testing.assert_array_equal(qw[e].cpu().numpy(), qw_o)
        np.testing.assert_array_equal(P[lo:hi].cpu().numpy(),
                                      oracle.group_partials(qa_o[lo:hi], qw_o))
        y_ref, T = oracle.gemm_blocks(qa_o[lo:hi], sa_o[lo:hi], qw_o, sw_o, 128)
        check_fp32(y[lo:hi].cpu().numpy(), y_ref, T, K)
