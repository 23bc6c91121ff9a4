"""GPU parity of the RMSNorm entry points (through the C ABI) against the CPU
oracle.

* ``rmsnorm``: every BF16 output within half a BF16 ulp plus 2^-19 relative
  of the FP64 definition (the kernel's fp32 value before rounding is within
  2^-19 relative of the exact one: at most 32 sequential fma terms per thread
  and 10 tree levels in the sum of squares, then five rounded operations).
* ``rmsnorm_quant``: codes and scales bit-identical to the oracle's
  quantizer applied to the kernel's own BF16 rows (the quantization decision
  is taken on the same BF16 values on both sides), in both scale modes.
* ``rmsnorm_linear``: bit-identical to ``rmsnorm`` followed by ``linear`` on
  every GEMM path (CUDA-core GEMV, narrow and 256-row tensor-core tiles), and
  within the GEMM's bound of the oracle.

Source: "Deploying Hunyuan 770B in INT8 on domestic accelerators", §4.1
(RMSNorm in high precision next to the INT8 GEMMs) and §3.1 (per-token
dynamic INT8 activations).
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
EPS = np.float32(1e-6)


def _inputs(M, K, seed, pad=0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K)).astype(np.float32)
    ch = rng.choice(K, size=max(1, K // 200), replace=False)
    x[:, ch] *= 40.0                                    # outlier channels
    x *= rng.uniform(0.05, 20.0, (M, 1)).astype(np.float32)
    x_bits = workloads.f32_to_bf16_bits(x)
    g_bits = workloads.f32_to_bf16_bits(rng.normal(1.0, 0.25, K).astype(np.float32))
    big = np.zeros((M, K + pad), np.uint16)
    big[:, :K] = x_bits
    x_dev = to_dev_bf16(big)[:, :K]
    return x_bits, g_bits, x_dev, to_dev_bf16(g_bits)


def _check_norm(y_bits, x_bits, g_bits, eps):
    exact = oracle.rmsnorm(x_bits, g_bits, float(eps))
    y = workloads.bf16_bits_to_f32(y_bits).astype(np.float64)
    ulp = np.maximum(oracle.bf16_ulp(y_bits), oracle.bf16_ulp(oracle.bf16_round(exact)))
    bound = 0.5 * ulp + 2.0 ** -19 * np.abs(exact)
    err = np.abs(y - exact)
    assert np.all(err <= bound), f"{np.sum(err > bound)} outputs out of bound"


@pytest.mark.parametrize("M,K,pad", [
    (1, 8, 0), (3, 136, 8), (17, 1024, 0), (64, 4096, 0), (33, 4104, 16),
    (9, 8192, 0), (5, 16384, 0), (2, 32768, 0), (300, 2048, 0),
])
def test_rmsnorm_matches_the_definition(M, K, pad):
    x_bits, g_bits, x, g = _inputs(M, K, M * 7 + K, pad)
    y = w8.rmsnorm(x, g, float(EPS))
    torch.cuda.synchronize()
    _check_norm(bf16_bits_of(y), x_bits, g_bits, EPS)


@pytest.mark.parametrize("M,K,pow2", [(1, 8, False), (7, 264, True), (100, 4096, False),
                                      (12, 8192, True), (3, 32768, False)])
def test_rmsnorm_quant_is_the_quantizer_on_the_normalised_rows(M, K, pow2):
    x_bits, g_bits, x, g = _inputs(M, K, M * 11 + K)
    mode = w8.SCALE_POW2 if pow2 else w8.SCALE_AMAX
    y = w8.rmsnorm(x, g, float(EPS))
    qa, sa = w8.rmsnorm_quant(x, g, float(EPS), scale_mode=mode)
    torch.cuda.synchronize()
    y_bits = bf16_bits_of(y)
    _check_norm(y_bits, x_bits, g_bits, EPS)
    qa_o, sa_o = (oracle.quant_act_pow2 if pow2 else oracle.quant_act)(y_bits)
    np.testing.assert_array_equal(qa.cpu().numpy(), qa_o)
    np.testing.assert_array_equal(sa.cpu().numpy(), sa_o)


def test_zero_rows_give_zero_codes_and_scales():
    K = 1024
    x = torch.zeros((4, K), dtype=torch.bfloat16, device=DEV)
    x[1, 5] = 3.0
    g = torch.ones(K, dtype=torch.bfloat16, device=DEV)
    qa, sa = w8.rmsnorm_quant(x, g, 1e-5)
    torch.cuda.synchronize()
    assert torch.count_nonzero(qa[[0, 2, 3]]) == 0
    assert sa[[0, 2, 3]].eq(0).all()
    assert int(qa[1, 5]) == 127


@pytest.mark.parametrize("M,N,K,out", [
    (1, 300, 1024, "fp32"), (4, 256, 512, "bf16"),       # CUDA-core GEMV
    (16, 520, 2048, "bf16"), (100, 264, 1024, "fp32"),    # narrow / 128-row tiles
    (300, 384, 1280, "bf16"),                              # 256-row tiles, ragged
])
def test_rmsnorm_linear_equals_rmsnorm_then_linear(M, N, K, out):
    x_bits, g_bits, x, g = _inputs(M, K, M + N + K)
    rng = np.random.default_rng(N)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    qw, sw = w8.quant_weight(torch.from_numpy(w).to(DEV))
    dt = torch.float32 if out == "fp32" else torch.bfloat16
    y_fused = torch.full((M, N), float("nan"), dtype=dt, device=DEV)
    w8.rmsnorm_linear(x, g, float(EPS), qw, sw, out_dtype=dt, out=y_fused)
    xn = w8.rmsnorm(x, g, float(EPS))
    y_two = w8.linear(xn, qw, sw, out_dtype=dt)
    torch.cuda.synchronize()
    assert torch.equal(y_fused, y_two)
    qa_o, sa_o = oracle.quant_act(bf16_bits_of(xn))
    qw_o, sw_o = oracle.quant_weight(w)
    y_ref, T = oracle.gemm(qa_o, sa_o, qw_o, sw_o)
    if out == "fp32":
        err = np.abs(y_fused.cpu().numpy().astype(np.float64) - y_ref)
        assert np.all(err <= 1e-5 * T)
    else:
        check_bf16(bf16_bits_of(y_fused), y_ref, T)
    assert w8.device_error() == 0


def test_rejected_arguments():
    x = torch.zeros((2, 64), dtype=torch.bfloat16, device=DEV)
    g = torch.ones(64, dtype=torch.bfloat16, device=DEV)
    for eps in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(RuntimeError):
            w8.rmsnorm(x, g, eps)
    x12 = torch.zeros((2, 12), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(RuntimeError):
        w8.rmsnorm(x12, torch.ones(12, dtype=torch.bfloat16, device=DEV), 1e-5)
    with pytest.raises(ValueError):
        w8.rmsnorm(x, torch.ones(32, dtype=torch.bfloat16, device=DEV), 1e-5)
    empty = torch.zeros((0, 64), dtype=torch.bfloat16, device=DEV)
    qa, sa = w8.rmsnorm_quant(empty, g, 1e-5)
    assert qa.shape == (0, 64) and sa.shape == (0,)
