"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bars (stated by the method's contract):
  * quantizer codes and scales, weight codes and scales, and the INT32 group
    partials (debug mode): bit-exact;
  * FP32 output: |y - y*| <= 1e-5 * T and <= (G + ceil(G/2) + 1) 2^-24 T,
    T = sum_g |sa sw P| (G group fmas, additions of K-split pieces, sa);
  * BF16 output: within 1 BF16 ulp of the correctly rounded y*, or
    |y - y*| <= 1e-5 T + ulp/2 (cancellation rows where T >> |y*|).
Outputs are poisoned with NaN first so unwritten elements are caught.
"""
import numpy as np
import pytest
import torch

import oracle
import parity_stats
import workloads

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU, never run there
    pytest.skip("needs a CUDA device", allow_module_level=True)

import moe_gemm_gb300 as w8  # noqa: E402

DEV = torch.device("cuda:0")
G = 128


# ---------------------------------------------------------------- helpers
def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(torch.bfloat16)


def bf16_bits_of(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def fp32_bound(K: int) -> float:
    """Relative FP32 bound on |Y - Y*| / T: G group fmas, at most ceil(G/2) - 1
    additions of K-split pieces, the token-scale multiply and one ulp of slack,
    capped by the 1e-5 * sum|terms| accuracy the FP32 output must meet."""
    Gn = K // G
    return min(1e-5, (Gn + (Gn + 1) // 2 + 1) * 2.0 ** -24)


def check_fp32(y: np.ndarray, y_ref: np.ndarray, T: np.ndarray, K: int):
    err = np.abs(y.astype(np.float64) - y_ref)
    assert not np.isnan(y).any(), "unwritten (NaN) outputs"
    bad = err > fp32_bound(K) * T
    assert not bad.any(), f"{bad.sum()} outputs out of tolerance; worst err/T {np.max(err / np.maximum(T, 1e-300)):.3e}"


def check_bf16(y_bits: np.ndarray, y_ref: np.ndarray, T: np.ndarray):
    ref_bits = oracle.bf16_round(y_ref)
    yv = oracle.bf16_to_float(y_bits)
    rv = oracle.bf16_to_float(ref_bits)
    assert not np.isnan(yv).any(), "unwritten (NaN) outputs"
    ulp = oracle.bf16_ulp(ref_bits)
    ok1 = np.abs(yv - rv) <= ulp
    ok2 = np.abs(yv - y_ref) <= 1e-5 * T + 0.5 * oracle.bf16_ulp(y_bits)
    bad = ~(ok1 | ok2)
    parity_stats.record_bf16(ok1.size, ok1.sum(), (ok2 & ~ok1).sum())
    assert not bad.any(), f"{bad.sum()} BF16 outputs out of tolerance"
    return ok1.mean()


def quantize_pair(a_bits, w):
    """GPU and oracle quantization of the same inputs; asserts bit-exactness."""
    a = to_dev_bf16(a_bits)
    qa, sa = w8.quant_act(a)
    qw, sw = w8.quant_weight(torch.from_numpy(np.ascontiguousarray(w)).to(DEV))
    qa_o, sa_o = oracle.quant_act(a_bits)
    qw_o, sw_o = oracle.quant_weight(w)
    np.testing.assert_array_equal(qa.cpu().numpy(), qa_o)
    np.testing.assert_array_equal(sa.cpu().numpy().view(np.uint32), sa_o.view(np.uint32))
    np.testing.assert_array_equal(qw.cpu().numpy(), qw_o)
    np.testing.assert_array_equal(sw.cpu().numpy().view(np.uint32), sw_o.view(np.uint32))
    return (qa, sa, qw, sw), (qa_o, sa_o, qw_o, sw_o)


def run_gemm(qa, sa, qw, sw, out_dtype, debug=False):
    M, N = qa.shape[0], qw.shape[0]
    y = torch.full((M, N), float("nan"), dtype=out_dtype, device=DEV)
    r = w8.gemm(qa, sa, qw, sw, out_dtype=out_dtype, out=y, debug_partials=debug)
    torch.cuda.synchronize()
    return r


# ------------------------------------------------------------- quantizers
@pytest.mark.parametrize("M,K", [(16, 1024), (3, 8192), (5, 16384), (7, 100), (2, 24576), (1, 8)])
def test_quant_act_bitexact(M, K):
    rng = np.random.default_rng(M * 1000 + K)
    x = rng.standard_normal((M, K)).astype(np.float32)
    x[0, : min(K, 64)] *= 50
    if M > 2:
        x[1] = 0.0                                   # amax = 0 row
        x[2] *= 2.0 ** -130                          # subnormal scale row
    bits = workloads.f32_to_bf16_bits(x)
    a = to_dev_bf16(bits)
    qa, sa = w8.quant_act(a)
    qa_o, sa_o = oracle.quant_act(bits)
    np.testing.assert_array_equal(qa.cpu().numpy(), qa_o)
    np.testing.assert_array_equal(sa.cpu().numpy().view(np.uint32), sa_o.view(np.uint32))


@pytest.mark.parametrize("M,K,pad,pow2", [
    (65, 1024, 0, False), (300, 4104, 8, False), (1000, 16384, 0, False), (129, 24, 8, True),
    (2000, 8192, 16, True), (70, 24576, 0, False),
])
def test_quant_act_many_rows_bitexact(M, K, pad, pow2):
    """More than 64 rows (K <= 16384, aligned) take the persistent row stream;
    K = 24576 takes the one-CTA-per-row kernel. Rows of every kind (zero,
    subnormal scale, halves, large) land in different CTAs and ring buffers,
    and the input rows may be padded (lda > K)."""
    rng = np.random.default_rng(M + K + pad)
    x = rng.standard_normal((M, K)).astype(np.float32)
    x *= rng.uniform(0.01, 30.0, (M, 1)).astype(np.float32)
    x[0, : min(K, 64)] *= 50
    x[1] = 0.0                                       # amax = 0 row
    x[2] *= 2.0 ** -130                              # subnormal scale row
    x[M - 1, : min(K, 8)] = [127.0, 2.5, 3.5, -2.5, 0.5, 1.5, 126.5, -126.5][: min(K, 8)]
    x[M - 1, 8:] = 0.0                               # ties at amax 127
    bits = workloads.f32_to_bf16_bits(x)
    big = np.zeros((M, K + pad), np.uint16)
    big[:, :K] = bits
    a = to_dev_bf16(big)[:, :K]
    mode = w8.SCALE_POW2 if pow2 else w8.SCALE_AMAX
    qa, sa = w8.quant_act(a, scale_mode=mode)
    qa_o, sa_o = (oracle.quant_act_pow2 if pow2 else oracle.quant_act)(bits)
    np.testing.assert_array_equal(qa.cpu().numpy(), qa_o)
    np.testing.assert_array_equal(sa.cpu().numpy().view(np.uint32), sa_o.view(np.uint32))
    assert w8.device_error() == 0


@pytest.mark.parametrize("M", [65, 300])
def test_linear_fp16_codes_equal_int8_codes_path(M):
    """The fused linear writes fp16 codes with the row stream (> 64 rows); the
    GEMM on the int8 codes of quant_act must give the same output, bit for bit."""
    K, N = 2048, 384
    rng = np.random.default_rng(M)
    bits = workloads.f32_to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    a = to_dev_bf16(bits)
    qw, sw = w8.quant_weight((torch.randn(N, K, device=DEV) * 0.02).float())
    qa, sa = w8.quant_act(a)
    y0 = run_gemm(qa, sa, qw, sw, torch.bfloat16)
    y1 = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    w8.linear(a, qw, sw, out_dtype=torch.bfloat16, out=y1)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1)


def test_quant_act_ties_and_strided_rows():
    rows = np.zeros((4, 256), np.float32)
    rows[0, :10] = [127.0, 2.5, 3.5, -2.5, 0.5, 1.5, 126.5, -126.5, -0.5, 5.5]
    rows[1, :5] = [254.0, 5.0, 7.0, -3.0, 1.0]
    rows[2] = np.linspace(-1, 1, 256)
    rows[3] = -np.linspace(0, 3, 256)
    bits = workloads.f32_to_bf16_bits(rows)
    big = np.zeros((4, 320), np.uint16)
    big[:, :256] = bits                              # lda = 320 > K
    a = to_dev_bf16(big)[:, :256]
    qa, sa = w8.quant_act(a)
    qa_o, sa_o = oracle.quant_act(bits)
    np.testing.assert_array_equal(qa.cpu().numpy(), qa_o)
    np.testing.assert_array_equal(sa.cpu().numpy(), sa_o)
    assert qa_o[0, :10].tolist() == [127, 2, 4, -2, 0, 2, 126, -126, 0, 6]


def test_quant_act_workload_rows_bitexact():
    for name, rows in (("decode_m32", None), ("prefill", np.arange(0, 4096, 97)),
                       ("stress", np.arange(0, 8192, 511))):
        spec = workloads.DENSE[name]
        bits = workloads.activations(spec, rows=rows)
        qa, sa = w8.quant_act(to_dev_bf16(bits))
        qa_o, sa_o = oracle.quant_act(bits)
        np.testing.assert_array_equal(qa.cpu().numpy(), qa_o)
        np.testing.assert_array_equal(sa.cpu().numpy().view(np.uint32), sa_o.view(np.uint32))


@pytest.mark.parametrize("N,K", [(3, 128), (64, 1024), (5, 4096)])
def test_quant_weight_bitexact(N, K):
    rng = np.random.default_rng(N + K)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    w[0, :128] = 0.0
    qw, sw = w8.quant_weight(torch.from_numpy(w).to(DEV))
    qw_o, sw_o = oracle.quant_weight(w)
    np.testing.assert_array_equal(qw.cpu().numpy(), qw_o)
    np.testing.assert_array_equal(sw.cpu().numpy().view(np.uint32), sw_o.view(np.uint32))


# ------------------------------------------------------------------ dense
def test_tiny_config_partials_bitexact_fp32():
    spec = workloads.DENSE["tiny"]
    (qa, sa, qw, sw), (qa_o, sa_o, qw_o, sw_o) = quantize_pair(
        workloads.activations(spec), workloads.weights(spec))
    y, P = run_gemm(qa, sa, qw, sw, torch.float32, debug=True)
    np.testing.assert_array_equal(P.cpu().numpy(), oracle.group_partials(qa_o, qw_o))
    y_ref, T = oracle.gemm(qa_o, sa_o, qw_o, sw_o)
    check_fp32(y.cpu().numpy(), y_ref, T, spec.K)


def test_integer_matmul_with_unit_scales():
    # sa = sw = 1 with integer codes reproduces the integer matmul exactly.
    rng = np.random.default_rng(0)
    M, N, K = 40, 256, 512
    qa_o = rng.integers(-127, 128, (M, K), dtype=np.int8)
    qw_o = rng.integers(-127, 128, (N, K), dtype=np.int8)
    qa, qw = torch.from_numpy(qa_o).to(DEV), torch.from_numpy(qw_o).to(DEV)
    sa = torch.ones(M, device=DEV)
    sw = torch.ones(N, K // G, device=DEV)
    y = run_gemm(qa, sa, qw, sw, torch.float32)
    exact = qa_o.astype(np.int64) @ qw_o.astype(np.int64).T
    np.testing.assert_array_equal(y.cpu().numpy().astype(np.int64), exact)


def test_extreme_codes_partials():
    M, N, K = 32, 128, 256
    qa_o = np.full((M, K), 127, np.int8)
    qw_o = np.full((N, K), 127, np.int8)
    qw_o[1::2] = -127
    qa, qw = torch.from_numpy(qa_o).to(DEV), torch.from_numpy(qw_o).to(DEV)
    _, P = run_gemm(qa, torch.ones(M, device=DEV), qw, torch.ones(N, 2, device=DEV),
                    torch.float32, debug=True)
    P = P.cpu().numpy()
    assert (P[:, 0::2] == 2064512).all() and (P[:, 1::2] == -2064512).all()


@pytest.mark.parametrize("M,N,K,out", [
    (1, 128, 128, "fp32"), (17, 200, 384, "bf16"), (100, 384, 256, "fp32"),
    (129, 256, 512, "bf16"), (255, 136, 128, "fp32"), (256, 128, 640, "bf16"),
    (300, 264, 256, "fp32"), (513, 128, 256, "bf16"),
])
def test_dense_ragged_shapes(M, N, K, out):
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    a_bits = workloads.f32_to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    (qa, sa, qw, sw), (qa_o, sa_o, qw_o, sw_o) = quantize_pair(a_bits, w)
    dt = torch.float32 if out == "fp32" else torch.bfloat16
    y, P = run_gemm(qa, sa, qw, sw, dt, debug=True)
    np.testing.assert_array_equal(P.cpu().numpy(), oracle.group_partials(qa_o, qw_o))
    # the kernel without the partials output computes the same outputs
    assert torch.equal(run_gemm(qa, sa, qw, sw, dt), y)
    y_ref, T = oracle.gemm(qa_o, sa_o, qw_o, sw_o)
    if out == "fp32":
        check_fp32(y.cpu().numpy(), y_ref, T, K)
    else:
        check_bf16(bf16_bits_of(y), y_ref, T)


def test_zero_rows_give_zero_outputs():
    M, N, K = 20, 128, 256
    rng = np.random.default_rng(1)
    x = rng.standard_normal((M, K)).astype(np.float32)
    x[[0, 7, 19]] = 0.0
    (qa, sa, qw, sw), _ = quantize_pair(workloads.f32_to_bf16_bits(x),
                                        (rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    y = run_gemm(qa, sa, qw, sw, torch.float32).cpu().numpy()
    assert (y[[0, 7, 19]] == 0).all()


def test_gemm_m0_is_noop():
    qa = torch.empty((0, 128), dtype=torch.int8, device=DEV)
    qw = torch.zeros((128, 128), dtype=torch.int8, device=DEV)
    y = w8.gemm(qa, torch.empty(0, device=DEV), qw, torch.ones(128, 1, device=DEV))
    assert y.shape == (0, 128)


# ---------------------------------------------------------------- grouped
def make_grouped(rng, R, E, N, K, off):
    a_bits = workloads.f32_to_bf16_bits(rng.standard_normal((R, K)).astype(np.float32))
    w = (rng.standard_normal((E * N, K)) * 0.02).astype(np.float32)
    (qa, sa, qw, sw), (qa_o, sa_o, qw_o, sw_o) = quantize_pair(a_bits, w)
    return ((qa, sa, qw.view(E, N, K), sw.view(E, N, K // G)),
            (qa_o, sa_o, qw_o.reshape(E, N, K), sw_o.reshape(E, N, K // G)))


@pytest.mark.parametrize("R,E,N,K,out", [
    (23, 5, 128, 256, "fp32"), (600, 7, 256, 384, "bf16"), (1000, 16, 128, 128, "fp32"),
])
def test_grouped_ragged(R, E, N, K, out):
    rng = np.random.default_rng(R + E)
    off = workloads.random_offsets(rng, R, E, empty_frac=0.3)
    off[E // 2 + 1:] = np.maximum(off[E // 2 + 1:], off[E // 2])
    (qa, sa, qw, sw), (qa_o, sa_o, qw_o, sw_o) = make_grouped(rng, R, E, N, K, off)
    dt = torch.float32 if out == "fp32" else torch.bfloat16
    y = torch.full((R, N), float("nan"), dtype=dt, device=DEV)
    y, P = w8.grouped_gemm(qa, sa, torch.from_numpy(off).to(DEV), qw, sw, out_dtype=dt, out=y,
                           debug_partials=True)
    torch.cuda.synchronize()
    y_ref, T = oracle.grouped_gemm(qa_o, sa_o, off, qw_o, sw_o)
    # partials: per routed row against its expert
    Pn = P.cpu().numpy()
    for e in range(E):
        lo, hi = off[e], off[e + 1]
        if hi > lo:
            np.testing.assert_array_equal(Pn[lo:hi], oracle.group_partials(qa_o[lo:hi], qw_o[e]))
    if out == "fp32":
        check_fp32(y.cpu().numpy(), y_ref, T, K)
    else:
        check_bf16(bf16_bits_of(y), y_ref, T)


def test_grouped_uncovered_rows_untouched_and_single_expert():
    rng = np.random.default_rng(5)
    R, E, N, K = 50, 3, 128, 256
    off = np.array([5, 20, 20, 41], np.int32)           # rows 0-4 and 41-49 uncovered
    (qa, sa, qw, sw), (qa_o, sa_o, qw_o, sw_o) = make_grouped(rng, R, E, N, K, off)
    y = torch.full((R, N), float("nan"), dtype=torch.float32, device=DEV)
    w8.grouped_gemm(qa, sa, torch.from_numpy(off).to(DEV), qw, sw, out_dtype=torch.float32, out=y)
    yn = y.cpu().numpy()
    assert np.isnan(yn[:5]).all() and np.isnan(yn[41:]).all()
    y_ref, T = oracle.grouped_gemm(qa_o, sa_o, off, qw_o, sw_o)
    check_fp32(yn[5:41], y_ref[5:41], T[5:41], K)
    # all rows in one expert == dense
    off1 = np.array([0, 0, R, R], np.int32)
    y1 = w8.grouped_gemm(qa, sa, torch.from_numpy(off1).to(DEV), qw, sw, out_dtype=torch.float32)
    yd = w8.gemm(qa, sa, qw[1].contiguous(), sw[1].contiguous(), out_dtype=torch.float32)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(y1.cpu().numpy(), yd.cpu().numpy())


def test_moe_t16_many_empty_segments():
    spec = workloads.MOE["moe_t16"]
    route = workloads.routing(spec)
    a_bits = workloads.moe_activations(spec, "down", route)
    R, E, N, K = spec.R, spec.E, spec.N_down, spec.K_down
    w = np.concatenate([workloads.moe_weights(spec, "down", e) for e in range(E)])
    (qa, sa, qw, sw), (qa_o, sa_o, qw_o, sw_o) = quantize_pair(a_bits, w)
    off = route.offsets
    y = torch.full((R, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    w8.grouped_gemm(qa, sa, torch.from_numpy(off).to(DEV), qw.view(E, N, K),
                    sw.view(E, N, K // G), out=y)
    torch.cuda.synchronize()
    y_ref, T = oracle.grouped_gemm(qa_o, sa_o, off, qw_o.reshape(E, N, K),
                                   sw_o.reshape(E, N, K // G))
    check_bf16(bf16_bits_of(y), y_ref, T)


def test_no_device_error_recorded():
    assert w8.device_error(clear=True) == 0


# ------------------------------------------------------- K-split (stream-K)
def _staging_only(rows, K):
    """A workspace holding only the fp16 staging copy: tiles are never split."""
    return torch.empty((rows * K * 2 + 255) // 256 * 256, dtype=torch.uint8, device=DEV)


@pytest.mark.parametrize("M,N,K,out", [
    (8, 4096, 8192, "fp32"),     # 32 tiles of 32 steps over all SMs: ~5 pieces per tile
    (5, 1000, 1152, "bf16"),     # odd group count, one step per CTA, ragged N
    (6, 28672, 1024, "fp32"),    # 224 tiles, ranges cross tile boundaries
    (33, 1000, 1152, "bf16"),    # tensor-core path: 8 tiles x 5 steps, one step per CTA
    (9, 2000, 2048, "fp32"),     # tensor-core path: 16 tiles x 8 steps over 128 CTAs
    (17, 28672, 1024, "bf16"),   # tensor-core path: one whole wave, 72 tiles split
    (64, 4096, 8192, "fp32"),    # tensor-core path: ~5 pieces per tile, 64-row tiles
    (20, 32256, 1024, "fp32"),   # 252 tiles: 100 left over > half a wave -> contiguous ranges,
    (40, 32256, 1024, "bf16"),   #   CTAs with two split pieces (32-row and 64-row tiles)
])
def test_dense_k_split_matches_oracle_and_unsplit(M, N, K, out):
    rng = np.random.default_rng(M + N + K)
    a_bits = workloads.f32_to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    (qa, sa, qw, sw), (qa_o, sa_o, qw_o, sw_o) = quantize_pair(a_bits, w)
    dt = torch.float32 if out == "fp32" else torch.bfloat16
    y_ref, T = oracle.gemm(qa_o, sa_o, qw_o, sw_o)
    ys = []
    for ws in (None, None, _staging_only(M, K)):     # split twice, then unsplit
        y = torch.full((M, N), float("nan"), dtype=dt, device=DEV)
        w8.gemm(qa, sa, qw, sw, out_dtype=dt, out=y, workspace=ws)
        torch.cuda.synchronize()
        ys.append(y)
        if out == "fp32":
            check_fp32(y.cpu().numpy(), y_ref, T, K)
        else:
            check_bf16(bf16_bits_of(y), y_ref, T)
    # the split result does not depend on which CTA finishes a tile last
    assert torch.equal(ys[0], ys[1])
    _, P = w8.gemm(qa, sa, qw, sw, out_dtype=dt, debug_partials=True)
    np.testing.assert_array_equal(P.cpu().numpy(), oracle.group_partials(qa_o, qw_o))
    assert w8.device_error(clear=True) == 0


def test_grouped_minimal_workspace_matches_oracle():
    rng = np.random.default_rng(77)
    R, E, N, K = 300, 6, 256, 1280
    off = workloads.random_offsets(rng, R, E, empty_frac=0.2)
    (qa, sa, qw, sw), (qa_o, sa_o, qw_o, sw_o) = make_grouped(rng, R, E, N, K, off)
    offs = torch.from_numpy(off).to(DEV)
    y_ref, T = oracle.grouped_gemm(qa_o, sa_o, off, qw_o, sw_o)
    covered = slice(int(off[0]), int(off[E]))
    for ws in (None, _staging_only(R, K)):
        y = torch.full((R, N), float("nan"), dtype=torch.float32, device=DEV)
        w8.grouped_gemm(qa, sa, offs, qw, sw, out_dtype=torch.float32, out=y, workspace=ws)
        torch.cuda.synchronize()
        check_fp32(y.cpu().numpy()[covered], y_ref[covered], T[covered], K)
    assert w8.device_error(clear=True) == 0


# --------------------------------------------- fused quantizer + GEMM entry
def _linear_only_workspace(M, K):
    """Codes and scales only: tiles are never split."""
    n = (M * K * 2 + 255) // 256 * 256 + (M * 4 + 255) // 256 * 256
    return torch.empty(n, dtype=torch.uint8, device=DEV)


@pytest.mark.parametrize("M,N,K,out,lda_pad", [
    (1, 1000, 1152, "bf16", 0),     # CUDA-core GEMV path (int8 codes in the workspace)
    (2, 20480, 512, "fp32", 0),     # GEMV: 160 tiles, 8 left over cut in 64-row halves
    (3, 256, 384, "fp32", 8),       # GEMV quantizing its own rows, strided activations
    (4, 512, 256, "bf16", 4),       # row stride not a multiple of 8: quantizer kernel + GEMV
    (8, 4096, 2048, "fp32", 0),     # tensor-core path, split
    (33, 1000, 1152, "bf16", 0),    # tensor-core path, split, ragged N
    (64, 28672, 1024, "bf16", 16),  # 64-row tiles, strided activations
    (130, 384, 640, "fp32", 0),     # 128-row tiles (wide form), ragged token tail
])
def test_linear_equals_quant_then_gemm(M, N, K, out, lda_pad):
    rng = np.random.default_rng(M + 3 * N + K)
    a_bits = workloads.f32_to_bf16_bits(rng.standard_normal((M, K + lda_pad)).astype(np.float32))
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    a_full = to_dev_bf16(a_bits)
    a = a_full[:, :K]                                   # row stride K + lda_pad
    qw, sw = w8.quant_weight(torch.from_numpy(np.ascontiguousarray(w)).to(DEV))
    dt = torch.float32 if out == "fp32" else torch.bfloat16
    qa, sa = w8.quant_act(a.contiguous())
    y_two = w8.gemm(qa, sa, qw, sw, out_dtype=dt)
    for ws in (None, _linear_only_workspace(M, K)):
        y = torch.full((M, N), float("nan"), dtype=dt, device=DEV)
        w8.linear(a, qw, sw, out_dtype=dt, out=y, workspace=ws)
        torch.cuda.synchronize()
        if ws is None:   # same codes, scales, kernels and split as the two calls
            assert torch.equal(y, y_two)
        qa_o, sa_o = oracle.quant_act(np.ascontiguousarray(a_bits[:, :K]))
        y_ref, T = oracle.gemm(qa_o, sa_o, *oracle.quant_weight(w))
        if out == "fp32":
            check_fp32(y.cpu().numpy(), y_ref, T, K)
        else:
            check_bf16(bf16_bits_of(y), y_ref, T)
    assert w8.device_error(clear=True) == 0


def test_grouped_linear_equals_quant_then_grouped_gemm():
    rng = np.random.default_rng(91)
    R, E, N, K = 700, 9, 256, 512
    off = workloads.random_offsets(rng, R, E, empty_frac=0.3)
    a_bits = workloads.f32_to_bf16_bits(rng.standard_normal((R, K)).astype(np.float32))
    w = (rng.standard_normal((E * N, K)) * 0.02).astype(np.float32)
    a = to_dev_bf16(a_bits)
    qw, sw = w8.quant_weight(torch.from_numpy(w).to(DEV))
    qw, sw = qw.view(E, N, K), sw.view(E, N, K // G)
    offs = torch.from_numpy(off).to(DEV)
    qa, sa = w8.quant_act(a)
    y_two = torch.full((R, N), float("nan"), dtype=torch.float32, device=DEV)
    w8.grouped_gemm(qa, sa, offs, qw, sw, out_dtype=torch.float32, out=y_two)
    y = torch.full((R, N), float("nan"), dtype=torch.float32, device=DEV)
    w8.grouped_linear(a, offs, qw, sw, out_dtype=torch.float32, out=y)
    torch.cuda.synchronize()
    covered = slice(int(off[0]), int(off[E]))
    assert torch.equal(y[covered], y_two[covered])
    qa_o, sa_o = oracle.quant_act(a_bits)
    qw_o, sw_o = oracle.quant_weight(w)
    y_ref, T = oracle.grouped_gemm(qa_o, sa_o, off, qw_o.reshape(E, N, K), sw_o.reshape(E, N, K // G))
    check_fp32(y.cpu().numpy()[covered], y_ref[covered], T[covered], K)
    assert w8.device_error(clear=True) == 0


def test_back_to_back_calls_share_workspace_and_graph_replay():
    """Consecutive calls on one stream reuse one workspace (split counters,
    partial slots, codes) while the previous GEMM may still be draining; a
    captured CUDA graph of the calls replays to the same bits."""
    rng = np.random.default_rng(2024)
    N, K = 28672, 1024
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    qw, sw = w8.quant_weight(torch.from_numpy(w).to(DEV))
    qw_o, sw_o = oracle.quant_weight(w)
    shapes = [1, 32, 8, 32, 3]                       # GEMV and split tensor-core calls mixed
    acts = [workloads.f32_to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
            for M in shapes]
    a_dev = [to_dev_bf16(b) for b in acts]
    ws = torch.empty(max(w8.linear_workspace_size(M, N, K) for M in shapes), dtype=torch.uint8,
                     device=DEV)
    outs = [torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV) for M in shapes]
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        for a, y in zip(a_dev, outs):
            w8.linear(a, qw, sw, out_dtype=torch.float32, out=y, workspace=ws, stream=st)
    st.synchronize()
    for a_bits, y, M in zip(acts, outs, shapes):
        qa_o, sa_o = oracle.quant_act(a_bits)
        y_ref, T = oracle.gemm(qa_o, sa_o, qw_o, sw_o)
        check_fp32(y.cpu().numpy(), y_ref, T, K)
    first = [y.clone() for y in outs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(st):
        with torch.cuda.graph(g, stream=st):
            for a, y in zip(a_dev, outs):
                w8.linear(a, qw, sw, out_dtype=torch.float32, out=y, workspace=ws, stream=st)
    for y in outs:
        y.fill_(float("nan"))
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for y, y0 in zip(outs, first):
        assert torch.equal(y, y0)
    assert w8.device_error(clear=True) == 0
