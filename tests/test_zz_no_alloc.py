"""w8a8_gemm_noalloc: the GEMM for callers that cannot allocate device memory
when the layer runs (an engine that only hands a plug-in a stream and
pre-planned buffers, a pool that forbids allocation on its hot path). Every
call reuses the library's one built-in scratch array, so each case runs two
different problems back to back: the second must not depend on what the first
left in the scratch.

Each output is checked element by element against the CPU oracle with the
tolerance the other parity tests use (FP32 within the bound of w8a8_gemm,
capped at 1e-5 * sum|terms|; BF16 within one ulp of the correctly rounded
exact value, or the cancellation clause), and against w8a8_gemm with a caller
workspace: bit-identical where both run the same split plan (M <= 4, and
5..64 rows whose split area fits the scratch), within the bound otherwise.

This file is collected last on purpose; it passes alone in a fresh process
and after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import moe_gemm_gb300 as w8  # noqa: E402

DEV = torch.device("cuda:0")
G = 128
W8A8_WORKSPACE = 4


def _inputs(seed, M, N, K):
    rng = np.random.default_rng(seed)
    qa = rng.integers(-127, 128, (M, K), dtype=np.int8)
    qw = rng.integers(-127, 128, (N, K), dtype=np.int8)
    sa = (rng.random(M) * 0.1 + 1e-3).astype(np.float32)
    sw = (rng.random((N, K // G)) * 1e-3 + 1e-5).astype(np.float32)
    return qa, sa, qw, sw


def _run(qa, sa, qw, sw, out_dtype):
    """No-alloc entry point and workspace entry point on the same device
    inputs; outputs start poisoned with NaN."""
    t = [torch.from_numpy(x).to(DEV) for x in (qa, sa, qw, sw)]
    M, N = qa.shape[0], qw.shape[0]
    y_na = torch.full((M, N), float("nan"), dtype=out_dtype, device=DEV)
    y_ws = torch.full((M, N), float("nan"), dtype=out_dtype, device=DEV)
    w8.gemm_noalloc(*t, out_dtype=out_dtype, out=y_na)
    w8.gemm(*t, out_dtype=out_dtype, out=y_ws)
    torch.cuda.synchronize()
    return y_na, y_ws


def _fp32_tol(K, T):
    Gn = K // G
    return min(1e-5, (Gn + (Gn + 1) // 2 + 1) * 2.0 ** -24) * T


def _check_vs_oracle(y, y_ref, T, K, out_dtype):
    if out_dtype == torch.float32:
        err = np.abs(y.cpu().numpy().astype(np.float64) - y_ref)
        assert np.all(err <= _fp32_tol(K, T)), f"max err/T {np.max(err / T)}"
        return
    bits = y.view(torch.int16).cpu().numpy().view(np.uint16)
    ref_bits = oracle.bf16_round(y_ref)
    ulp = oracle.bf16_ulp(ref_bits)
    yv = oracle.bf16_to_float(bits)
    within_ulp = np.abs(yv - oracle.bf16_to_float(ref_bits)) <= ulp
    within_bound = np.abs(yv - y_ref) <= 1e-5 * T + 0.5 * ulp
    assert np.all(within_ulp | within_bound)


def _split_fits(M, K):
    r = lambda v: (v + 255) // 256 * 256  # noqa: E731
    return r(M * K * 2) + r(1280 + 163840 * M) <= w8.NOALLOC_SCRATCH_BYTES


# (M, N, K): the CUDA-core GEMV (M = 1), a K-split call whose split area fits
# the scratch (M = 32, K = 8192) and one whose split area does not (M = 64,
# K = 8192: runs unsplit); each followed by a second, different problem.
CASES = [
    ((1, 4096, 8192, torch.bfloat16), (3, 1000, 384, torch.float32)),
    ((32, 4096, 8192, torch.bfloat16), (7, 1000, 384, torch.float32)),
    ((64, 4096, 8192, torch.float32), (40, 1280, 1024, torch.bfloat16)),
]


@pytest.mark.parametrize("first,second", CASES, ids=["gemv", "split", "unsplit"])
def test_noalloc_matches_oracle_on_two_calls_in_a_row(first, second):
    for seed, (M, N, K, dt) in enumerate((first, second), start=11):
        qa, sa, qw, sw = _inputs(seed + M, M, N, K)
        y_na, y_ws = _run(qa, sa, qw, sw, dt)
        assert not torch.isnan(y_na.float()).any().item(), "no-alloc call left outputs unwritten"
        y_ref, T = oracle.gemm(qa, sa, qw, sw)
        _check_vs_oracle(y_na, y_ref, T, K, dt)
        if M <= 4 or M > 64 or _split_fits(M, K):
            assert torch.equal(y_na, y_ws), "same kernels and split plan, different bits"
        else:
            _check_vs_oracle(y_ws, y_ref, T, K, dt)
    assert w8.device_error(clear=True) == 0


def test_noalloc_rejects_problems_larger_than_its_scratch():
    lib = w8.lib()
    K = 8192
    M = w8.NOALLOC_SCRATCH_BYTES // (2 * K) + 1        # one row too many
    fake = ctypes.c_void_p(1 << 20)                    # never dereferenced: refused on the host
    st = lib.w8a8_gemm_noalloc(fake, fake, fake, fake, fake, 0, M, 128, K, None)
    assert st == W8A8_WORKSPACE
    assert lib.w8a8_gemm_noalloc(fake, fake, fake, fake, fake, 0, M - 1, 128, 100, None) == 1
