"""w8a8_gemm_noalloc: the GEMM for callers that cannot allocate device memory
when the layer runs (an engine that only hands a plug-in a stream and
pre-planned buffers, a pool that forbids allocation on its hot path). It must
give the same output as w8a8_gemm with a caller workspace, call after call,
although every call reuses the library's one built-in scratch array.

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


def _both(qa, sa, qw, sw, out_dtype):
    """Run the no-alloc entry point and the workspace entry point on the same
    device inputs; outputs start poisoned with NaN."""
    t = [torch.from_numpy(x).to(DEV) for x in (qa, sa, qw, sw)]
    M, N = qa.shape[0], qw.shape[0]
    y_na = torch.full((M, N), float("nan"), dtype=out_dtype, device=DEV)
    y_ws = torch.full((M, N), float("nan"), dtype=out_dtype, device=DEV)
    w8.gemm_noalloc(*t, out_dtype=out_dtype, out=y_na)
    w8.gemm(*t, out_dtype=out_dtype, out=y_ws)
    torch.cuda.synchronize()
    return y_na.float().cpu().numpy().astype(np.float64), y_ws.float().cpu().numpy().astype(
        np.float64)


def test_noalloc_matches_workspace_gemm_on_two_calls_in_a_row():
    # Two different problems back to back: the second call must not depend on
    # what the first left in the shared scratch.
    cases = [(11, 32, 4096, 8192, torch.bfloat16), (12, 7, 1000, 384, torch.float32)]
    for seed, M, N, K, dt in cases:
        qa, sa, qw, sw = _inputs(seed, M, N, K)
        y_na, y_ws = _both(qa, sa, qw, sw, dt)
        assert not np.isnan(y_na).any(), "no-alloc call left outputs unwritten"
        _, T = oracle.gemm(qa, sa, qw, sw)
        Gn = K // G
        tol = min(1e-5, (Gn + (Gn + 1) // 2 + 1) * 2.0 ** -24) * T
        if dt == torch.bfloat16:
            tol = tol + 2.0 ** -8 * np.abs(y_ws)      # one BF16 ulp
        assert np.all(np.abs(y_na - y_ws) <= tol)
    assert w8.device_error(clear=True) == 0


def test_noalloc_rejects_problems_larger_than_its_scratch():
    lib = w8.lib()
    K = 8192
    M = w8.NOALLOC_SCRATCH_BYTES // (2 * K) + 1        # one row too many
    fake = ctypes.c_void_p(1 << 20)                    # never dereferenced: refused on the host
    st = lib.w8a8_gemm_noalloc(fake, fake, fake, fake, fake, 0, M, 128, K, None)
    assert st == W8A8_WORKSPACE
    assert lib.w8a8_gemm_noalloc(fake, fake, fake, fake, fake, 0, M - 1, 128, 100, None) == 1
