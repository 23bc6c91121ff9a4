"""Device-side failure path without a GPU fault: a bounded wait that can
never complete (a barrier armed for bytes no copy delivers) gives up, writes
its code into the library's error word, and the context stays usable.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import moe_gemm_gb300 as w8  # noqa: E402

DEV = torch.device("cuda:0")


def test_bounded_wait_records_code_and_context_survives():
    assert w8.device_error(clear=True) == 0
    w8.selftest_wait_timeout(20000)          # 20 ms limit
    code = w8.device_error(clear=False)      # synchronises
    assert code != 0
    assert code >> 56 == 2                   # kernel: the diagnostic
    assert (code >> 48) & 0xFF == 5          # role
    assert (code >> 32) & 0xFFFF == 1        # wait site
    assert code & 0xFFFFFFFF == 0            # CTA
    assert w8.device_error(clear=True) == code
    assert w8.device_error(clear=True) == 0
    # the context still runs the GEMM correctly
    rng = np.random.default_rng(3)
    M, N, K = 8, 256, 512
    qa = rng.integers(-127, 128, (M, K), dtype=np.int8)
    qw = rng.integers(-127, 128, (N, K), dtype=np.int8)
    sa = np.ones(M, np.float32)
    sw = np.ones((N, K // 128), np.float32)
    y = w8.gemm(*(torch.from_numpy(x).to(DEV) for x in (qa, sa, qw, sw)), out_dtype=torch.float32)
    torch.cuda.synchronize()
    exact = qa.astype(np.int64) @ qw.astype(np.int64).T
    np.testing.assert_array_equal(y.cpu().numpy().astype(np.int64), exact)
    assert w8.device_error(clear=True) == 0
