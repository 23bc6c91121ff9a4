"""CPU tests of the C ABI: the library loads, exports every function that
include/w8a8.h declares, and rejects bad arguments on the host before any
device work (no compute calls here: no GPU is needed or touched)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w8a8.h")

OK, INVALID, UNSUPPORTED, CUDA_ERR, WORKSPACE = 0, 1, 2, 3, 4


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__._build_module().build()
    L = ctypes.CDLL(path)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    L.w8a8_quant_act.argtypes = [vp, i64, i64, i64, vp, i64, vp, vp]
    L.w8a8_quant_weight.argtypes = [vp, i64, i64, vp, vp, vp]
    L.w8a8_gemm.argtypes = [vp, vp, vp, vp, vp, i32, i64, i64, i64, vp, vp, ctypes.c_size_t, vp]
    L.w8a8_grouped_gemm.argtypes = [vp, vp, vp, vp, vp, vp, i32, i64, i64, i64, i64, vp, vp,
                                    ctypes.c_size_t, vp]
    L.w8a8_gemm_workspace_size.argtypes = [i64, i64, i64]
    L.w8a8_gemm_workspace_size.restype = ctypes.c_size_t
    L.w8a8_grouped_gemm_workspace_size.argtypes = [i64, i64, i64, i64]
    L.w8a8_grouped_gemm_workspace_size.restype = ctypes.c_size_t
    L.w8a8_status_string.argtypes = [i32]
    L.w8a8_status_string.restype = ctypes.c_char_p
    L.w8a8_linear_workspace_size.argtypes = [i64, i64, i64]
    L.w8a8_linear_workspace_size.restype = ctypes.c_size_t
    L.w8a8_grouped_linear_workspace_size.argtypes = [i64, i64, i64, i64]
    L.w8a8_grouped_linear_workspace_size.restype = ctypes.c_size_t
    L.w8a8_linear.argtypes = [vp, i64, vp, vp, vp, i32, i64, i64, i64, vp, ctypes.c_size_t, vp]
    L.w8a8_grouped_linear.argtypes = [vp, i64, vp, vp, vp, vp, i32, i64, i64, i64, i64, vp,
                                      ctypes.c_size_t, vp]
    return L


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(w8a8_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_function(lib):
    names = declared_functions()
    assert {"w8a8_quant_act", "w8a8_gemm", "w8a8_grouped_gemm"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in w8a8.h but not exported"


def test_status_strings(lib):
    for code, name in [(0, b"W8A8_OK"), (1, b"W8A8_ERR_INVALID_ARG"), (4, b"W8A8_ERR_WORKSPACE"),
                       (99, b"W8A8_UNKNOWN_STATUS")]:
        assert lib.w8a8_status_string(code) == name


def _staging(rows, K):
    return (rows * K * 2 + 255) // 256 * 256


def _split_area(rows):
    # 320 int32 arrival counters + 160 CTAs x 2 FP32 partial slots of rows x 128
    return (1280 + 160 * 2 * rows * 128 * 4 + 255) // 256 * 256


def test_workspace_size(lib):
    # fp16 staging copy of the activation codes (rounded up to 256 bytes), then
    # the optional K-split area of dense calls of 5..64 token rows.
    assert lib.w8a8_gemm_workspace_size(0, 128, 128) == 0
    assert lib.w8a8_gemm_workspace_size(3, 128, 128) == 768
    assert lib.w8a8_gemm_workspace_size(1, 128, 128) == 256
    assert lib.w8a8_gemm_workspace_size(4, 128, 128) == _staging(4, 128)
    assert lib.w8a8_gemm_workspace_size(5, 128, 128) == _staging(5, 128) + _split_area(5)
    assert lib.w8a8_gemm_workspace_size(8, 28672, 8192) == 8 * 8192 * 2 + _split_area(8)
    assert lib.w8a8_gemm_workspace_size(9, 128, 128) == _staging(9, 128) + _split_area(9)
    assert lib.w8a8_gemm_workspace_size(64, 128, 256) == _staging(64, 256) + _split_area(64)
    assert lib.w8a8_gemm_workspace_size(65, 128, 256) == _staging(65, 256)
    assert lib.w8a8_gemm_workspace_size(129, 128, 384) == (129 * 384 * 2 + 255) // 256 * 256
    assert lib.w8a8_gemm_workspace_size(32, 28672, 8192) == 32 * 8192 * 2 + _split_area(32)
    assert lib.w8a8_grouped_gemm_workspace_size(4096, 64, 3072, 4096) == 4096 * 4096 * 2
    assert lib.w8a8_grouped_gemm_workspace_size(8, 64, 3072, 4096) == 8 * 4096 * 2
    assert lib.w8a8_grouped_gemm_workspace_size(0, 64, 3072, 4096) == 0


FAKE = 1 << 20      # a 16-byte aligned non-null value; never dereferenced here


def gemm(lib, qa=FAKE, sa=FAKE, qw=FAKE, sw=FAKE, y=FAKE, dt=0, M=16, N=128, K=128, dbg=None,
         ws=FAKE, wsb=1 << 30):
    return lib.w8a8_gemm(qa, sa, qw, sw, y, dt, M, N, K, dbg, ws, wsb, None)


def test_gemm_host_validation(lib):
    assert gemm(lib, K=100) == INVALID                 # K % 128 != 0
    assert gemm(lib, K=0) == INVALID
    assert gemm(lib, N=0) == INVALID
    assert gemm(lib, M=-1) == INVALID
    assert gemm(lib, qa=None) == INVALID
    assert gemm(lib, sw=None) == INVALID
    assert gemm(lib, qa=FAKE + 8) == INVALID           # TMA operand not 16-byte aligned
    assert gemm(lib, sa=FAKE + 2) == INVALID
    assert gemm(lib, dt=7) == INVALID
    assert gemm(lib, ws=None) == WORKSPACE
    assert gemm(lib, wsb=16 * 128 * 2 - 1) == WORKSPACE
    assert gemm(lib, ws=FAKE + 16) == WORKSPACE        # workspace must be 256-byte aligned
    assert gemm(lib, M=1 << 24, K=1 << 10) == INVALID  # operand above 2^31 elements
    assert gemm(lib, M=0) == OK                        # no-op, no device work


def test_grouped_host_validation(lib):
    def call(off=FAKE, E=4, R=64, N=128, K=256, wsb=1 << 30):
        return lib.w8a8_grouped_gemm(FAKE, FAKE, off, FAKE, FAKE, FAKE, 0, R, E, N, K, None,
                                     FAKE, wsb, None)
    assert call(off=None) == INVALID
    assert call(E=0) == INVALID
    assert call(E=1025) == INVALID
    assert call(K=129) == INVALID
    assert call(off=FAKE + 2) == INVALID
    assert call(wsb=10) == WORKSPACE
    assert call(R=0) == OK


def test_quant_host_validation(lib):
    assert lib.w8a8_quant_act(FAKE, 4, 0, 0, FAKE, 0, FAKE, None) == INVALID
    assert lib.w8a8_quant_act(FAKE, 4, 64, 32, FAKE, 64, FAKE, None) == INVALID   # lda < K
    assert lib.w8a8_quant_act(None, 4, 64, 64, FAKE, 64, FAKE, None) == INVALID
    assert lib.w8a8_quant_act(FAKE, 0, 64, 64, FAKE, 64, FAKE, None) == OK
    assert lib.w8a8_quant_weight(FAKE, 4, 100, FAKE, FAKE, None) == INVALID
    assert lib.w8a8_quant_weight(FAKE + 4, 4, 128, FAKE, FAKE, None) == INVALID
    assert lib.w8a8_quant_weight(FAKE, 0, 128, FAKE, FAKE, None) == OK


def test_no_device_gives_cuda_error(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("only meaningful without a GPU")
    # Valid arguments reach the device check, which fails without a GPU; the
    # fake pointers are never used.
    assert lib.w8a8_quant_act(FAKE, 4, 64, 64, FAKE, 64, FAKE, None) in (CUDA_ERR, UNSUPPORTED)


def test_selftest_wait_validation(lib):
    lib.w8a8_selftest_wait_timeout.argtypes = [ctypes.c_uint32, ctypes.c_void_p]
    lib.w8a8_selftest_wait_timeout.restype = ctypes.c_int
    # refused on the host: never launches
    assert lib.w8a8_selftest_wait_timeout(0, None) == INVALID
    assert lib.w8a8_selftest_wait_timeout(2000001, None) == INVALID


def test_linear_workspace_size(lib):
    # codes (M*K*2) and scales (M*4), each rounded up to 256 bytes, then the
    # optional K-split area for 5..64 dense rows
    def base(M, K):
        return _staging(M, K) + (M * 4 + 255) // 256 * 256
    assert lib.w8a8_linear_workspace_size(0, 128, 128) == 0
    assert lib.w8a8_linear_workspace_size(1, 28672, 8192) == base(1, 8192)
    assert lib.w8a8_linear_workspace_size(4, 128, 128) == base(4, 128)
    assert lib.w8a8_linear_workspace_size(32, 28672, 8192) == base(32, 8192) + _split_area(32)
    assert lib.w8a8_linear_workspace_size(65, 128, 256) == base(65, 256)
    assert lib.w8a8_grouped_linear_workspace_size(4096, 64, 3072, 4096) == base(4096, 4096)
    assert lib.w8a8_grouped_linear_workspace_size(8, 64, 3072, 4096) == base(8, 4096)


def test_linear_host_validation(lib):
    def call(a=FAKE, lda=256, qw=FAKE, sw=FAKE, y=FAKE, dt=0, M=16, N=128, K=256, ws=FAKE,
             wsb=1 << 30):
        return lib.w8a8_linear(a, lda, qw, sw, y, dt, M, N, K, ws, wsb, None)
    assert call(K=100, lda=100) == INVALID              # K % 128 != 0
    assert call(lda=128) == INVALID                     # lda < K
    assert call(a=None) == INVALID
    assert call(a=FAKE + 1) == INVALID                  # BF16 rows must be 2-byte aligned
    assert call(qw=FAKE + 8) == INVALID                 # TMA operand not 16-byte aligned
    assert call(dt=5) == INVALID
    assert call(N=0) == INVALID
    assert call(ws=None) == WORKSPACE
    assert call(ws=FAKE + 16) == WORKSPACE
    assert call(wsb=16 * 256 * 2) == WORKSPACE          # no room for the scales
    assert call(M=0) == OK

    def gcall(off=FAKE, E=4, R=64, wsb=1 << 30):
        return lib.w8a8_grouped_linear(FAKE, 256, off, FAKE, FAKE, FAKE, 0, R, E, 128, 256,
                                       FAKE, wsb, None)
    assert gcall(off=None) == INVALID
    assert gcall(E=1025) == INVALID
    assert gcall(wsb=100) == WORKSPACE
    assert gcall(R=0) == OK


def test_rmsnorm_host_validation(lib):
    vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    lib.w8a8_rmsnorm.argtypes = [vp, i64, vp, f32, i64, i64, vp, i64, vp]
    lib.w8a8_rmsnorm_quant.argtypes = [vp, i64, vp, f32, i32, i64, i64, vp, i64, vp, vp]
    lib.w8a8_rmsnorm_linear.argtypes = [vp, i64, vp, f32, vp, vp, vp, i32, i64, i64, i64, vp,
                                        ctypes.c_size_t, vp]

    def norm(x=FAKE, ldx=64, g=FAKE, eps=1e-5, M=4, K=64, y=FAKE, ldy=64):
        return lib.w8a8_rmsnorm(x, ldx, g, eps, M, K, y, ldy, None)
    assert norm(eps=0.0) == INVALID
    assert norm(eps=-1.0) == INVALID
    assert norm(eps=float("inf")) == INVALID
    assert norm(eps=float("nan")) == INVALID
    assert norm(K=12, ldx=16, ldy=16) == INVALID        # K % 8 != 0
    assert norm(K=32776, ldx=32776, ldy=32776) == INVALID   # K above 32768
    assert norm(ldx=68) == INVALID                      # row stride not a multiple of 8
    assert norm(ldx=56) == INVALID                      # ldx < K
    assert norm(x=FAKE + 8) == INVALID                  # x not 16-byte aligned
    assert norm(g=FAKE + 8) == INVALID
    assert norm(y=None) == INVALID
    assert norm(M=0, x=None, g=None, y=None) == OK
    assert lib.w8a8_rmsnorm_quant(FAKE, 64, FAKE, 1e-5, 7, 4, 64, FAKE, 64, FAKE, None) == INVALID
    assert lib.w8a8_rmsnorm_quant(FAKE, 64, FAKE, 1e-5, 0, 4, 64, FAKE + 4, 64, FAKE,
                                  None) == INVALID      # codes not 8-byte aligned
    # linear: K % 128 and the workspace as for w8a8_linear
    assert lib.w8a8_rmsnorm_linear(FAKE, 64, FAKE, 1e-5, FAKE, FAKE, FAKE, 0, 4, 128, 64, FAKE,
                                   1 << 30, None) == INVALID
    assert lib.w8a8_rmsnorm_linear(FAKE, 256, FAKE, 1e-5, FAKE, FAKE, FAKE, 0, 4, 128, 256, None,
                                   0, None) == WORKSPACE
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        assert norm() in (CUDA_ERR, UNSUPPORTED)
