"""Python binding of libw8a8 (GB300 / sm_103a W8A8 group-scaled GEMM).

Argument marshalling only: every computation runs in the CUDA kernels of
``libw8a8.so`` behind the C ABI declared in ``include/w8a8.h``. PyTorch
provides device memory and streams. There is no CPU path: importing this
package fails if the shared library has not been built.

Functions (names match the C entry points):
  quant_act(a_bf16)                       -> (qa int8 [M,K], sa f32 [M])
  quant_weight(w_f32)                     -> (qw int8 [N,K], sw f32 [N,K/128])
  gemm(qa, sa, qw, sw, out_dtype, ...)    -> y [M,N]  (+ partials when debug)
  grouped_gemm(qa, sa, offsets, qw, sw, out_dtype, ...) -> y [R,N]
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

from . import _build

GROUP = 128
W8A8_BF16, W8A8_FP32 = 0, 1
_STATUS = {0: "W8A8_OK", 1: "W8A8_ERR_INVALID_ARG", 2: "W8A8_ERR_UNSUPPORTED",
           3: "W8A8_ERR_CUDA", 4: "W8A8_ERR_WORKSPACE", 5: "W8A8_ERR_DEVICE_TIMEOUT"}


class W8A8Error(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {_STATUS.get(status, status)}")
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(_build.LIB):
        raise ImportError(
            f"{_build.LIB} is missing: build it with `python -c \"import __graft_entry__ as g; "
            f"g.build()\"` (the W8A8 path has no CPU fallback)")
    lib = ctypes.CDLL(_build.LIB)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.w8a8_quant_act.argtypes = [vp, i64, i64, i64, vp, i64, vp, vp]
    lib.w8a8_quant_weight.argtypes = [vp, i64, i64, vp, vp, vp]
    lib.w8a8_gemm_workspace_size.argtypes = [i64, i64, i64]
    lib.w8a8_gemm_workspace_size.restype = ctypes.c_size_t
    lib.w8a8_grouped_gemm_workspace_size.argtypes = [i64, i64, i64, i64]
    lib.w8a8_grouped_gemm_workspace_size.restype = ctypes.c_size_t
    lib.w8a8_gemm.argtypes = [vp, vp, vp, vp, vp, i32, i64, i64, i64, vp, vp, ctypes.c_size_t, vp]
    lib.w8a8_grouped_gemm.argtypes = [vp, vp, vp, vp, vp, vp, i32, i64, i64, i64, i64, vp, vp,
                                      ctypes.c_size_t, vp]
    lib.w8a8_gemm_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, i64, i64, i64, vp]
    lib.w8a8_status_string.argtypes = [i32]
    lib.w8a8_status_string.restype = ctypes.c_char_p
    lib.w8a8_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint64), i32]
    lib.w8a8_selftest_wait_timeout.argtypes = [ctypes.c_uint32, vp]
    lib.w8a8_linear_workspace_size.argtypes = [i64, i64, i64]
    lib.w8a8_linear_workspace_size.restype = ctypes.c_size_t
    lib.w8a8_grouped_linear_workspace_size.argtypes = [i64, i64, i64, i64]
    lib.w8a8_grouped_linear_workspace_size.restype = ctypes.c_size_t
    lib.w8a8_linear.argtypes = [vp, i64, vp, vp, vp, i32, i64, i64, i64, vp, ctypes.c_size_t, vp]
    lib.w8a8_grouped_linear.argtypes = [vp, i64, vp, vp, vp, vp, i32, i64, i64, i64, i64, vp,
                                        ctypes.c_size_t, vp]
    lib.w8a8_version.restype = i32
    for name in ("w8a8_quant_act", "w8a8_quant_weight", "w8a8_gemm", "w8a8_grouped_gemm",
                 "w8a8_gemm_noalloc", "w8a8_device_error", "w8a8_selftest_wait_timeout",
                 "w8a8_linear", "w8a8_grouped_linear"):
        getattr(lib, name).restype = i32
    return lib


_lib = _load()


def lib() -> ctypes.CDLL:
    """The loaded C library (for callers that pass raw pointers)."""
    return _lib


def library_path() -> str:
    return _build.LIB


def _check(status: int, what: str) -> None:
    if status != 0:
        raise W8A8Error(status, what)


def _stream(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _require(t: torch.Tensor, dtype: torch.dtype, name: str, ndim: int) -> None:
    if not t.is_cuda or t.dtype != dtype or t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous CUDA {dtype} tensor of rank {ndim}, "
                         f"got {t.dtype} {tuple(t.shape)} on {t.device}")


def quant_act(a: torch.Tensor, qa: Optional[torch.Tensor] = None,
              sa: Optional[torch.Tensor] = None,
              stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Per-token dynamic INT8 quantization of BF16 activations [M, K]."""
    if not a.is_cuda or a.dtype != torch.bfloat16 or a.dim() != 2 or a.stride(1) != 1:
        raise ValueError("a: expected a CUDA bf16 [M, K] tensor with unit column stride")
    M, K = a.shape
    qa = torch.empty((M, K), dtype=torch.int8, device=a.device) if qa is None else qa
    sa = torch.empty((M,), dtype=torch.float32, device=a.device) if sa is None else sa
    _check(_lib.w8a8_quant_act(_ptr(a), M, K, a.stride(0), _ptr(qa), qa.stride(0), _ptr(sa),
                               _stream(stream)), "w8a8_quant_act")
    return qa, sa


def quant_weight(w: torch.Tensor, stream: Optional[torch.cuda.Stream] = None
                 ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Per-row, per-128-K-group INT8 quantization of FP32 weights [N, K]."""
    _require(w, torch.float32, "w", 2)
    N, K = w.shape
    qw = torch.empty((N, K), dtype=torch.int8, device=w.device)
    sw = torch.empty((N, K // GROUP), dtype=torch.float32, device=w.device)
    _check(_lib.w8a8_quant_weight(_ptr(w), N, K, _ptr(qw), _ptr(sw), _stream(stream)),
           "w8a8_quant_weight")
    return qw, sw


def gemm_workspace_size(M: int, N: int, K: int) -> int:
    return int(_lib.w8a8_gemm_workspace_size(M, N, K))


def grouped_gemm_workspace_size(R: int, E: int, N: int, K: int) -> int:
    return int(_lib.w8a8_grouped_gemm_workspace_size(R, E, N, K))


def _dtype_code(out_dtype: torch.dtype) -> int:
    if out_dtype == torch.bfloat16:
        return W8A8_BF16
    if out_dtype == torch.float32:
        return W8A8_FP32
    raise ValueError("out_dtype must be torch.bfloat16 or torch.float32")


def gemm(qa: torch.Tensor, sa: torch.Tensor, qw: torch.Tensor, sw: torch.Tensor,
         out_dtype: torch.dtype = torch.bfloat16, out: Optional[torch.Tensor] = None,
         workspace: Optional[torch.Tensor] = None, debug_partials: bool = False,
         stream: Optional[torch.cuda.Stream] = None):
    """Y[M,N] = sa[m] * sum_g sw[n,g] * P[m,n,g]; returns y, or (y, P) with
    debug_partials=True (P int32 [M, N, K/128])."""
    _require(qa, torch.int8, "qa", 2)
    _require(qw, torch.int8, "qw", 2)
    _require(sa, torch.float32, "sa", 1)
    _require(sw, torch.float32, "sw", 2)
    M, K = qa.shape
    N = qw.shape[0]
    dev = qa.device
    y = torch.empty((M, N), dtype=out_dtype, device=dev) if out is None else out
    if workspace is None:
        workspace = torch.empty(max(gemm_workspace_size(M, N, K), 1), dtype=torch.uint8,
                                device=dev)
    P = torch.empty((M, N, K // GROUP), dtype=torch.int32, device=dev) if debug_partials else None
    _check(_lib.w8a8_gemm(_ptr(qa), _ptr(sa), _ptr(qw), _ptr(sw), _ptr(y), _dtype_code(out_dtype),
                          M, N, K, _ptr(P), _ptr(workspace), workspace.numel(), _stream(stream)),
           "w8a8_gemm")
    return (y, P) if debug_partials else y


NOALLOC_SCRATCH_BYTES = 8 << 20


def gemm_noalloc(qa: torch.Tensor, sa: torch.Tensor, qw: torch.Tensor, sw: torch.Tensor,
                 out_dtype: torch.dtype = torch.bfloat16, out: Optional[torch.Tensor] = None,
                 stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Same result as gemm(), for callers that cannot allocate device memory
    when the layer runs: the library stages the activation codes in its own
    fixed 8 MiB scratch array instead of a workspace (M*K*2 bytes must fit).
    Calls that may overlap on the GPU share that array and must be ordered."""
    _require(qa, torch.int8, "qa", 2)
    _require(qw, torch.int8, "qw", 2)
    _require(sa, torch.float32, "sa", 1)
    _require(sw, torch.float32, "sw", 2)
    M, K = qa.shape
    N = qw.shape[0]
    if out is None:
        raise ValueError("gemm_noalloc writes into a caller-provided `out` tensor")
    _check(_lib.w8a8_gemm_noalloc(_ptr(qa), _ptr(sa), _ptr(qw), _ptr(sw), _ptr(out),
                                  _dtype_code(out_dtype), M, N, K, _stream(stream)),
           "w8a8_gemm_noalloc")
    return out


def grouped_gemm(qa: torch.Tensor, sa: torch.Tensor, offsets: torch.Tensor, qw: torch.Tensor,
                 sw: torch.Tensor, out_dtype: torch.dtype = torch.bfloat16,
                 out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                 debug_partials: bool = False, stream: Optional[torch.cuda.Stream] = None):
    """MoE grouped GEMM over rows sorted by expert; offsets int32 [E+1] on device."""
    _require(qa, torch.int8, "qa", 2)
    _require(qw, torch.int8, "qw", 3)
    _require(sa, torch.float32, "sa", 1)
    _require(sw, torch.float32, "sw", 3)
    _require(offsets, torch.int32, "offsets", 1)
    R, K = qa.shape
    E, N, _ = qw.shape
    dev = qa.device
    if out is None:
        y = torch.empty((R, N), dtype=out_dtype, device=dev)
    else:
        y = out
    if workspace is None:
        workspace = torch.empty(max(grouped_gemm_workspace_size(R, E, N, K), 1),
                                dtype=torch.uint8, device=dev)
    P = torch.empty((R, N, K // GROUP), dtype=torch.int32, device=dev) if debug_partials else None
    _check(_lib.w8a8_grouped_gemm(_ptr(qa), _ptr(sa), _ptr(offsets), _ptr(qw), _ptr(sw), _ptr(y),
                                  _dtype_code(out_dtype), R, E, N, K, _ptr(P), _ptr(workspace),
                                  workspace.numel(), _stream(stream)), "w8a8_grouped_gemm")
    return (y, P) if debug_partials else y


def linear_workspace_size(M: int, N: int, K: int) -> int:
    return int(_lib.w8a8_linear_workspace_size(M, N, K))


def grouped_linear_workspace_size(R: int, E: int, N: int, K: int) -> int:
    return int(_lib.w8a8_grouped_linear_workspace_size(R, E, N, K))


def _require_act(a: torch.Tensor) -> int:
    if a.dtype != torch.bfloat16 or a.dim() != 2 or not a.is_cuda or a.stride(1) != 1:
        raise ValueError("a must be a CUDA bfloat16 [M, K] tensor with unit column stride")
    return a.stride(0)


def linear(a: torch.Tensor, qw: torch.Tensor, sw: torch.Tensor,
           out_dtype: torch.dtype = torch.bfloat16, out: Optional[torch.Tensor] = None,
           workspace: Optional[torch.Tensor] = None,
           stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """quant_act + gemm in one call: Y[M,N] from BF16 activations a [M, K]
    (the quantizer writes the GEMM's operand directly into the workspace)."""
    lda = _require_act(a)
    _require(qw, torch.int8, "qw", 2)
    _require(sw, torch.float32, "sw", 2)
    M, K = a.shape
    N = qw.shape[0]
    y = torch.empty((M, N), dtype=out_dtype, device=a.device) if out is None else out
    if workspace is None:
        workspace = torch.empty(max(linear_workspace_size(M, N, K), 1), dtype=torch.uint8,
                                device=a.device)
    _check(_lib.w8a8_linear(_ptr(a), lda, _ptr(qw), _ptr(sw), _ptr(y), _dtype_code(out_dtype),
                            M, N, K, _ptr(workspace), workspace.numel(), _stream(stream)),
           "w8a8_linear")
    return y


def grouped_linear(a: torch.Tensor, offsets: torch.Tensor, qw: torch.Tensor, sw: torch.Tensor,
                   out_dtype: torch.dtype = torch.bfloat16, out: Optional[torch.Tensor] = None,
                   workspace: Optional[torch.Tensor] = None,
                   stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """quant_act + grouped_gemm in one call over rows sorted by expert."""
    lda = _require_act(a)
    _require(qw, torch.int8, "qw", 3)
    _require(sw, torch.float32, "sw", 3)
    _require(offsets, torch.int32, "offsets", 1)
    R, K = a.shape
    E, N, _ = qw.shape
    y = torch.empty((R, N), dtype=out_dtype, device=a.device) if out is None else out
    if workspace is None:
        workspace = torch.empty(max(grouped_linear_workspace_size(R, E, N, K), 1),
                                dtype=torch.uint8, device=a.device)
    _check(_lib.w8a8_grouped_linear(_ptr(a), lda, _ptr(offsets), _ptr(qw), _ptr(sw), _ptr(y),
                                    _dtype_code(out_dtype), R, E, N, K, _ptr(workspace),
                                    workspace.numel(), _stream(stream)), "w8a8_grouped_linear")
    return y


def selftest_wait_timeout(limit_us: int = 20000,
                          stream: Optional[torch.cuda.Stream] = None) -> None:
    """Drives the device-side bounded-wait failure path: a wait that can never
    complete gives up after limit_us and records its code (read it with
    device_error())."""
    _check(_lib.w8a8_selftest_wait_timeout(limit_us, _stream(stream)),
           "w8a8_selftest_wait_timeout")


def device_error(clear: bool = True) -> int:
    """The library's device error word (0 = none); synchronises the device."""
    v = ctypes.c_uint64(0)
    st = _lib.w8a8_device_error(ctypes.byref(v), 1 if clear else 0)
    if st not in (0, 5):
        raise W8A8Error(st, "w8a8_device_error")
    return int(v.value)
