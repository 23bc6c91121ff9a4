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
SCALE_AMAX, SCALE_POW2 = 0, 1     # w8a8_scale_mode
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
    lib.w8a8_probe_tc_rate.argtypes = [i32, i32, i32, i64, ctypes.POINTER(i64), vp]
    lib.w8a8_probe_dp4a_rate.argtypes = [i64, ctypes.POINTER(i64), vp]
    lib.w8a8_quant_act_ex.argtypes = [vp, i64, i64, i64, vp, i64, vp, i32, vp]
    lib.w8a8_quant_weight_ex.argtypes = [vp, i64, i64, i32, i32, vp, vp, vp]
    lib.w8a8_gemm_ex.argtypes = [vp, vp, vp, vp, i32, vp, i32, i64, i64, i64, vp, vp,
                                 ctypes.c_size_t, vp]
    lib.w8a8_grouped_gemm_ex.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i64, i64, i64, i64,
                                         vp, vp, ctypes.c_size_t, vp]
    lib.w8a8_linear_ex.argtypes = [vp, i64, i32, vp, vp, i32, vp, i32, i64, i64, i64, vp,
                                   ctypes.c_size_t, vp]
    lib.w8a8_w8a16_gemm.argtypes = [vp, i64, vp, vp, i32, vp, i32, i64, i64, i64, vp]
    lib.w8a8_w8a16_grouped_gemm.argtypes = [vp, i64, vp, vp, vp, i32, vp, i32, i64, i64, i64, i64,
                                            vp]
    lib.w8a8_kv_quant.argtypes = [vp, i64, i64, vp, vp, vp, vp]
    lib.w8a8_attention_decode_workspace_size.argtypes = [i64, i64, i64, i64]
    lib.w8a8_attention_decode_workspace_size.restype = ctypes.c_size_t
    lib.w8a8_attention_decode_int8kv.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64,
                                                 ctypes.c_float, vp, i32, vp, ctypes.c_size_t, vp]
    lib.w8a8_attention_decode_bf16kv.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64,
                                                 ctypes.c_float, vp, i32, vp, ctypes.c_size_t, vp]
    lib.w8a8_moe_route.argtypes = [vp, i64, i64, i64, vp, vp, vp, vp, vp]
    lib.w8a8_quant_act_rows.argtypes = [vp, i64, vp, i64, i64, vp, vp, vp]
    lib.w8a8_swiglu_quant.argtypes = [vp, i64, i64, vp, i64, vp, vp, vp]
    lib.w8a8_swiglu.argtypes = [vp, i64, i64, vp, vp]
    lib.w8a8_moe_unpermute.argtypes = [vp, vp, vp, i64, i64, i64, vp, i32, vp]
    lib.w8a8_moe_ffn_workspace_size.argtypes = [i64, i64, i64, i64, i64]
    lib.w8a8_moe_ffn_workspace_size.restype = ctypes.c_size_t
    lib.w8a8_moe_ffn.argtypes = [vp, i64, vp, vp, i64, i64, i64, i64, i64, vp, vp, vp, vp, vp,
                                 i32, vp, ctypes.c_size_t, vp]
    lib.w8a8_rmsnorm.argtypes = [vp, i64, vp, ctypes.c_float, i64, i64, vp, i64, vp]
    lib.w8a8_rmsnorm_quant.argtypes = [vp, i64, vp, ctypes.c_float, i32, i64, i64, vp, i64, vp, vp]
    lib.w8a8_rmsnorm_linear.argtypes = [vp, i64, vp, ctypes.c_float, vp, vp, vp, i32, i64, i64,
                                        i64, vp, ctypes.c_size_t, vp]
    lib.w8a8_version.restype = i32
    for name in ("w8a8_quant_act", "w8a8_quant_weight", "w8a8_gemm", "w8a8_grouped_gemm",
                 "w8a8_gemm_noalloc", "w8a8_device_error", "w8a8_selftest_wait_timeout",
                 "w8a8_linear", "w8a8_grouped_linear", "w8a8_probe_tc_rate",
                 "w8a8_probe_dp4a_rate", "w8a8_moe_route", "w8a8_quant_act_rows",
                 "w8a8_swiglu_quant", "w8a8_swiglu", "w8a8_moe_unpermute", "w8a8_moe_ffn",
                 "w8a8_quant_act_ex", "w8a8_quant_weight_ex", "w8a8_gemm_ex",
                 "w8a8_grouped_gemm_ex", "w8a8_linear_ex", "w8a8_w8a16_gemm",
                 "w8a8_w8a16_grouped_gemm", "w8a8_kv_quant", "w8a8_attention_decode_int8kv",
                 "w8a8_attention_decode_bf16kv", "w8a8_rmsnorm", "w8a8_rmsnorm_quant",
                 "w8a8_rmsnorm_linear"):
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


def _require(t: torch.Tensor, dtype: torch.dtype, name: str, ndim: int,
             shape: Optional[Tuple[int, ...]] = None,
             device: Optional[torch.device] = None) -> None:
    if not t.is_cuda or t.dtype != dtype or t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous CUDA {dtype} tensor of rank {ndim}, "
                         f"got {t.dtype} {tuple(t.shape)} on {t.device}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if device is not None and t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device}")


def _require_out(out: torch.Tensor, out_dtype: torch.dtype, shape: Tuple[int, int],
                 device: torch.device) -> None:
    """The kernels write exactly shape[0] * shape[1] elements of out_dtype
    into `out`: anything else would be written past its end or half-filled."""
    _require(out, out_dtype, "out", 2, shape, device)


def _require_workspace(ws: torch.Tensor, device: torch.device) -> None:
    if not ws.is_cuda or ws.dtype != torch.uint8 or not ws.is_contiguous() or ws.device != device:
        raise ValueError(f"workspace: expected a contiguous uint8 tensor on {device}")


def _on_device(device: torch.device, stream: Optional[torch.cuda.Stream]):
    """Makes the operands' device current for the call (the library resolves
    per-device state, such as its built-in scratch, on the current device);
    a stream of another device is refused."""
    if stream is not None and stream.device != device:
        raise ValueError(f"stream belongs to {stream.device}, the operands to {device}")
    return torch.cuda.device(device)


def quant_act(a: torch.Tensor, qa: Optional[torch.Tensor] = None,
              sa: Optional[torch.Tensor] = None,
              stream: Optional[torch.cuda.Stream] = None,
              scale_mode: int = SCALE_AMAX) -> Tuple[torch.Tensor, torch.Tensor]:
    """Per-token dynamic INT8 quantization of BF16 activations [M, K]
    (scale amax/127, or a power of two with scale_mode=SCALE_POW2)."""
    if not a.is_cuda or a.dtype != torch.bfloat16 or a.dim() != 2 or a.stride(1) != 1:
        raise ValueError("a: expected a CUDA bf16 [M, K] tensor with unit column stride")
    M, K = a.shape
    dev = a.device
    if qa is None:
        qa = torch.empty((M, K), dtype=torch.int8, device=dev)
    elif (not qa.is_cuda or qa.dtype != torch.int8 or qa.dim() != 2 or tuple(qa.shape) != (M, K)
          or qa.stride(1) != 1 or qa.device != dev):
        raise ValueError(f"qa: expected an int8 [{M}, {K}] tensor with unit column stride on {dev}")
    if sa is None:
        sa = torch.empty((M,), dtype=torch.float32, device=dev)
    else:
        _require(sa, torch.float32, "sa", 1, (M,), dev)
    with _on_device(dev, stream):
        if scale_mode == SCALE_AMAX:
            _check(_lib.w8a8_quant_act(_ptr(a), M, K, a.stride(0), _ptr(qa), qa.stride(0),
                                       _ptr(sa), _stream(stream)), "w8a8_quant_act")
        else:
            _check(_lib.w8a8_quant_act_ex(_ptr(a), M, K, a.stride(0), _ptr(qa), qa.stride(0),
                                          _ptr(sa), scale_mode, _stream(stream)),
                   "w8a8_quant_act_ex")
    return qa, sa


def quant_weight(w: torch.Tensor, stream: Optional[torch.cuda.Stream] = None,
                 block_rows: int = 1, scale_mode: int = SCALE_AMAX
                 ) -> Tuple[torch.Tensor, torch.Tensor]:
    """INT8 quantization of FP32 weights [N, K] over [block_rows x 128]
    blocks (1: per-row groups; 128: [128, 128] blocks); returns (qw [N, K],
    sw [ceil(N / block_rows), K / 128])."""
    _require(w, torch.float32, "w", 2)
    N, K = w.shape
    nb = (N + block_rows - 1) // block_rows
    qw = torch.empty((N, K), dtype=torch.int8, device=w.device)
    sw = torch.empty((nb, K // GROUP), dtype=torch.float32, device=w.device)
    with _on_device(w.device, stream):
        if block_rows == 1 and scale_mode == SCALE_AMAX:
            _check(_lib.w8a8_quant_weight(_ptr(w), N, K, _ptr(qw), _ptr(sw), _stream(stream)),
                   "w8a8_quant_weight")
        else:
            _check(_lib.w8a8_quant_weight_ex(_ptr(w), N, K, block_rows, scale_mode, _ptr(qw),
                                             _ptr(sw), _stream(stream)), "w8a8_quant_weight_ex")
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


def _dense_operands(qa, sa, qw, sw, sw_block_rows=1):
    """Checks the dense GEMM operands against each other; returns M, N, K."""
    if sw_block_rows not in (1, 128):
        raise ValueError("sw_block_rows must be 1 or 128")
    _require(qa, torch.int8, "qa", 2)
    dev = qa.device
    M, K = qa.shape
    _require(qw, torch.int8, "qw", 2, device=dev)
    N = qw.shape[0]
    if qw.shape[1] != K:
        raise ValueError(f"qw: expected K = {K} columns, got {qw.shape[1]}")
    _require(sa, torch.float32, "sa", 1, (M,), dev)
    nb = (N + sw_block_rows - 1) // sw_block_rows
    _require(sw, torch.float32, "sw", 2, (nb, K // GROUP), dev)
    return M, N, K


def gemm(qa: torch.Tensor, sa: torch.Tensor, qw: torch.Tensor, sw: torch.Tensor,
         out_dtype: torch.dtype = torch.bfloat16, out: Optional[torch.Tensor] = None,
         workspace: Optional[torch.Tensor] = None, debug_partials: bool = False,
         stream: Optional[torch.cuda.Stream] = None, sw_block_rows: int = 1):
    """Y[M,N] = sa[m] * sum_g sw[n / sw_block_rows, g] * P[m,n,g]; returns y,
    or (y, P) with debug_partials=True (P int32 [M, N, K/128])."""
    M, N, K = _dense_operands(qa, sa, qw, sw, sw_block_rows)
    code = _dtype_code(out_dtype)
    dev = qa.device
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=dev)
    else:
        _require_out(out, out_dtype, (M, N), dev)
    if workspace is None:
        workspace = torch.empty(max(gemm_workspace_size(M, N, K), 1), dtype=torch.uint8,
                                device=dev)
    else:
        _require_workspace(workspace, dev)
    P = torch.empty((M, N, K // GROUP), dtype=torch.int32, device=dev) if debug_partials else None
    with _on_device(dev, stream):
        if sw_block_rows == 1:
            _check(_lib.w8a8_gemm(_ptr(qa), _ptr(sa), _ptr(qw), _ptr(sw), _ptr(out), code, M, N,
                                  K, _ptr(P), _ptr(workspace), workspace.numel(),
                                  _stream(stream)), "w8a8_gemm")
        else:
            _check(_lib.w8a8_gemm_ex(_ptr(qa), _ptr(sa), _ptr(qw), _ptr(sw), sw_block_rows,
                                     _ptr(out), code, M, N, K, _ptr(P), _ptr(workspace),
                                     workspace.numel(), _stream(stream)), "w8a8_gemm_ex")
    return (out, P) if debug_partials else out


NOALLOC_SCRATCH_BYTES = 8 << 20


def gemm_noalloc(qa: torch.Tensor, sa: torch.Tensor, qw: torch.Tensor, sw: torch.Tensor,
                 out_dtype: torch.dtype = torch.bfloat16, out: Optional[torch.Tensor] = None,
                 stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """The GEMM for callers that cannot allocate device memory when the layer
    runs: the library stages the activation codes (and, when they fit, the
    K-split partial sums) in its own fixed 8 MiB scratch array instead of a
    workspace (M*K*2 bytes must fit). Writes into the caller's `out`. Calls
    that may overlap on the GPU share that array and must be ordered."""
    M, N, K = _dense_operands(qa, sa, qw, sw)
    code = _dtype_code(out_dtype)
    if out is None:
        raise ValueError("gemm_noalloc writes into a caller-provided `out` tensor")
    _require_out(out, out_dtype, (M, N), qa.device)
    with _on_device(qa.device, stream):
        _check(_lib.w8a8_gemm_noalloc(_ptr(qa), _ptr(sa), _ptr(qw), _ptr(sw), _ptr(out), code,
                                      M, N, K, _stream(stream)), "w8a8_gemm_noalloc")
    return out


def grouped_gemm(qa: torch.Tensor, sa: torch.Tensor, offsets: torch.Tensor, qw: torch.Tensor,
                 sw: torch.Tensor, out_dtype: torch.dtype = torch.bfloat16,
                 out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                 debug_partials: bool = False, stream: Optional[torch.cuda.Stream] = None,
                 sw_block_rows: int = 1):
    """MoE grouped GEMM over rows sorted by expert; offsets int32 [E+1] on
    device; sw [E, ceil(N / sw_block_rows), K/128]."""
    _require(qa, torch.int8, "qa", 2)
    dev = qa.device
    R, K = qa.shape
    _require(qw, torch.int8, "qw", 3, device=dev)
    E, N, K2 = qw.shape
    if K2 != K:
        raise ValueError(f"qw: expected K = {K} columns, got {K2}")
    _require(sa, torch.float32, "sa", 1, (R,), dev)
    if sw_block_rows not in (1, 128):
        raise ValueError("sw_block_rows must be 1 or 128")
    nb = (N + sw_block_rows - 1) // sw_block_rows
    _require(sw, torch.float32, "sw", 3, (E, nb, K // GROUP), dev)
    _require(offsets, torch.int32, "offsets", 1, (E + 1,), dev)
    code = _dtype_code(out_dtype)
    if out is None:
        out = torch.empty((R, N), dtype=out_dtype, device=dev)
    else:
        _require_out(out, out_dtype, (R, N), dev)
    if workspace is None:
        workspace = torch.empty(max(grouped_gemm_workspace_size(R, E, N, K), 1),
                                dtype=torch.uint8, device=dev)
    else:
        _require_workspace(workspace, dev)
    P = torch.empty((R, N, K // GROUP), dtype=torch.int32, device=dev) if debug_partials else None
    with _on_device(dev, stream):
        if sw_block_rows == 1:
            _check(_lib.w8a8_grouped_gemm(_ptr(qa), _ptr(sa), _ptr(offsets), _ptr(qw), _ptr(sw),
                                          _ptr(out), code, R, E, N, K, _ptr(P), _ptr(workspace),
                                          workspace.numel(), _stream(stream)),
                   "w8a8_grouped_gemm")
        else:
            _check(_lib.w8a8_grouped_gemm_ex(_ptr(qa), _ptr(sa), _ptr(offsets), _ptr(qw),
                                             _ptr(sw), sw_block_rows, _ptr(out), code, R, E, N,
                                             K, _ptr(P), _ptr(workspace), workspace.numel(),
                                             _stream(stream)), "w8a8_grouped_gemm_ex")
    return (out, P) if debug_partials else out


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
           stream: Optional[torch.cuda.Stream] = None, act_scale_mode: int = SCALE_AMAX,
           sw_block_rows: int = 1) -> torch.Tensor:
    """quant_act + gemm in one call: Y[M,N] from BF16 activations a [M, K]
    (the quantizer writes the GEMM's operand directly into the workspace)."""
    lda = _require_act(a)
    dev = a.device
    M, K = a.shape
    _require(qw, torch.int8, "qw", 2, device=dev)
    N = qw.shape[0]
    if qw.shape[1] != K:
        raise ValueError(f"qw: expected K = {K} columns, got {qw.shape[1]}")
    if sw_block_rows not in (1, 128):
        raise ValueError("sw_block_rows must be 1 or 128")
    _require(sw, torch.float32, "sw", 2, ((N + sw_block_rows - 1) // sw_block_rows, K // GROUP),
             dev)
    code = _dtype_code(out_dtype)
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=dev)
    else:
        _require_out(out, out_dtype, (M, N), dev)
    if workspace is None:
        workspace = torch.empty(max(linear_workspace_size(M, N, K), 1), dtype=torch.uint8,
                                device=dev)
    else:
        _require_workspace(workspace, dev)
    with _on_device(dev, stream):
        if act_scale_mode == SCALE_AMAX and sw_block_rows == 1:
            _check(_lib.w8a8_linear(_ptr(a), lda, _ptr(qw), _ptr(sw), _ptr(out), code, M, N, K,
                                    _ptr(workspace), workspace.numel(), _stream(stream)),
                   "w8a8_linear")
        else:
            _check(_lib.w8a8_linear_ex(_ptr(a), lda, act_scale_mode, _ptr(qw), _ptr(sw),
                                       sw_block_rows, _ptr(out), code, M, N, K, _ptr(workspace),
                                       workspace.numel(), _stream(stream)), "w8a8_linear_ex")
    return out


def _require_norm_input(x: torch.Tensor, gamma: torch.Tensor) -> int:
    ldx = _require_act(x)
    K = x.shape[1]
    _require(gamma, torch.bfloat16, "gamma", 1, (K,), x.device)
    return ldx


def rmsnorm(x: torch.Tensor, gamma: torch.Tensor, eps: float, out: Optional[torch.Tensor] = None,
            stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """RMSNorm of BF16 rows x [M, K] with BF16 weights gamma [K]:
    bf16((x / sqrt(mean(x^2) + eps)) * gamma), fp32 arithmetic."""
    ldx = _require_norm_input(x, gamma)
    M, K = x.shape
    dev = x.device
    if out is None:
        out = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    elif (not out.is_cuda or out.dtype != torch.bfloat16 or out.dim() != 2
          or tuple(out.shape) != (M, K) or out.stride(1) != 1 or out.device != dev):
        raise ValueError(f"out: expected a bf16 [{M}, {K}] tensor with unit column stride on {dev}")
    with _on_device(dev, stream):
        _check(_lib.w8a8_rmsnorm(_ptr(x), ldx, _ptr(gamma), eps, M, K, _ptr(out), out.stride(0),
                                 _stream(stream)), "w8a8_rmsnorm")
    return out


def rmsnorm_quant(x: torch.Tensor, gamma: torch.Tensor, eps: float,
                  qa: Optional[torch.Tensor] = None, sa: Optional[torch.Tensor] = None,
                  stream: Optional[torch.cuda.Stream] = None,
                  scale_mode: int = SCALE_AMAX) -> Tuple[torch.Tensor, torch.Tensor]:
    """RMSNorm and per-token INT8 quantization in one kernel: the codes and
    scales quant_act gives for rmsnorm(x, gamma, eps)."""
    ldx = _require_norm_input(x, gamma)
    M, K = x.shape
    dev = x.device
    if qa is None:
        qa = torch.empty((M, K), dtype=torch.int8, device=dev)
    elif (not qa.is_cuda or qa.dtype != torch.int8 or qa.dim() != 2 or tuple(qa.shape) != (M, K)
          or qa.stride(1) != 1 or qa.device != dev):
        raise ValueError(f"qa: expected an int8 [{M}, {K}] tensor with unit column stride on {dev}")
    if sa is None:
        sa = torch.empty((M,), dtype=torch.float32, device=dev)
    else:
        _require(sa, torch.float32, "sa", 1, (M,), dev)
    with _on_device(dev, stream):
        _check(_lib.w8a8_rmsnorm_quant(_ptr(x), ldx, _ptr(gamma), eps, scale_mode, M, K, _ptr(qa),
                                       qa.stride(0), _ptr(sa), _stream(stream)),
               "w8a8_rmsnorm_quant")
    return qa, sa


def rmsnorm_linear(x: torch.Tensor, gamma: torch.Tensor, eps: float, qw: torch.Tensor,
                   sw: torch.Tensor, out_dtype: torch.dtype = torch.bfloat16,
                   out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                   stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """linear(rmsnorm(x, gamma, eps), qw, sw) with the normalisation inside
    the quantizer kernel (the normalised rows never reach HBM)."""
    ldx = _require_norm_input(x, gamma)
    dev = x.device
    M, K = x.shape
    _require(qw, torch.int8, "qw", 2, device=dev)
    N = qw.shape[0]
    if qw.shape[1] != K:
        raise ValueError(f"qw: expected K = {K} columns, got {qw.shape[1]}")
    _require(sw, torch.float32, "sw", 2, (N, K // GROUP), dev)
    code = _dtype_code(out_dtype)
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=dev)
    else:
        _require_out(out, out_dtype, (M, N), dev)
    if workspace is None:
        workspace = torch.empty(max(linear_workspace_size(M, N, K), 1), dtype=torch.uint8,
                                device=dev)
    else:
        _require_workspace(workspace, dev)
    with _on_device(dev, stream):
        _check(_lib.w8a8_rmsnorm_linear(_ptr(x), ldx, _ptr(gamma), eps, _ptr(qw), _ptr(sw),
                                        _ptr(out), code, M, N, K, _ptr(workspace),
                                        workspace.numel(), _stream(stream)),
               "w8a8_rmsnorm_linear")
    return out


def grouped_linear(a: torch.Tensor, offsets: torch.Tensor, qw: torch.Tensor, sw: torch.Tensor,
                   out_dtype: torch.dtype = torch.bfloat16, out: Optional[torch.Tensor] = None,
                   workspace: Optional[torch.Tensor] = None,
                   stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """quant_act + grouped_gemm in one call over rows sorted by expert."""
    lda = _require_act(a)
    dev = a.device
    R, K = a.shape
    _require(qw, torch.int8, "qw", 3, device=dev)
    E, N, K2 = qw.shape
    if K2 != K:
        raise ValueError(f"qw: expected K = {K} columns, got {K2}")
    _require(sw, torch.float32, "sw", 3, (E, N, K // GROUP), dev)
    _require(offsets, torch.int32, "offsets", 1, (E + 1,), dev)
    code = _dtype_code(out_dtype)
    if out is None:
        out = torch.empty((R, N), dtype=out_dtype, device=dev)
    else:
        _require_out(out, out_dtype, (R, N), dev)
    if workspace is None:
        workspace = torch.empty(max(grouped_linear_workspace_size(R, E, N, K), 1),
                                dtype=torch.uint8, device=dev)
    else:
        _require_workspace(workspace, dev)
    with _on_device(dev, stream):
        _check(_lib.w8a8_grouped_linear(_ptr(a), lda, _ptr(offsets), _ptr(qw), _ptr(sw),
                                        _ptr(out), code, R, E, N, K, _ptr(workspace),
                                        workspace.numel(), _stream(stream)),
               "w8a8_grouped_linear")
    return out


# ------------------------------------------------- weight-only INT8 (W8A16)
def w8a16_gemm(a: torch.Tensor, qw: torch.Tensor, sw: torch.Tensor,
               out_dtype: torch.dtype = torch.bfloat16, out: Optional[torch.Tensor] = None,
               sw_block_rows: int = 1,
               stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Y = a (BF16, not quantized) x dequantized INT8 weights, the group
    scales applied per group in the epilogue."""
    lda = _require_act(a)
    dev = a.device
    M, K = a.shape
    _require(qw, torch.int8, "qw", 2, device=dev)
    N = qw.shape[0]
    if qw.shape[1] != K:
        raise ValueError(f"qw: expected K = {K} columns, got {qw.shape[1]}")
    _require(sw, torch.float32, "sw", 2, ((N + sw_block_rows - 1) // sw_block_rows, K // GROUP),
             dev)
    code = _dtype_code(out_dtype)
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=dev)
    else:
        _require_out(out, out_dtype, (M, N), dev)
    with _on_device(dev, stream):
        _check(_lib.w8a8_w8a16_gemm(_ptr(a), lda, _ptr(qw), _ptr(sw), sw_block_rows, _ptr(out),
                                    code, M, N, K, _stream(stream)), "w8a8_w8a16_gemm")
    return out


def w8a16_grouped_gemm(a: torch.Tensor, offsets: torch.Tensor, qw: torch.Tensor,
                       sw: torch.Tensor, out_dtype: torch.dtype = torch.bfloat16,
                       out: Optional[torch.Tensor] = None, sw_block_rows: int = 1,
                       stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """The grouped (MoE expert) weight-only GEMM over rows sorted by expert."""
    lda = _require_act(a)
    dev = a.device
    R, K = a.shape
    _require(qw, torch.int8, "qw", 3, device=dev)
    E, N, K2 = qw.shape
    if K2 != K:
        raise ValueError(f"qw: expected K = {K} columns, got {K2}")
    _require(sw, torch.float32, "sw", 3,
             (E, (N + sw_block_rows - 1) // sw_block_rows, K // GROUP), dev)
    _require(offsets, torch.int32, "offsets", 1, (E + 1,), dev)
    code = _dtype_code(out_dtype)
    if out is None:
        out = torch.empty((R, N), dtype=out_dtype, device=dev)
    else:
        _require_out(out, out_dtype, (R, N), dev)
    with _on_device(dev, stream):
        _check(_lib.w8a8_w8a16_grouped_gemm(_ptr(a), lda, _ptr(offsets), _ptr(qw), _ptr(sw),
                                            sw_block_rows, _ptr(out), code, R, E, N, K,
                                            _stream(stream)), "w8a8_w8a16_grouped_gemm")
    return out


# ------------------------------------------------- INT8 KV cache + attention
HEAD_DIM = 128


def kv_quant(x: torch.Tensor, cache: torch.Tensor, scales: torch.Tensor,
             dst_rows: Optional[torch.Tensor] = None,
             stream: Optional[torch.cuda.Stream] = None) -> None:
    """Quantizes K or V vectors x [n, 128] (BF16) into rows dst_rows (or 0..n-1)
    of cache (int8, last dim 128) with one scale per row in scales."""
    _require(x, torch.bfloat16, "x", 2)
    dev = x.device
    n, D = x.shape
    if not cache.is_cuda or cache.dtype != torch.int8 or not cache.is_contiguous() \
            or cache.shape[-1] != D or cache.device != dev:
        raise ValueError("cache: expected a contiguous int8 CUDA tensor with last dim 128")
    rows = cache.numel() // D
    if not scales.is_cuda or scales.dtype != torch.float32 or not scales.is_contiguous() \
            or scales.numel() != rows or scales.device != dev:
        raise ValueError("scales: expected one float32 per cache row")
    if dst_rows is not None:
        _require(dst_rows, torch.int32, "dst_rows", 1, (n,), dev)
    elif n > rows:
        raise ValueError("more vectors than cache rows")
    with _on_device(dev, stream):
        _check(_lib.w8a8_kv_quant(_ptr(x), n, D, _ptr(dst_rows), _ptr(cache), _ptr(scales),
                                  _stream(stream)), "w8a8_kv_quant")


def attention_decode_workspace_size(B: int, Hq: int, S_max: int) -> int:
    return int(_lib.w8a8_attention_decode_workspace_size(B, Hq, S_max, HEAD_DIM))


def attention_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                     lens: torch.Tensor, softmax_scale: float,
                     k_scale: Optional[torch.Tensor] = None, v_scale: Optional[torch.Tensor] = None,
                     out_dtype: torch.dtype = torch.bfloat16, out: Optional[torch.Tensor] = None,
                     workspace: Optional[torch.Tensor] = None,
                     stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Decode attention of q [B, Hq, 128] over a KV cache [B, Hkv, S_max, 128]:
    INT8 codes with per-vector scales k_scale / v_scale [B, Hkv, S_max], or a
    BF16 cache (no scales); lens [B] int32 on the device."""
    _require(q, torch.bfloat16, "q", 3)
    dev = q.device
    B, Hq, D = q.shape
    int8 = k_cache.dtype == torch.int8
    dt = torch.int8 if int8 else torch.bfloat16
    _require(k_cache, dt, "k_cache", 4, device=dev)
    _, Hkv, S_max, D2 = k_cache.shape
    if D2 != D or k_cache.shape[0] != B:
        raise ValueError("k_cache must be [B, Hkv, S_max, 128]")
    _require(v_cache, dt, "v_cache", 4, tuple(k_cache.shape), dev)
    if int8:
        _require(k_scale, torch.float32, "k_scale", 3, (B, Hkv, S_max), dev)
        _require(v_scale, torch.float32, "v_scale", 3, (B, Hkv, S_max), dev)
    _require(lens, torch.int32, "lens", 1, (B,), dev)
    code = _dtype_code(out_dtype)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=out_dtype, device=dev)
    elif (not out.is_cuda or out.dtype != out_dtype or tuple(out.shape) != (B, Hq, D)
          or not out.is_contiguous() or out.device != dev):
        raise ValueError(f"out: expected a contiguous {out_dtype} tensor of shape {(B, Hq, D)}")
    if workspace is None:
        workspace = torch.empty(max(attention_decode_workspace_size(B, Hq, S_max), 1),
                                dtype=torch.uint8, device=dev)
    else:
        _require_workspace(workspace, dev)
    with _on_device(dev, stream):
        if int8:
            _check(_lib.w8a8_attention_decode_int8kv(
                _ptr(q), _ptr(k_cache), _ptr(k_scale), _ptr(v_cache), _ptr(v_scale), _ptr(lens),
                B, Hq, Hkv, S_max, D, float(softmax_scale), _ptr(out), code, _ptr(workspace),
                workspace.numel(), _stream(stream)), "w8a8_attention_decode_int8kv")
        else:
            _check(_lib.w8a8_attention_decode_bf16kv(
                _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(lens), B, Hq, Hkv, S_max, D,
                float(softmax_scale), _ptr(out), code, _ptr(workspace), workspace.numel(),
                _stream(stream)), "w8a8_attention_decode_bf16kv")
    return out


# ------------------------------------------------------------ MoE expert FFN
def moe_route(topk_ids: torch.Tensor, E: int, stream: Optional[torch.cuda.Stream] = None):
    """Routing of topk_ids [T, k] (int32): returns (offsets [E+1], row_of
    [T*k], token_of_row [T*k], pair_of_row [T*k]), all int32 on the device."""
    _require(topk_ids, torch.int32, "topk_ids", 2)
    dev = topk_ids.device
    T, k = topk_ids.shape
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    row_of = torch.empty(T * k, dtype=torch.int32, device=dev)
    tok = torch.empty(T * k, dtype=torch.int32, device=dev)
    pair = torch.empty(T * k, dtype=torch.int32, device=dev)
    with _on_device(dev, stream):
        _check(_lib.w8a8_moe_route(_ptr(topk_ids), T, k, E, _ptr(offsets), _ptr(row_of),
                                   _ptr(tok), _ptr(pair), _stream(stream)), "w8a8_moe_route")
    return offsets, row_of, tok, pair


def quant_act_rows(a: torch.Tensor, src_rows: torch.Tensor, qa: Optional[torch.Tensor] = None,
                   sa: Optional[torch.Tensor] = None,
                   stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Per-token quantization of the gathered rows a[src_rows[r]] (rows with a
    negative entry are left untouched in qa / sa)."""
    lda = _require_act(a)
    dev = a.device
    _require(src_rows, torch.int32, "src_rows", 1, device=dev)
    rows, K = src_rows.shape[0], a.shape[1]
    if qa is None:
        qa = torch.zeros((rows, K), dtype=torch.int8, device=dev)
    else:
        _require(qa, torch.int8, "qa", 2, (rows, K), dev)
    if sa is None:
        sa = torch.zeros((rows,), dtype=torch.float32, device=dev)
    else:
        _require(sa, torch.float32, "sa", 1, (rows,), dev)
    with _on_device(dev, stream):
        _check(_lib.w8a8_quant_act_rows(_ptr(a), lda, _ptr(src_rows), rows, K, _ptr(qa), _ptr(sa),
                                        _stream(stream)), "w8a8_quant_act_rows")
    return qa, sa


def swiglu_quant(U: torch.Tensor, offsets: Optional[torch.Tensor] = None,
                 stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """h = silu(U[:, :I]) * U[:, I:] then per-row quantization: (qh int8
    [R, I], sh float32 [R]); with offsets [E+1], rows >= offsets[E] are
    skipped (left zero)."""
    _require(U, torch.float32, "U", 2)
    dev = U.device
    R, I2 = U.shape
    if I2 % 2:
        raise ValueError("U must have an even number of columns (gate | up)")
    I = I2 // 2
    E = 0
    if offsets is not None:
        _require(offsets, torch.int32, "offsets", 1, device=dev)
        E = offsets.shape[0] - 1
    qh = torch.zeros((R, I), dtype=torch.int8, device=dev)
    sh = torch.zeros((R,), dtype=torch.float32, device=dev)
    with _on_device(dev, stream):
        _check(_lib.w8a8_swiglu_quant(_ptr(U), R, I, _ptr(offsets), E, _ptr(qh), _ptr(sh),
                                      _stream(stream)), "w8a8_swiglu_quant")
    return qh, sh


def swiglu(U: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """h = silu(U[:, :I]) * U[:, I:] (FP32, the arithmetic of swiglu_quant)."""
    _require(U, torch.float32, "U", 2)
    R, I2 = U.shape
    h = torch.empty((R, I2 // 2), dtype=torch.float32, device=U.device)
    with _on_device(U.device, stream):
        _check(_lib.w8a8_swiglu(_ptr(U), R, I2 // 2, _ptr(h), _stream(stream)), "w8a8_swiglu")
    return h


def moe_unpermute(D: torch.Tensor, row_of: torch.Tensor, topk_w: torch.Tensor,
                  out_dtype: torch.dtype = torch.bfloat16, out: Optional[torch.Tensor] = None,
                  stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """y[t] = sum_j topk_w[t, j] * D[row_of[t*k + j]] over routed entries."""
    _require(D, torch.float32, "D", 2)
    dev = D.device
    _require(topk_w, torch.float32, "topk_w", 2, device=dev)
    T, k = topk_w.shape
    _require(row_of, torch.int32, "row_of", 1, (T * k,), dev)
    H = D.shape[1]
    code = _dtype_code(out_dtype)
    if out is None:
        out = torch.empty((T, H), dtype=out_dtype, device=dev)
    else:
        _require_out(out, out_dtype, (T, H), dev)
    with _on_device(dev, stream):
        _check(_lib.w8a8_moe_unpermute(_ptr(D), _ptr(row_of), _ptr(topk_w), T, k, H, _ptr(out),
                                       code, _stream(stream)), "w8a8_moe_unpermute")
    return out


def moe_ffn_workspace_size(T: int, k: int, H: int, I: int, E: int) -> int:
    return int(_lib.w8a8_moe_ffn_workspace_size(T, k, H, I, E))


def moe_ffn(x: torch.Tensor, topk_ids: torch.Tensor, topk_w: torch.Tensor,
            qw_up: torch.Tensor, sw_up: torch.Tensor, qw_down: torch.Tensor,
            sw_down: torch.Tensor, out_dtype: torch.dtype = torch.bfloat16,
            out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
            stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """The MoE expert FFN: y [T, H] from tokens x [T, H] (BF16), the router's
    topk_ids / topk_w [T, k], qw_up [E, 2I, H] (gate rows first) and
    qw_down [E, H, I] with their group scales."""
    ldx = _require_act(x)
    dev = x.device
    T, H = x.shape
    _require(topk_ids, torch.int32, "topk_ids", 2, device=dev)
    k = topk_ids.shape[1]
    _require(topk_w, torch.float32, "topk_w", 2, (T, k), dev)
    if topk_ids.shape[0] != T:
        raise ValueError("topk_ids must have one row per token")
    _require(qw_up, torch.int8, "qw_up", 3, device=dev)
    E, I2, H2 = qw_up.shape
    if H2 != H or I2 % 2:
        raise ValueError("qw_up must be [E, 2I, H]")
    I = I2 // 2
    _require(sw_up, torch.float32, "sw_up", 3, (E, I2, H // GROUP), dev)
    _require(qw_down, torch.int8, "qw_down", 3, (E, H, I), dev)
    _require(sw_down, torch.float32, "sw_down", 3, (E, H, I // GROUP), dev)
    code = _dtype_code(out_dtype)
    if out is None:
        out = torch.empty((T, H), dtype=out_dtype, device=dev)
    else:
        _require_out(out, out_dtype, (T, H), dev)
    if workspace is None:
        workspace = torch.empty(max(moe_ffn_workspace_size(T, k, H, I, E), 1), dtype=torch.uint8,
                                device=dev)
    else:
        _require_workspace(workspace, dev)
    with _on_device(dev, stream):
        _check(_lib.w8a8_moe_ffn(_ptr(x), ldx, _ptr(topk_ids), _ptr(topk_w), T, k, H, I, E,
                                 _ptr(qw_up), _ptr(sw_up), _ptr(qw_down), _ptr(sw_down),
                                 _ptr(out), code, _ptr(workspace), workspace.numel(),
                                 _stream(stream)), "w8a8_moe_ffn")
    return out


def selftest_wait_timeout(limit_us: int = 20000,
                          stream: Optional[torch.cuda.Stream] = None) -> None:
    """Drives the device-side bounded-wait failure path: a wait that can never
    complete gives up after limit_us and records its code (read it with
    device_error())."""
    _check(_lib.w8a8_selftest_wait_timeout(limit_us, _stream(stream)),
           "w8a8_selftest_wait_timeout")


def probe_tc_rate(n: int, chains: int, steps: int, distinct: bool = False,
                  stream: Optional[torch.cuda.Stream] = None) -> int:
    """Launches the tcgen05 kind::f16 rate probe (M=128, N=n, K=16 per
    instruction, `chains` accumulators taking turns, on shared or distinct
    operands); returns the int8 multiply-adds it performs (time the launch
    to get the rate)."""
    macs = ctypes.c_int64(0)
    _check(_lib.w8a8_probe_tc_rate(n, chains, 1 if distinct else 0, steps, ctypes.byref(macs),
                                   _stream(stream)),
           "w8a8_probe_tc_rate")
    return int(macs.value)


def probe_dp4a_rate(iters: int, stream: Optional[torch.cuda.Stream] = None) -> int:
    """Launches the dp4a rate probe; returns the int8 multiply-adds it performs."""
    macs = ctypes.c_int64(0)
    _check(_lib.w8a8_probe_dp4a_rate(iters, ctypes.byref(macs), _stream(stream)),
           "w8a8_probe_dp4a_rate")
    return int(macs.value)


def device_error(clear: bool = True) -> int:
    """The library's device error word (0 = none); synchronises the device."""
    v = ctypes.c_uint64(0)
    st = _lib.w8a8_device_error(ctypes.byref(v), 1 if clear else 0)
    if st not in (0, 5):
        raise W8A8Error(st, "w8a8_device_error")
    return int(v.value)
