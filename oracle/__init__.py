"""CPU oracle for the W8A8 group-scaled GEMM (numpy front end over plain C).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``; never by the product path. It shares
no code with the CUDA library (``moe_gemm_gb300``) and neither imports the
other. The arithmetic lives in ``w8a8_oracle.c``; this module only builds the
shared object with gcc and marshals numpy arrays.

Functions follow "Deploying Hunyuan 770B in INT8 on domestic accelerators"
§3.1 (per-group-128 weights, per-token dynamic activations, round(x/scale),
INT8 x INT8 into INT32, FP32 scales applied at the end) and §1.3/§4.4 (MoE
tokens processed by their routed experts).

Pins: every function is checked by ``tests/test_oracle_pins.py`` against
exact rational arithmetic, closed forms, brute force and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Tuple

import numpy as np

GROUP = 128
_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w8a8_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_w8a8.so")
_lock = threading.Lock()
_lib = None

_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-shared", "-fPIC"]


def build(force: bool = False) -> str:
    """Compile the oracle shared object with gcc (no-op when up to date)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        p = ctypes.c_void_p
        i64 = ctypes.c_int64
        lib.oracle_quant_act.argtypes = [p, i64, i64, i64, p, i64, p]
        lib.oracle_quant_weight.argtypes = [p, i64, i64, p, p]
        lib.oracle_group_partials.argtypes = [p, p, i64, i64, i64, p]
        lib.oracle_gemm.argtypes = [p, p, p, p, i64, i64, i64, p, p]
        lib.oracle_grouped_gemm.argtypes = [p, p, p, p, p, i64, i64, i64, i64, p, p]
        lib.oracle_bf16_round.argtypes = [p, i64, p]
        lib.oracle_bf16_from_double.argtypes = [ctypes.c_double]
        lib.oracle_bf16_from_double.restype = ctypes.c_uint16
        lib.oracle_set_threads.argtypes = [ctypes.c_int]
        lib.oracle_max_threads.restype = ctypes.c_int
        lib.oracle_group_size.restype = ctypes.c_int
        assert lib.oracle_group_size() == GROUP
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def quant_act(a_bf16: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Per-token quantization of BF16 activations (uint16 bit patterns [M,K]).
    Returns (qa int8 [M,K], sa float32 [M])."""
    a = np.ascontiguousarray(a_bf16, dtype=np.uint16)
    M, K = a.shape
    qa = np.empty((M, K), dtype=np.int8)
    sa = np.empty(M, dtype=np.float32)
    _load().oracle_quant_act(_ptr(a), M, K, K, _ptr(qa), K, _ptr(sa))
    return qa, sa


def quant_weight(w: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Per-row, per-128-K-group quantization of FP32 weights [N,K].
    Returns (qw int8 [N,K], sw float32 [N,K/128])."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    if K % GROUP:
        raise ValueError("K must be a multiple of 128")
    qw = np.empty((N, K), dtype=np.int8)
    sw = np.empty((N, K // GROUP), dtype=np.float32)
    _load().oracle_quant_weight(_ptr(w), N, K, _ptr(qw), _ptr(sw))
    return qw, sw


def group_partials(qa: np.ndarray, qw: np.ndarray) -> np.ndarray:
    """Exact INT32 partials P[m,n,g] of each 128-wide K group."""
    qa = np.ascontiguousarray(qa, dtype=np.int8)
    qw = np.ascontiguousarray(qw, dtype=np.int8)
    M, K = qa.shape
    N = qw.shape[0]
    assert qw.shape[1] == K and K % GROUP == 0
    P = np.empty((M, N, K // GROUP), dtype=np.int32)
    _load().oracle_group_partials(_ptr(qa), _ptr(qw), M, N, K, _ptr(P))
    return P


def gemm(qa: np.ndarray, sa: np.ndarray, qw: np.ndarray, sw: np.ndarray,
         want_T: bool = True) -> Tuple[np.ndarray, Optional[np.ndarray]]:
    """y* = sum_g sa*sw*P in FP64 [M,N], and T = sum_g |sa*sw*P| [M,N]."""
    qa = np.ascontiguousarray(qa, dtype=np.int8)
    qw = np.ascontiguousarray(qw, dtype=np.int8)
    sa = np.ascontiguousarray(sa, dtype=np.float32)
    sw = np.ascontiguousarray(sw, dtype=np.float32)
    M, K = qa.shape
    N = qw.shape[0]
    assert qw.shape[1] == K and sw.shape == (N, K // GROUP) and sa.shape == (M,)
    y = np.empty((M, N), dtype=np.float64)
    T = np.empty((M, N), dtype=np.float64) if want_T else None
    _load().oracle_gemm(_ptr(qa), _ptr(sa), _ptr(qw), _ptr(sw), M, N, K, _ptr(y),
                        _ptr(T) if want_T else None)
    return y, T


def grouped_gemm(qa: np.ndarray, sa: np.ndarray, offsets: np.ndarray, qw: np.ndarray,
                 sw: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Expert-grouped GEMM. qa [R,K] rows sorted by expert, offsets [E+1],
    qw [E,N,K], sw [E,N,K/128]. Rows outside every segment are NaN."""
    qa = np.ascontiguousarray(qa, dtype=np.int8)
    qw = np.ascontiguousarray(qw, dtype=np.int8)
    sa = np.ascontiguousarray(sa, dtype=np.float32)
    sw = np.ascontiguousarray(sw, dtype=np.float32)
    off = np.ascontiguousarray(offsets, dtype=np.int32)
    R, K = qa.shape
    E, N, K2 = qw.shape
    assert K2 == K and off.shape == (E + 1,) and sw.shape == (E, N, K // GROUP)
    y = np.full((R, N), np.nan, dtype=np.float64)
    T = np.full((R, N), np.nan, dtype=np.float64)
    _load().oracle_grouped_gemm(_ptr(qa), _ptr(sa), _ptr(off), _ptr(qw), _ptr(sw), R, E, N,
                                K, _ptr(y), _ptr(T))
    return y, T


def bf16_round(v: np.ndarray) -> np.ndarray:
    """Correctly rounded FP64 -> BF16 bit patterns (ties to even)."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().oracle_bf16_round(_ptr(v), v.size, _ptr(out))
    return out


def bf16_to_float(h: np.ndarray) -> np.ndarray:
    """BF16 bit patterns -> float64 values (exact)."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
        np.float32).astype(np.float64)


def bf16_ulp(h: np.ndarray) -> np.ndarray:
    """Spacing of BF16 numbers at each (finite) BF16 value h: 2^(e-7) for a
    normal number with unbiased exponent e, 2^-133 for subnormals and zero."""
    u = np.asarray(h, dtype=np.uint16).astype(np.int64)
    bexp = (u >> 7) & 0xFF
    e = np.where(bexp == 0, -126, bexp - 127)
    return np.ldexp(1.0, (e - 7).astype(np.int64))
