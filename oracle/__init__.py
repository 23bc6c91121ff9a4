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

MoE expert FFN (same page §4.4: count tokens per destination expert first,
then transfer them; §4.1: SwiGLU between the two expert GEMMs; §3.1: every
INT8 GEMM input quantized per token): ``moe_route``, ``swiglu_quant``,
``moe_unpermute`` and their composition ``moe_ffn``.

Pins: every function is checked by ``tests/test_oracle_pins.py`` and
``tests/test_oracle_moe_pins.py`` against exact rational arithmetic, closed
forms, brute force and invariants.
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
        lib.oracle_moe_route.argtypes = [p, i64, i64, i64, p, p, p, p]
        lib.oracle_exp_f32_n.argtypes = [p, i64, p]
        lib.oracle_silu_f32_n.argtypes = [p, i64, p]
        lib.oracle_swiglu_quant.argtypes = [p, i64, i64, p, p]
        lib.oracle_moe_unpermute.argtypes = [p, p, p, i64, i64, i64, p]
        lib.oracle_quant_act_pow2.argtypes = [p, i64, i64, i64, p, i64, p]
        lib.oracle_quant_weight_blocks.argtypes = [p, i64, i64, i64, ctypes.c_int, p, p]
        lib.oracle_gemm_blocks.argtypes = [p, p, p, p, i64, i64, i64, i64, p, p]
        lib.oracle_w8a16_gemm.argtypes = [p, p, p, i64, i64, i64, i64, p, p]
        lib.oracle_rmsnorm.argtypes = [p, i64, i64, i64, p, ctypes.c_double, p]
        lib.oracle_kv_dequant.argtypes = [p, p, i64, i64, p]
        lib.oracle_attention_decode.argtypes = [p, p, p, p, i64, i64, i64, i64, i64,
                                                ctypes.c_double, p, p]
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


# ------------------------------------------------------------ MoE expert FFN
def moe_route(ids: np.ndarray, E: int):
    """Routing histogram, offsets and permutation of the top-k expert ids
    ([T, k] int32). Returns (offsets [E+1], row_of [T*k], token_of_row [T*k],
    pair_of_row [T*k]) as int32; entries with ids outside [0, E) are not
    routed (row_of = -1); rows >= offsets[E] have token/pair -1."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, k = ids.shape
    n = T * k
    offsets = np.empty(E + 1, dtype=np.int32)
    row_of = np.empty(n, dtype=np.int32)
    tok = np.empty(n, dtype=np.int32)
    pair = np.empty(n, dtype=np.int32)
    _load().oracle_moe_route(_ptr(ids), T, k, E, _ptr(offsets), _ptr(row_of), _ptr(tok),
                             _ptr(pair))
    return offsets, row_of, tok, pair


def exp_f32(x: np.ndarray) -> np.ndarray:
    """The SwiGLU's binary32 exponential, element-wise."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty_like(x)
    _load().oracle_exp_f32_n(_ptr(x), x.size, _ptr(out))
    return out


def silu_f32(x: np.ndarray) -> np.ndarray:
    """silu(x) = x / (1 + e^-x) in binary32, element-wise."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty_like(x)
    _load().oracle_silu_f32_n(_ptr(x), x.size, _ptr(out))
    return out


def swiglu_quant(U: np.ndarray, nrows: Optional[int] = None):
    """h = silu(U[:, :I]) * U[:, I:] (binary32), then per-row quantization:
    returns (qh int8 [R, I], sh float32 [R]); rows >= nrows are zero."""
    U = np.ascontiguousarray(U, dtype=np.float32)
    R, I2 = U.shape
    assert I2 % 2 == 0
    I = I2 // 2
    nrows = R if nrows is None else int(nrows)
    qh = np.zeros((R, I), dtype=np.int8)
    sh = np.zeros(R, dtype=np.float32)
    _load().oracle_swiglu_quant(_ptr(U), nrows, I, _ptr(qh), _ptr(sh))
    return qh, sh


def moe_unpermute(D: np.ndarray, row_of: np.ndarray, w: np.ndarray) -> np.ndarray:
    """Y[t] = sum_j w[t, j] * D[row_of[t, j]] (FP64); w and row_of [T, k]."""
    D = np.ascontiguousarray(D, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float32)
    T, k = w.shape
    row_of = np.ascontiguousarray(row_of, dtype=np.int32).reshape(T * k)
    H = D.shape[1]
    Y = np.empty((T, H), dtype=np.float64)
    _load().oracle_moe_unpermute(_ptr(D), _ptr(row_of), _ptr(w), T, k, H, _ptr(Y))
    return Y


def moe_ffn(x_bits: np.ndarray, ids: np.ndarray, w: np.ndarray, qw_up: np.ndarray,
            sw_up: np.ndarray, qw_down: np.ndarray, sw_down: np.ndarray) -> dict:
    """The MoE expert FFN, step by step: route -> per-token quantization of
    the permuted token rows -> gate_up grouped GEMM (FP32 output: the FP64
    result rounded to binary32) -> SwiGLU + per-token requantization -> down
    grouped GEMM (FP64) -> weighted un-permute (FP64). x_bits [T, H] BF16 bit
    patterns; ids, w [T, k]; qw_up [E, 2I, H], qw_down [E, H, I]. Returns every
    intermediate and y [T, H] (FP64)."""
    E = qw_up.shape[0]
    T, k = ids.shape
    offsets, row_of, tok, pair = moe_route(ids, E)
    R = int(offsets[E])
    n = T * k
    H = x_bits.shape[1]
    xr = np.zeros((n, H), dtype=np.uint16)
    xr[:R] = x_bits[tok[:R]]
    qa, sa = quant_act(xr)
    qa[R:] = 0
    sa[R:] = 0
    U64, T_up = grouped_gemm(qa, sa, offsets, qw_up, sw_up)
    U = np.zeros(U64.shape, dtype=np.float32)
    U[:R] = U64[:R].astype(np.float32)
    qh, sh = swiglu_quant(U, R)
    D64, T_down = grouped_gemm(qh, sh, offsets, qw_down, sw_down)
    D = np.where(np.isnan(D64), 0.0, D64)
    Tdn = np.where(np.isnan(T_down), 0.0, T_down)
    y = moe_unpermute(D, row_of.reshape(T, k), w)
    # sum_j |w| * T_down[row]: the magnitude the output's error is measured against
    Ty = moe_unpermute(Tdn, row_of.reshape(T, k), np.abs(w).astype(np.float32))
    return {"offsets": offsets, "row_of": row_of, "token_of_row": tok, "pair_of_row": pair,
            "R": R, "qa": qa, "sa": sa, "U": U, "T_up": T_up, "qh": qh, "sh": sh, "D": D,
            "T_down": Tdn, "y": y, "T_y": Ty}


# ------------------------------------------- scale formats and W8A16 (NEXT)
def quant_act_pow2(a_bf16: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Per-token quantization with power-of-two (UE8M0) scales."""
    a = np.ascontiguousarray(a_bf16, dtype=np.uint16)
    M, K = a.shape
    qa = np.empty((M, K), dtype=np.int8)
    sa = np.empty(M, dtype=np.float32)
    _load().oracle_quant_act_pow2(_ptr(a), M, K, K, _ptr(qa), K, _ptr(sa))
    return qa, sa


def quant_weight_blocks(w: np.ndarray, block_rows: int = 1,
                        pow2: bool = False) -> Tuple[np.ndarray, np.ndarray]:
    """Weight quantization over [block_rows x 128] blocks (1: per-row
    groups, 128: [128, 128] blocks), amax/127 or power-of-two scales.
    Returns (qw int8 [N, K], sw float32 [ceil(N/block_rows), K/128])."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    if K % GROUP:
        raise ValueError("K must be a multiple of 128")
    nb = (N + block_rows - 1) // block_rows
    qw = np.empty((N, K), dtype=np.int8)
    sw = np.empty((nb, K // GROUP), dtype=np.float32)
    _load().oracle_quant_weight_blocks(_ptr(w), N, K, block_rows, 1 if pow2 else 0, _ptr(qw),
                                       _ptr(sw))
    return qw, sw


def gemm_blocks(qa: np.ndarray, sa: np.ndarray, qw: np.ndarray, sw: np.ndarray,
                block_rows: int) -> Tuple[np.ndarray, np.ndarray]:
    """The group-scaled GEMM with one weight scale per [block_rows x 128]
    block: y* (FP64) and T."""
    qa = np.ascontiguousarray(qa, dtype=np.int8)
    qw = np.ascontiguousarray(qw, dtype=np.int8)
    sa = np.ascontiguousarray(sa, dtype=np.float32)
    sw = np.ascontiguousarray(sw, dtype=np.float32)
    M, K = qa.shape
    N = qw.shape[0]
    assert sw.shape == ((N + block_rows - 1) // block_rows, K // GROUP)
    y = np.empty((M, N), dtype=np.float64)
    T = np.empty((M, N), dtype=np.float64)
    _load().oracle_gemm_blocks(_ptr(qa), _ptr(sa), _ptr(qw), _ptr(sw), M, N, K, block_rows,
                               _ptr(y), _ptr(T))
    return y, T


def w8a16_gemm(a_bf16: np.ndarray, qw: np.ndarray, sw: np.ndarray,
               block_rows: int = 1) -> Tuple[np.ndarray, np.ndarray]:
    """Weight-only INT8 GEMM with BF16 activations: y* (FP64) and T."""
    a = np.ascontiguousarray(a_bf16, dtype=np.uint16)
    qw = np.ascontiguousarray(qw, dtype=np.int8)
    sw = np.ascontiguousarray(sw, dtype=np.float32)
    M, K = a.shape
    N = qw.shape[0]
    assert qw.shape[1] == K and sw.shape == ((N + block_rows - 1) // block_rows, K // GROUP)
    y = np.empty((M, N), dtype=np.float64)
    T = np.empty((M, N), dtype=np.float64)
    _load().oracle_w8a16_gemm(_ptr(a), _ptr(qw), _ptr(sw), M, N, K, block_rows, _ptr(y), _ptr(T))
    return y, T


# ------------------------------------------------- INT8 KV cache + attention
def kv_quant(x_bf16: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Per-vector quantization of K or V vectors [..., D] (BF16 bit patterns):
    one scale per vector, exactly the per-token activation quantizer."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    D = x.shape[-1]
    q, s = quant_act(x.reshape(-1, D))
    return q.reshape(x.shape), s.reshape(x.shape[:-1])


def kv_dequant(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """q * s per vector (FP64, exact)."""
    q = np.ascontiguousarray(q, dtype=np.int8)
    s = np.ascontiguousarray(s, dtype=np.float32)
    D = q.shape[-1]
    n = q.size // D
    out = np.empty(q.shape, dtype=np.float64)
    _load().oracle_kv_dequant(_ptr(q), _ptr(s), n, D, _ptr(out))
    return out


def attention_decode(q_bf16: np.ndarray, K: np.ndarray, V: np.ndarray, lens: np.ndarray,
                     scale: float) -> Tuple[np.ndarray, np.ndarray]:
    """Decode attention (one query per sequence, grouped-query heads) in FP64:
    q [B, Hq, D] BF16 bits, K and V [B, Hkv, S_max, D] (FP64 values), lens [B].
    Returns (out [B, Hq, D], T [B, Hq, D])."""
    q = np.ascontiguousarray(q_bf16, dtype=np.uint16)
    K = np.ascontiguousarray(K, dtype=np.float64)
    V = np.ascontiguousarray(V, dtype=np.float64)
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    B, Hq, D = q.shape
    _, Hkv, S_max, D2 = K.shape
    assert D2 == D and Hq % Hkv == 0 and V.shape == K.shape and lens.shape == (B,)
    out = np.empty((B, Hq, D), dtype=np.float64)
    T = np.empty((B, Hq, D), dtype=np.float64)
    _load().oracle_attention_decode(_ptr(q), _ptr(K), _ptr(V), _ptr(lens), B, Hq, Hkv, S_max, D,
                                    float(scale), _ptr(out), _ptr(T))
    return out, T


def rmsnorm(x_bf16: np.ndarray, gamma_bf16: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm of BF16 rows [M, K] (uint16 bit patterns) with BF16 weights
    gamma [K], in FP64: x / sqrt(mean(x^2) + eps) * gamma ("Deploying Hunyuan
    770B in INT8 on domestic accelerators", §4.1, RMSNorm in high precision
    before the INT8 GEMM). eps is taken as given (pass the FP32 value the
    kernel uses)."""
    lib = _load()
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    g = np.ascontiguousarray(gamma_bf16, dtype=np.uint16)
    M, K = x.shape
    if g.shape != (K,):
        raise ValueError("gamma must have K entries")
    y = np.empty((M, K), np.float64)
    lib.oracle_rmsnorm(_ptr(x), M, K, K, _ptr(g), float(eps), _ptr(y))
    return y
