"""Seeded synthetic inputs for the W8A8 group-scaled GEMM workloads.

This module is shared by the tests, the benchmark and the CPU oracle's
callers. It holds NO arithmetic of the method itself (no amax, no scale, no
rounding to int8, no GEMM): only random draws, the outlier-channel scaling of
the draws, the BF16 encoding of FP32 draws (which is how the workloads define
their BF16 activations), and MoE routing.

Determinism: every tensor is drawn from numpy ``PCG64`` streams built as
``SeedSequence(seed, spawn_key=(config_tag, tensor_tag, block))``; rows are
drawn in fixed blocks of ``ROW_BLOCK`` rows, each from its own stream, so any
subset of rows can be regenerated without drawing the whole tensor, and the
values do not depend on how a caller slices the tensor.

Workloads (sizes and distributions of the quantized-linear layers described
on the Hunyuan-770B INT8 deployment page, §3.1, and the MoE expert layers of
the same page §1.3 / §4.4):

* ``tiny``     M=16,  K=1024,  N=1024;  A ~ N(0,1); W ~ N(0,0.02); FP32 out.
* ``decode``   M in {1,8,32}, K=8192, N=28672; A ~ N(0,1) with round(1% K)
               fixed channels x30; W ~ N(0,0.02); BF16 out.
* ``prefill``  M=4096, K=8192, N=8192; A ~ N(0,1) with round(0.5% K)
               channels x50; BF16 out.
* ``moe``      E=64 experts, T=512 tokens, top-8 distinct experts per token,
               expert weight proportional to rank^-1.1 over a seeded
               permutation of expert ids, the 4 lowest-ranked experts given
               weight 0 (so some segments are empty); gate_up W [E,3072,4096],
               down W [E,4096,1536]; BF16 out.
* ``stress``   M=8192, K=16384, N=16384; A ~ Student-t(3) times a per-token
               magnitude 10^U(-2,2); FP32 out.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

ROW_BLOCK = 64
DEFAULT_SEED = 0

# Stable integer tags for the seed spawn keys.
_TENSOR_TAGS = {"act": 1, "weight": 2, "outlier_channels": 3, "routing": 4,
                "act_down": 5, "weight_down": 6, "gate_weight": 7, "norm_weight": 8}


@dataclass(frozen=True)
class DenseSpec:
    """One dense workload: Y[M,N] = quantized-linear(A[M,K], W[N,K])."""
    name: str
    tag: int
    M: int
    N: int
    K: int
    out_dtype: str                     # "bf16" or "fp32"
    act_kind: str = "normal"           # "normal" or "student_t_lognormal"
    outlier_frac: float = 0.0          # fraction of K channels scaled
    outlier_scale: float = 1.0
    w_std: float = 0.02

    @property
    def n_outliers(self) -> int:
        return int(round(self.outlier_frac * self.K))


@dataclass(frozen=True)
class MoESpec:
    """Grouped (MoE expert) workload: two expert GEMMs over routed rows."""
    name: str
    tag: int
    E: int
    T: int
    topk: int
    zipf_s: float
    zero_tail: int                     # lowest-ranked experts given weight 0
    N_up: int
    K_up: int
    N_down: int
    K_down: int
    out_dtype: str = "bf16"
    w_std: float = 0.02

    @property
    def R(self) -> int:
        return self.T * self.topk


DENSE: Dict[str, DenseSpec] = {
    "tiny": DenseSpec("tiny", 10, 16, 1024, 1024, "fp32"),
    "decode_m1": DenseSpec("decode_m1", 21, 1, 28672, 8192, "bf16", "normal", 0.01, 30.0),
    "decode_m8": DenseSpec("decode_m8", 22, 8, 28672, 8192, "bf16", "normal", 0.01, 30.0),
    "decode_m32": DenseSpec("decode_m32", 23, 32, 28672, 8192, "bf16", "normal", 0.01, 30.0),
    "prefill": DenseSpec("prefill", 30, 4096, 8192, 8192, "bf16", "normal", 0.005, 50.0),
    "stress": DenseSpec("stress", 50, 8192, 16384, 16384, "fp32", "student_t_lognormal"),
}

MOE: Dict[str, MoESpec] = {
    "moe": MoESpec("moe", 40, E=64, T=512, topk=8, zipf_s=1.1, zero_tail=4,
                   N_up=3072, K_up=4096, N_down=4096, K_down=1536),
    # Small routing edge case: few tokens over many experts, many empty segments.
    "moe_t16": MoESpec("moe_t16", 41, E=64, T=16, topk=8, zipf_s=1.1, zero_tail=4,
                       N_up=3072, K_up=4096, N_down=4096, K_down=1536),
}

# The decode workload is quoted over three token counts.
DECODE_MS = (1, 8, 32)


def _rng(seed: int, cfg_tag: int, tensor: str, block: int = 0) -> np.random.Generator:
    ss = np.random.SeedSequence(seed, spawn_key=(cfg_tag, _TENSOR_TAGS[tensor], block))
    return np.random.Generator(np.random.PCG64(ss))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Encode FP32 draws as BF16 bit patterns (round to nearest, ties to even).

    This is how the workloads define BF16 activations ("FP32 draws, then
    rounded to BF16"); inputs are finite by construction.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    bias = ((u >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)
    return ((u + bias) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """Widen BF16 bit patterns to FP32 (exact)."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def outlier_channels(spec: DenseSpec, seed: int = DEFAULT_SEED) -> np.ndarray:
    """The fixed K-channels that carry the outlier scale (sorted)."""
    n = spec.n_outliers
    if n == 0:
        return np.zeros(0, dtype=np.int64)
    rng = _rng(seed, spec.tag, "outlier_channels")
    return np.sort(rng.choice(spec.K, size=n, replace=False)).astype(np.int64)


def _act_block_f32(spec: DenseSpec, block: int, rows: int, seed: int,
                   channels: np.ndarray) -> np.ndarray:
    rng = _rng(seed, spec.tag, "act", block)
    if spec.act_kind == "normal":
        x = rng.standard_normal((rows, spec.K), dtype=np.float32)
    elif spec.act_kind == "student_t_lognormal":
        t = rng.standard_t(3.0, size=(rows, spec.K))
        mag = 10.0 ** rng.uniform(-2.0, 2.0, size=(rows, 1))
        x = (t * mag).astype(np.float32)
    else:
        raise ValueError(spec.act_kind)
    if channels.size:
        x[:, channels] *= np.float32(spec.outlier_scale)
    return x


def activations(spec: DenseSpec, rows: Optional[Sequence[int]] = None,
                M: Optional[int] = None, seed: int = DEFAULT_SEED) -> np.ndarray:
    """BF16 activations as uint16 bit patterns, shape [len(rows), K].

    ``rows`` selects token rows (default: all ``M`` rows, ``M`` defaulting to
    ``spec.M``). Row r always has the same values whatever else is selected.
    """
    M = spec.M if M is None else M
    rows = np.arange(M) if rows is None else np.asarray(rows, dtype=np.int64)
    ch = outlier_channels(spec, seed)
    out = np.empty((rows.size, spec.K), dtype=np.uint16)
    for b in np.unique(rows // ROW_BLOCK):
        sel = np.nonzero(rows // ROW_BLOCK == b)[0]
        blk = f32_to_bf16_bits(_act_block_f32(spec, int(b), ROW_BLOCK, seed, ch))
        out[sel] = blk[rows[sel] - b * ROW_BLOCK]
    return out


def _weight_block(tag: int, tensor: str, block: int, K: int, std: float,
                  seed: int) -> np.ndarray:
    rng = _rng(seed, tag, tensor, block)
    return (rng.standard_normal((ROW_BLOCK, K), dtype=np.float32) * np.float32(std))


def norm_weight(spec: DenseSpec, seed: int = DEFAULT_SEED) -> np.ndarray:
    """BF16 bit patterns [K] of an RMSNorm weight for the spec's activation
    rows: gamma ~ N(1, 0.25) (trained norm weights sit around 1; a few are
    small or negative)."""
    g = _rng(seed, spec.tag, "norm_weight").normal(1.0, 0.25, spec.K).astype(np.float32)
    return f32_to_bf16_bits(g)


def weights(spec: DenseSpec, rows: Optional[Sequence[int]] = None,
            seed: int = DEFAULT_SEED) -> np.ndarray:
    """FP32 weights [len(rows), K] (row n of the [N,K] weight matrix)."""
    rows = np.arange(spec.N) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.empty((rows.size, spec.K), dtype=np.float32)
    for b in np.unique(rows // ROW_BLOCK):
        sel = np.nonzero(rows // ROW_BLOCK == b)[0]
        blk = _weight_block(spec.tag, "weight", int(b), spec.K, spec.w_std, seed)
        out[sel] = blk[rows[sel] - b * ROW_BLOCK]
    return out


def weight_blocks(spec: DenseSpec, seed: int = DEFAULT_SEED, block_rows: int = 4096):
    """Yield (row0, W[row0:row0+block_rows]) FP32 chunks covering all N rows."""
    assert block_rows % ROW_BLOCK == 0
    for r0 in range(0, spec.N, block_rows):
        r1 = min(spec.N, r0 + block_rows)
        yield r0, weights(spec, np.arange(r0, r1), seed)


# ---------------------------------------------------------------- MoE inputs
@dataclass(frozen=True)
class Routing:
    token_of_row: np.ndarray   # [R] token id of each routed row (sorted by expert, then token)
    expert_of_row: np.ndarray  # [R]
    offsets: np.ndarray        # [E+1] int32, rows of expert e are [off[e], off[e+1])
    choice: np.ndarray         # [T, k] int32: each token's experts in the order they were drawn

    @property
    def counts(self) -> np.ndarray:
        return np.diff(self.offsets)


def expert_probabilities(spec: MoESpec, seed: int = DEFAULT_SEED) -> np.ndarray:
    """Routing weight of each expert: rank^-s over a seeded permutation of
    expert ids; the ``zero_tail`` lowest-ranked experts get weight 0."""
    rng = _rng(seed, spec.tag, "routing", 0)
    perm = rng.permutation(spec.E)             # perm[rank] = expert id
    ranks = np.arange(1, spec.E + 1, dtype=np.float64)
    w = ranks ** (-spec.zipf_s)
    if spec.zero_tail:
        w[-spec.zero_tail:] = 0.0
    p = np.zeros(spec.E)
    p[perm] = w / w.sum()
    return p


def routing(spec: MoESpec, seed: int = DEFAULT_SEED) -> Routing:
    """Top-k distinct experts per token, drawn without replacement with the
    Zipf-like expert weights; rows sorted by expert, ties by token id."""
    p = expert_probabilities(spec, seed)
    rng = _rng(seed, spec.tag, "routing", 1)
    choice = np.empty((spec.T, spec.topk), dtype=np.int64)
    for t in range(spec.T):
        choice[t] = rng.choice(spec.E, size=spec.topk, replace=False, p=p)
    tok = np.repeat(np.arange(spec.T), spec.topk)
    exp = choice.reshape(-1)
    order = np.lexsort((tok, exp))            # by expert, then token
    tok, exp = tok[order], exp[order]
    counts = np.bincount(exp, minlength=spec.E)
    offsets = np.zeros(spec.E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    return Routing(tok.astype(np.int64), exp.astype(np.int64), offsets, choice.astype(np.int32))


def moe_spec_as_dense(spec: MoESpec, which: str) -> DenseSpec:
    """Dense view of one MoE GEMM, used to draw activations row-blockwise."""
    if which == "up":
        return DenseSpec(spec.name + "_up", spec.tag * 10 + 1, spec.T, spec.N_up, spec.K_up,
                         spec.out_dtype)
    return DenseSpec(spec.name + "_down", spec.tag * 10 + 2, spec.R, spec.N_down, spec.K_down,
                     spec.out_dtype)


def moe_activations(spec: MoESpec, which: str, route: Routing,
                    seed: int = DEFAULT_SEED) -> np.ndarray:
    """BF16 activations of the routed rows, [R, K].

    gate_up: each routed row is its token's vector (duplicated tokens share
    values and therefore scales). down: an independent N(0,1) draw per
    routed row (the expert-local intermediate)."""
    d = moe_spec_as_dense(spec, which)
    if which == "up":
        x = activations(d, M=spec.T, seed=seed)
        return x[route.token_of_row]
    return activations(d, M=spec.R, seed=seed)


def moe_weights(spec: MoESpec, which: str, expert: int, rows: Optional[Sequence[int]] = None,
                seed: int = DEFAULT_SEED) -> np.ndarray:
    """FP32 weights of one expert, [len(rows), K] (default all N rows)."""
    N, K = (spec.N_up, spec.K_up) if which == "up" else (spec.N_down, spec.K_down)
    tensor = "weight" if which == "up" else "weight_down"
    rows = np.arange(N) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.empty((rows.size, K), dtype=np.float32)
    tag = spec.tag * 1000 + expert
    for b in np.unique(rows // ROW_BLOCK):
        sel = np.nonzero(rows // ROW_BLOCK == b)[0]
        blk = _weight_block(tag, tensor, int(b), K, spec.w_std, seed)
        out[sel] = blk[rows[sel] - b * ROW_BLOCK]
    return out


def random_offsets(rng: np.random.Generator, R: int, E: int, empty_frac: float = 0.3) -> np.ndarray:
    """Arbitrary nondecreasing offsets [E+1] with off[0]=0, off[E]=R and a
    share of empty segments (for ragged edge-case tests)."""
    w = rng.random(E)
    w[rng.random(E) < empty_frac] = 0.0
    if w.sum() == 0:
        w[0] = 1.0
    counts = np.floor(w / w.sum() * R).astype(np.int64)
    counts[np.argmax(w)] += R - counts.sum()
    off = np.zeros(E + 1, dtype=np.int32)
    off[1:] = np.cumsum(counts)
    return off


# -------------------------------------------------------- MoE expert FFN inputs
def moe_tokens(spec: MoESpec, seed: int = DEFAULT_SEED) -> np.ndarray:
    """The T token vectors (BF16 bit patterns [T, K_up]) entering the FFN: the
    same draws the gate_up workload routes (row t of the token matrix)."""
    return activations(moe_spec_as_dense(spec, "up"), M=spec.T, seed=seed)


def moe_gate_weights(spec: MoESpec, seed: int = DEFAULT_SEED) -> np.ndarray:
    """Router gate weights [T, k] float32: positive draws U(0.05, 1) scaled so
    each token's k weights sum to 1."""
    rng = _rng(seed, spec.tag, "gate_weight", 0)
    w = rng.uniform(0.05, 1.0, size=(spec.T, spec.topk))
    return (w / w.sum(axis=1, keepdims=True)).astype(np.float32)


# ---------------------------------------------------- INT8 KV cache decode
@dataclass(frozen=True)
class AttnSpec:
    """Decode attention over one layer's KV cache: B sequences of S positions
    each (all full), Hq query heads sharing Hkv kv heads, head dim D. The
    page's common configuration is a batch of 32 at a 4096-token context
    ("Deploying Hunyuan 770B in INT8 on domestic accelerators", §2.2); the
    head counts are a grouped-query shape of that model class."""
    name: str
    tag: int
    B: int
    Hq: int
    Hkv: int
    S: int
    D: int = 128
    k_outlier_frac: float = 0.02        # K channels scaled (keys carry channel outliers)
    k_outlier_scale: float = 8.0


ATTN: Dict[str, AttnSpec] = {
    "decode": AttnSpec("decode", 60, B=32, Hq=64, Hkv=8, S=4096),
}


def attn_inputs(spec: AttnSpec, seed: int = DEFAULT_SEED):
    """q [B, Hq, D], k and v [B, Hkv, S, D] as BF16 bit patterns: N(0,1) draws,
    a fixed round(k_outlier_frac * D) K channels scaled by k_outlier_scale."""
    rng = _rng(seed, spec.tag, "act", 0)
    q = f32_to_bf16_bits(rng.standard_normal((spec.B, spec.Hq, spec.D), dtype=np.float32))
    ch = np.sort(_rng(seed, spec.tag, "outlier_channels").choice(
        spec.D, size=int(round(spec.k_outlier_frac * spec.D)), replace=False))
    k = np.empty((spec.B, spec.Hkv, spec.S, spec.D), dtype=np.uint16)
    v = np.empty_like(k)
    for b in range(spec.B):
        kb = _rng(seed, spec.tag, "weight", b).standard_normal(
            (spec.Hkv, spec.S, spec.D), dtype=np.float32)
        kb[..., ch] *= np.float32(spec.k_outlier_scale)
        k[b] = f32_to_bf16_bits(kb)
        v[b] = f32_to_bf16_bits(_rng(seed, spec.tag, "weight_down", b).standard_normal(
            (spec.Hkv, spec.S, spec.D), dtype=np.float32))
    return q, k, v
