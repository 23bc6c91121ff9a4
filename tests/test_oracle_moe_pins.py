"""Pins of the oracle's MoE expert-FFN steps (CPU only): routing histogram,
offsets and permutation against a numpy brute force; the binary32 exponential
and silu against FP64 closed forms and identities; SwiGLU + per-token
requantization against exact rational arithmetic on rows where silu is exact;
the weighted un-permute against a brute-force sum; the whole FFN against its
dense special case.

Sources: "Deploying Hunyuan 770B in INT8 on domestic accelerators" §4.4 (a
global per-destination count first, then the transfer), §4.1 (SwiGLU next to
the INT8 GEMMs), §3.1 (per-token dynamic quantization of every GEMM input).
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads
from exact import f32_value, quantize_exact, round_to_f32


# ---------------------------------------------------------------- routing
def _route_brute(ids, E):
    T, k = ids.shape
    flat = ids.reshape(-1)
    valid = (flat >= 0) & (flat < E)
    counts = np.bincount(flat[valid], minlength=E)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    order = np.nonzero(valid)[0]
    order = order[np.lexsort((order, flat[order]))]   # by expert, then flattened index
    row_of = np.full(T * k, -1, np.int32)
    row_of[order] = np.arange(order.size)
    tok = np.full(T * k, -1, np.int32)
    pair = np.full(T * k, -1, np.int32)
    tok[:order.size] = order // k
    pair[:order.size] = order
    return offsets, row_of, tok, pair


@pytest.mark.parametrize("T,k,E,seed", [(1, 1, 1, 0), (7, 2, 5, 1), (64, 8, 16, 2),
                                        (33, 3, 40, 3)])
def test_route_matches_brute_force(T, k, E, seed):
    rng = np.random.default_rng(seed)
    ids = rng.integers(-2, E + 2, (T, k)).astype(np.int32)   # includes ids outside [0, E)
    got = oracle.moe_route(ids, E)
    want = _route_brute(ids, E)
    for g, w in zip(got, want):
        np.testing.assert_array_equal(g, w)


def test_route_of_the_moe_workload():
    spec = workloads.MOE["moe"]
    route = workloads.routing(spec)
    # the workload's (token, expert) pairs in token order give the ids matrix
    ids = np.empty((spec.T, spec.topk), np.int32)
    fill = np.zeros(spec.T, np.int64)
    for t, e in sorted(zip(route.token_of_row, route.expert_of_row)):
        ids[t, fill[t]] = e
        fill[t] += 1
    offsets, row_of, tok, _ = oracle.moe_route(ids, spec.E)
    np.testing.assert_array_equal(offsets, route.offsets)
    np.testing.assert_array_equal(tok, route.token_of_row)
    assert (np.diff(offsets) == 0).any()          # some experts get no token
    assert sorted(row_of.tolist()) == list(range(spec.R))


# ------------------------------------------------------- exp, silu (binary32)
def test_exp_f32_within_two_ulp_of_fp64_and_clamped():
    x = np.linspace(-87.0, 88.0, 200001).astype(np.float32)
    e = oracle.exp_f32(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    ulp = np.spacing(ref.astype(np.float32)).astype(np.float64)
    assert np.max(np.abs(e - ref) / ulp) <= 2.0
    assert oracle.exp_f32(np.float32([0.0]))[0] == 1.0
    big = oracle.exp_f32(np.float32([88.0, 100.0, 1e30]))
    small = oracle.exp_f32(np.float32([-87.0, -100.0, -1e30]))
    assert big[0] == big[1] == big[2] and np.isfinite(big).all()
    assert small[0] == small[1] == small[2] and small[0] > 0


def test_silu_identities_and_fp64_agreement():
    x = np.linspace(-40.0, 40.0, 80001).astype(np.float32)
    s = oracle.silu_f32(x).astype(np.float64)
    xd = x.astype(np.float64)
    ref = xd / (1.0 + np.exp(-xd))
    assert np.all(np.abs(s - ref) <= 4 * np.spacing(np.abs(ref).astype(np.float32)) + 1e-45)
    assert oracle.silu_f32(np.float32([0.0]))[0] == 0.0
    # silu(x) - silu(-x) = x
    sm = oracle.silu_f32(-x).astype(np.float64)
    assert np.all(np.abs((s - sm) - xd) <= 8 * np.spacing(np.abs(x)).astype(np.float64) + 1e-30)
    # e^-x underflows below half an ulp of 1 for x >= 17: silu is the identity
    big = np.float32([17.0, 20.5, 1000.0, 3.0e38])
    np.testing.assert_array_equal(oracle.silu_f32(big), big)


# ------------------------------------------- SwiGLU + per-token requantization
def test_swiglu_quant_matches_exact_rationals_where_silu_is_exact():
    rng = np.random.default_rng(5)
    R, I = 6, 64
    gate = rng.uniform(17.0, 60.0, (R, I)).astype(np.float32)   # silu(gate) == gate
    up = rng.standard_normal((R, I)).astype(np.float32)
    up[2] = 0.0                                                  # an all-zero row
    U = np.concatenate([gate, up], axis=1)
    qh, sh = oracle.swiglu_quant(U)
    for r in range(R):
        h = [round_to_f32(f32_value(g) * f32_value(u)) for g, u in zip(gate[r], up[r])]
        amax = max(abs(v) for v in h)
        s = round_to_f32(amax / 127)
        assert f32_value(sh[r]) == s
        want = [0 if s == 0 else quantize_exact(v, s) for v in h]
        assert qh[r].tolist() == want
    assert (qh[2] == 0).all() and sh[2] == 0.0


def test_swiglu_quant_invariants_on_random_rows():
    rng = np.random.default_rng(6)
    R, I = 32, 96
    U = (rng.standard_normal((R, 2 * I)) * 4).astype(np.float32)
    qh, sh = oracle.swiglu_quant(U)
    h = (oracle.silu_f32(U[:, :I]) * U[:, I:]).astype(np.float32)   # binary32 product
    np.testing.assert_array_equal(sh, (np.abs(h).max(axis=1) / np.float32(127)).astype(np.float32))
    deq = qh.astype(np.float64) * sh[:, None].astype(np.float64)
    assert np.all(np.abs(deq - h) <= sh[:, None] / 2 * (1 + 2.0 ** -16))
    assert (np.abs(qh).max(axis=1) == 127).all()
    # rows past nrows are untouched (zero)
    qh2, sh2 = oracle.swiglu_quant(U, nrows=10)
    np.testing.assert_array_equal(qh2[:10], qh[:10])
    assert (qh2[10:] == 0).all() and (sh2[10:] == 0).all()


# ------------------------------------------------------- weighted un-permute
def test_unpermute_matches_brute_force_and_one_hot_weights():
    rng = np.random.default_rng(7)
    T, k, E, H = 20, 3, 6, 40
    ids = rng.integers(-1, E, (T, k)).astype(np.int32)
    offsets, row_of, _, _ = oracle.moe_route(ids, E)
    D = rng.standard_normal((T * k, H))
    w = rng.random((T, k)).astype(np.float32)
    Y = oracle.moe_unpermute(D, row_of.reshape(T, k), w)
    want = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            r = row_of[t * k + j]
            if r >= 0:
                want[t] += np.float64(w[t, j]) * D[r]
    np.testing.assert_allclose(Y, want, rtol=0, atol=1e-12)
    onehot = np.zeros((T, k), np.float32)
    onehot[:, 1] = 1.0
    Y1 = oracle.moe_unpermute(D, row_of.reshape(T, k), onehot)
    for t in range(T):
        r = row_of[t * k + 1]
        np.testing.assert_array_equal(Y1[t], D[r] if r >= 0 else np.zeros(H))


# ------------------------------------------------------------- the whole FFN
def test_ffn_with_one_expert_and_top1_equals_the_dense_chain():
    rng = np.random.default_rng(8)
    T, H, I = 12, 256, 128
    x = workloads.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    w_up = (rng.standard_normal((2 * I, H)) * 0.05).astype(np.float32)
    w_dn = (rng.standard_normal((H, I)) * 0.05).astype(np.float32)
    qw_up, sw_up = oracle.quant_weight(w_up)
    qw_dn, sw_dn = oracle.quant_weight(w_dn)
    ids = np.zeros((T, 1), np.int32)
    wts = np.ones((T, 1), np.float32)
    out = oracle.moe_ffn(x, ids, wts, qw_up[None], sw_up[None], qw_dn[None], sw_dn[None])
    qa, sa = oracle.quant_act(x)
    U, _ = oracle.gemm(qa, sa, qw_up, sw_up)
    qh, sh = oracle.swiglu_quant(U.astype(np.float32))
    D, _ = oracle.gemm(qh, sh, qw_dn, sw_dn)
    np.testing.assert_array_equal(out["qh"], qh)
    np.testing.assert_array_equal(out["y"], D)


def test_ffn_is_linear_in_the_gate_weights_and_drops_unrouted_entries():
    rng = np.random.default_rng(9)
    T, k, E, H, I = 10, 2, 3, 128, 128
    x = workloads.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    qw_up, sw_up = zip(*[oracle.quant_weight((rng.standard_normal((2 * I, H)) * 0.05)
                                             .astype(np.float32)) for _ in range(E)])
    qw_dn, sw_dn = zip(*[oracle.quant_weight((rng.standard_normal((H, I)) * 0.05)
                                             .astype(np.float32)) for _ in range(E)])
    W = (np.stack(qw_up), np.stack(sw_up), np.stack(qw_dn), np.stack(sw_dn))
    ids = rng.integers(0, E, (T, k)).astype(np.int32)
    ids[3, 1] = E + 5                                  # not routed
    w = rng.random((T, k)).astype(np.float32)
    base = oracle.moe_ffn(x, ids, w, *W)
    twice = oracle.moe_ffn(x, ids, (2 * w).astype(np.float32), *W)
    np.testing.assert_allclose(twice["y"], 2 * base["y"], rtol=1e-15, atol=0)
    w2 = w.copy()
    w2[3, 1] = 123.0                                   # weight of the unrouted entry: no effect
    np.testing.assert_array_equal(oracle.moe_ffn(x, ids, w2, *W)["y"], base["y"])
    assert base["R"] == T * k - 1
