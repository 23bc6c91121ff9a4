"""GPU parity of the MoE expert FFN (through the C ABI) against the CPU oracle.

Every step is compared with the oracle on the oracle's own inputs:
  * routing (offsets, permutation): bit-exact;
  * transfer + per-token quantization of the permuted rows: bit-exact;
  * SwiGLU (binary32, same exponential on both sides): bit-exact h, and the
    requantized codes and scales bit-exact;
  * weighted un-permute: FP32 accumulation over k entries,
    |y - y*| <= (k + 1) 2^-24 sum_j |w_j D_j| (+ half a BF16 ulp for BF16);
  * the grouped GEMMs are the kernels of tests/test_gpu_parity.py.
The fused call must then equal the composition of the separate calls bit for
bit, and the end-to-end result is compared with the oracle's FFN: the codes
of the down GEMM's input may differ from the oracle's only where the gate_up
outputs (FP32 vs the oracle's FP64) straddle a rounding boundary.
Sources: "Deploying Hunyuan 770B in INT8 on domestic accelerators" §4.4,
§4.1 and §3.1.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import moe_gemm_gb300 as w8  # noqa: E402

DEV = torch.device("cuda:0")
G = 128


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(DEV)


def bf16_dev(bits):
    return dev(bits.view(np.int16)).view(torch.bfloat16)


def small_problem(seed, T=48, k=4, E=8, H=512, I=256, invalid=True):
    rng = np.random.default_rng(seed)
    x = workloads.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    if invalid:
        ids[1, 0] = -1
        ids[5, k - 1] = E + 3
    ids[:, 0][ids[:, 0] == E - 1] = 0              # expert E-1 gets fewer rows
    w = rng.uniform(0.05, 1.0, (T, k)).astype(np.float32)
    wu = [(rng.standard_normal((2 * I, H)) * 0.05).astype(np.float32) for _ in range(E)]
    wd = [(rng.standard_normal((H, I)) * 0.05).astype(np.float32) for _ in range(E)]
    qu = [oracle.quant_weight(a) for a in wu]
    qd = [oracle.quant_weight(a) for a in wd]
    W = (np.stack([q for q, _ in qu]), np.stack([s for _, s in qu]),
         np.stack([q for q, _ in qd]), np.stack([s for _, s in qd]))
    return x, ids, w, W


# ------------------------------------------------------------------ routing
@pytest.mark.parametrize("T,k,E,seed", [(1, 1, 1, 0), (37, 3, 11, 1), (512, 8, 64, 2),
                                        (2000, 6, 1024, 3)])
def test_route_bitexact(T, k, E, seed):
    rng = np.random.default_rng(seed)
    ids = rng.integers(-1, E + 1, (T, k)).astype(np.int32)
    got = [t.cpu().numpy() for t in w8.moe_route(dev(ids), E)]
    want = oracle.moe_route(ids, E)
    for g, x in zip(got, want):
        np.testing.assert_array_equal(g, x)


def test_route_of_the_moe_workload():
    spec = workloads.MOE["moe"]
    route = workloads.routing(spec)
    got = [t.cpu().numpy() for t in w8.moe_route(dev(route.choice), spec.E)]
    want = oracle.moe_route(route.choice, spec.E)
    for g, x in zip(got, want):
        np.testing.assert_array_equal(g, x)
    np.testing.assert_array_equal(got[0], route.offsets)


# ------------------------------------------------ transfer + quantization
def test_quant_act_rows_is_the_quantizer_on_gathered_rows():
    spec = workloads.MOE["moe"]
    route = workloads.routing(spec)
    x = workloads.moe_tokens(spec)
    offsets, _, tok, _ = oracle.moe_route(route.choice, spec.E)
    qa, sa = w8.quant_act_rows(bf16_dev(x), dev(tok))
    R = int(offsets[-1])
    qa_o, sa_o = oracle.quant_act(x[tok[:R]])
    np.testing.assert_array_equal(qa.cpu().numpy()[:R], qa_o)
    np.testing.assert_array_equal(sa.cpu().numpy()[:R].view(np.uint32), sa_o.view(np.uint32))


# ------------------------------------------------------------------ SwiGLU
def test_swiglu_bitexact_over_a_sweep():
    g = np.concatenate([np.linspace(-100, 100, 40001), [0.0, -0.0, 1e-30, -1e-30, 87.0, -87.0,
                                                        88.5, -88.5, 3e38, -3e38]])
    g = g.astype(np.float32)
    n = (g.size + 63) // 64 * 64
    gate = np.zeros(n, np.float32)
    gate[:g.size] = g
    up = np.random.default_rng(0).standard_normal(n).astype(np.float32)
    up[::7] = 1.0
    I = 64
    U = np.concatenate([gate.reshape(-1, I), up.reshape(-1, I)], axis=1)
    h = w8.swiglu(dev(U)).cpu().numpy()
    with np.errstate(over="ignore"):   # +-3e38 gates times |up| > 1.13 overflow on both sides
        want = (oracle.silu_f32(gate) * up).astype(np.float32).reshape(-1, I)   # binary32 product
    np.testing.assert_array_equal(h.view(np.uint32), want.view(np.uint32))


def test_swiglu_quant_bitexact_on_the_oracle_gate_up_output():
    x, ids, w, W = small_problem(11)
    ref = oracle.moe_ffn(x, ids, w, *W)
    U = ref["U"]                                   # the oracle's FP32 gate_up output
    off = ref["offsets"]
    qh, sh = w8.swiglu_quant(dev(U), dev(off))
    qh_o, sh_o = oracle.swiglu_quant(U, int(off[-1]))
    np.testing.assert_array_equal(qh.cpu().numpy(), qh_o)
    np.testing.assert_array_equal(sh.cpu().numpy().view(np.uint32), sh_o.view(np.uint32))


def test_swiglu_quant_zero_and_tiny_rows():
    I = 128
    U = np.zeros((4, 2 * I), np.float32)
    U[1, :I] = 30.0                                # gate saturated, up zero: h = 0
    U[2, :I], U[2, I:] = 20.0, 1e-30               # subnormal-range products
    U[3] = np.random.default_rng(1).standard_normal(2 * I).astype(np.float32)
    qh, sh = w8.swiglu_quant(dev(U))
    qh_o, sh_o = oracle.swiglu_quant(U)
    np.testing.assert_array_equal(qh.cpu().numpy(), qh_o)
    np.testing.assert_array_equal(sh.cpu().numpy().view(np.uint32), sh_o.view(np.uint32))
    assert (qh_o[0] == 0).all() and sh_o[0] == 0.0


# -------------------------------------------------------------- un-permute
@pytest.mark.parametrize("out", ["fp32", "bf16"])
def test_unpermute_within_fp32_bound(out):
    x, ids, w, W = small_problem(12)
    ref = oracle.moe_ffn(x, ids, w, *W)
    D32 = ref["D"].astype(np.float32)
    T, k = ids.shape
    dt = torch.float32 if out == "fp32" else torch.bfloat16
    y = w8.moe_unpermute(dev(D32), dev(ref["row_of"]), dev(w), out_dtype=dt)
    y_ref = oracle.moe_unpermute(D32.astype(np.float64), ref["row_of"].reshape(T, k), w)
    mag = oracle.moe_unpermute(np.abs(D32).astype(np.float64), ref["row_of"].reshape(T, k), w)
    bound = (k + 1) * 2.0 ** -24 * mag
    if out == "fp32":
        yv = y.cpu().numpy().astype(np.float64)
    else:
        yv = oracle.bf16_to_float(y.view(torch.int16).cpu().numpy().view(np.uint16))
        bound = bound + 0.5 * oracle.bf16_ulp(oracle.bf16_round(y_ref))
    assert np.all(np.abs(yv - y_ref) <= bound)


# --------------------------------------------------------------- fused FFN
def _staged(x_d, ids_d, w_d, W_d, E, out_dtype):
    """The FFN as separate library calls (int8 codes between them)."""
    qw_up, sw_up, qw_dn, sw_dn = W_d
    T, k = ids_d.shape
    offsets, row_of, tok, _ = w8.moe_route(ids_d, E)
    qa, sa = w8.quant_act_rows(x_d, tok)
    U = w8.grouped_gemm(qa, sa, offsets, qw_up, sw_up, out_dtype=torch.float32)
    qh, sh = w8.swiglu_quant(U, offsets)
    D = w8.grouped_gemm(qh, sh, offsets, qw_dn, sw_dn, out_dtype=torch.float32)
    # (rows past offsets[E] of U and D are never written, and never read)
    y = w8.moe_unpermute(D, row_of, w_d, out_dtype=out_dtype)
    return y, dict(offsets=offsets, row_of=row_of, tok=tok, qa=qa, sa=sa, U=U, qh=qh, sh=sh, D=D)


@pytest.mark.parametrize("out", ["bf16", "fp32"])
def test_fused_ffn_equals_the_separate_calls_and_tracks_the_oracle(out):
    x, ids, w, W = small_problem(13)
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    W_d = [dev(a) for a in W]
    x_d, ids_d, w_d = bf16_dev(x), dev(ids), dev(w)
    y = torch.full((x.shape[0], x.shape[1]), float("nan"), dtype=dt, device=DEV)
    w8.moe_ffn(x_d, ids_d, w_d, *W_d, out_dtype=dt, out=y)
    y_st, st = _staged(x_d, ids_d, w_d, W_d, W[0].shape[0], dt)
    torch.cuda.synchronize()
    assert torch.equal(y, y_st), "fused FFN differs from the composition of its steps"
    assert w8.device_error() == 0

    ref = oracle.moe_ffn(x, ids, w, *W)
    R = ref["R"]
    np.testing.assert_array_equal(st["offsets"].cpu().numpy(), ref["offsets"])
    np.testing.assert_array_equal(st["qa"].cpu().numpy()[:R], ref["qa"][:R])
    # gate_up output within the GEMM's FP32 bound of the exact values
    Ug = st["U"].cpu().numpy()[:R].astype(np.float64)
    Ux, Tu = oracle.grouped_gemm(ref["qa"], ref["sa"], ref["offsets"], W[0], W[1])
    K = x.shape[1]
    assert np.all(np.abs(Ug - Ux[:R]) <= (K // G + 2) * 2.0 ** -24 * Tu[:R])
    # down-GEMM input codes: equal to the oracle's wherever the FP32 gate_up
    # output leaves the requantization decision unchanged; a differing code
    # is off by one and its exact quotient lies within the FP32 perturbation
    # of a rounding boundary
    qh = st["qh"].cpu().numpy()[:R].astype(np.int64)
    qh_o = ref["qh"][:R].astype(np.int64)
    diff = qh != qh_o
    assert np.all(np.abs(qh - qh_o) <= 1)
    assert diff.mean() < 1e-3, f"{diff.sum()} of {diff.size} down-GEMM input codes differ"
    # end to end: relative RMS error small, compared against the output scale
    yv = y.float().cpu().numpy().astype(np.float64)
    y_ref = ref["y"]
    rms = np.sqrt(np.mean(y_ref ** 2))
    assert not np.isnan(yv).any()
    assert np.sqrt(np.mean((yv - y_ref) ** 2)) <= 1e-2 * rms
    assert np.max(np.abs(yv - y_ref)) <= 0.1 * rms


def test_ffn_with_all_tokens_on_one_expert_and_top1():
    x, _, _, W = small_problem(14, T=40, k=1, E=3, invalid=False)
    ids = np.full((40, 1), 2, np.int32)
    w = np.ones((40, 1), np.float32)
    W_d = [dev(a) for a in W]
    y = w8.moe_ffn(bf16_dev(x), dev(ids), dev(w), *W_d, out_dtype=torch.float32)
    # the dense chain through the library: linear -> swiglu_quant -> gemm,
    # with workspaces that hold no K-split area, so every output accumulates
    # its groups in one chain, as the grouped GEMM does
    T, H = x.shape
    I = W[2].shape[2]
    r = lambda v: (v + 255) // 256 * 256  # noqa: E731
    ws1 = torch.empty(r(T * H * 2) + r(T * 4), dtype=torch.uint8, device=DEV)
    U = w8.linear(bf16_dev(x), W_d[0][2], W_d[1][2], out_dtype=torch.float32, workspace=ws1)
    qh, sh = w8.swiglu_quant(U)
    ws2 = torch.empty(r(T * I * 2), dtype=torch.uint8, device=DEV)
    D = w8.gemm(qh, sh, W_d[2][2], W_d[3][2], out_dtype=torch.float32, workspace=ws2)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(y.cpu().numpy(), D.cpu().numpy())


def test_ffn_full_size_workload_sampled_tokens():
    spec = workloads.MOE["moe"]
    route = workloads.routing(spec)
    x = workloads.moe_tokens(spec)
    w = workloads.moe_gate_weights(spec)
    E, H, I = spec.E, spec.K_up, spec.K_down
    qw_up = torch.empty((E, 2 * I, H), dtype=torch.int8, device=DEV)
    sw_up = torch.empty((E, 2 * I, H // G), dtype=torch.float32, device=DEV)
    qw_dn = torch.empty((E, H, I), dtype=torch.int8, device=DEV)
    sw_dn = torch.empty((E, H, I // G), dtype=torch.float32, device=DEV)
    for e in range(E):
        q, s = w8.quant_weight(dev(workloads.moe_weights(spec, "up", e)))
        qw_up[e].copy_(q)
        sw_up[e].copy_(s)
        q, s = w8.quant_weight(dev(workloads.moe_weights(spec, "down", e)))
        qw_dn[e].copy_(q)
        sw_dn[e].copy_(s)
    W_d = (qw_up, sw_up, qw_dn, sw_dn)
    x_d, ids_d, w_d = bf16_dev(x), dev(route.choice), dev(w)
    y = torch.full((spec.T, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    w8.moe_ffn(x_d, ids_d, w_d, *W_d, out=y)
    y_st, _ = _staged(x_d, ids_d, w_d, W_d, E, torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(y, y_st)
    assert not torch.isnan(y.float()).any().item()
    # a few tokens through the oracle's FFN (each token alone: k routed rows)
    for t in (0, 77, 300, 511):
        ids_t = route.choice[t:t + 1]
        used = np.unique(ids_t)
        remap = {int(e): i for i, e in enumerate(used)}
        Wt = []
        for which in ("up", "down"):
            qs = [oracle.quant_weight(workloads.moe_weights(spec, which, int(e))) for e in used]
            Wt += [np.stack([q for q, _ in qs]), np.stack([s for _, s in qs])]
        ids_local = np.vectorize(remap.get)(ids_t).astype(np.int32)
        ref = oracle.moe_ffn(x[t:t + 1], ids_local, w[t:t + 1], *Wt)
        yv = y[t].float().cpu().numpy().astype(np.float64)
        rms = np.sqrt(np.mean(ref["y"] ** 2))
        assert np.sqrt(np.mean((yv - ref["y"][0]) ** 2)) <= 1e-2 * rms
