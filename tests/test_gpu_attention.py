"""GPU parity of the INT8 KV cache and decode attention (through the C ABI)
against the CPU oracle: the cache write (per-vector scales and codes)
bit-exact; attention over the INT8 cache (dequantized inside the kernel) and
over a BF16 cache within the FP32 error bound derived below; grouped-query
heads that share a kv head and a query give identical outputs; empty and
clamped sequence lengths.

Bound: a score is a 128-term FP32 dot product of exact products, then scaled
(2 roundings): |ds_j| <= (D + 2) 2^-24 A_j with A_j = scale * sum_d |q_d k_jd|.
Each output is a convex combination of the V rows, so with T_d = sum_j p_j
|v_jd| (the oracle's magnitude):
  |out - out*| <= (2 max_j A_j (D + 2) 2^-24 + (S + 64) 2^-24 + 16 * 2^-22) T_d
(the score error moves the weights by at most 2 max |ds|; the sums over
positions, chunk merges and exp add the rest), plus half a BF16 ulp for BF16.

Source: "Deploying Hunyuan 770B in INT8 on domestic accelerators" §3.4, §2.2.
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
D = 128


def bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(torch.bfloat16)


def _bound(q_bits, K, lens, scale, T):
    """Per-output bound (see the module docstring)."""
    qf = np.abs(workloads.bf16_bits_to_f32(q_bits).astype(np.float64))
    B, Hq, _ = q_bits.shape
    Hkv, S = K.shape[1], K.shape[2]
    G = Hq // Hkv
    bound = np.zeros_like(T)
    for b in range(B):
        L = int(min(max(lens[b], 0), S))
        if L == 0:
            continue
        for h in range(Hq):
            A = scale * (np.abs(K[b, h // G, :L]) @ qf[b, h])
            rel = 2 * A.max() * (D + 2) * 2.0 ** -24 + (S + 64) * 2.0 ** -24 + 16 * 2.0 ** -22
            bound[b, h] = rel * T[b, h]
    return bound


def _run(q, kc, vc, lens, scale, ks=None, vs=None, out_dtype=torch.float32):
    out = torch.full((q.shape[0], q.shape[1], D), float("nan"), dtype=out_dtype, device=DEV)
    w8.attention_decode(q, kc, vc, lens, scale, k_scale=ks, v_scale=vs, out_dtype=out_dtype,
                        out=out)
    torch.cuda.synchronize()
    return out


def test_kv_quant_scatter_bitexact():
    rng = np.random.default_rng(40)
    n, rows = 50, 80
    x = workloads.f32_to_bf16_bits((rng.standard_normal((n, D)) * 3).astype(np.float32))
    x[4] = 0
    dst = rng.permutation(rows)[:n].astype(np.int32)
    dst[7] = -1                                              # not written
    cache = torch.zeros((rows, D), dtype=torch.int8, device=DEV)
    scales = torch.full((rows,), -1.0, dtype=torch.float32, device=DEV)
    w8.kv_quant(bf16_dev(x), cache, scales, dst_rows=torch.from_numpy(dst).to(DEV))
    torch.cuda.synchronize()
    q_o, s_o = oracle.kv_quant(x)
    c, s = cache.cpu().numpy(), scales.cpu().numpy()
    for i in range(n):
        if dst[i] < 0:
            continue
        np.testing.assert_array_equal(c[dst[i]], q_o[i])
        assert s[dst[i]].view(np.uint32) == s_o[i].view(np.uint32)
    untouched = np.setdiff1d(np.arange(rows), dst[dst >= 0])
    assert (c[untouched] == 0).all() and (s[untouched] == -1.0).all()


def _problem(seed, B=4, Hq=16, Hkv=2, S=300):
    rng = np.random.default_rng(seed)
    q = workloads.f32_to_bf16_bits(rng.standard_normal((B, Hq, D)).astype(np.float32))
    k = workloads.f32_to_bf16_bits((rng.standard_normal((B, Hkv, S, D)) *
                                    rng.uniform(0.5, 4, (1, 1, 1, D))).astype(np.float32))
    v = workloads.f32_to_bf16_bits(rng.standard_normal((B, Hkv, S, D)).astype(np.float32))
    lens = np.array([S, 129, 1, 0][:B], np.int32)
    return q, k, v, lens


@pytest.mark.parametrize("out", ["fp32", "bf16"])
def test_int8_cache_attention_within_bound(out):
    q, k, v, lens = _problem(41)
    B, Hkv, S, _ = k.shape
    scale = 1 / np.sqrt(D)
    kc = torch.empty((B, Hkv, S, D), dtype=torch.int8, device=DEV)
    vc = torch.empty_like(kc)
    ks = torch.empty((B, Hkv, S), dtype=torch.float32, device=DEV)
    vs = torch.empty_like(ks)
    w8.kv_quant(bf16_dev(k.reshape(-1, D)), kc, ks)
    w8.kv_quant(bf16_dev(v.reshape(-1, D)), vc, vs)
    qk, sk = oracle.kv_quant(k)
    qv, sv = oracle.kv_quant(v)
    np.testing.assert_array_equal(kc.cpu().numpy(), qk)
    np.testing.assert_array_equal(vs.cpu().numpy().view(np.uint32), sv.view(np.uint32))
    dt = torch.float32 if out == "fp32" else torch.bfloat16
    y = _run(bf16_dev(q), kc, vc, torch.from_numpy(lens).to(DEV), scale, ks, vs, dt)
    K, V = oracle.kv_dequant(qk, sk), oracle.kv_dequant(qv, sv)
    y_ref, T = oracle.attention_decode(q, K, V, lens, scale)
    bound = _bound(q, K, lens, scale, T)
    yv = y.float().cpu().numpy().astype(np.float64)
    if out == "bf16":
        bound = bound + 0.5 * oracle.bf16_ulp(oracle.bf16_round(y_ref))
    assert not np.isnan(yv).any()
    assert np.all(np.abs(yv - y_ref) <= bound), f"worst {np.max(np.abs(yv - y_ref) - bound)}"
    assert (yv[3] == 0).all()                                # empty sequence


def test_bf16_cache_attention_within_bound():
    q, k, v, lens = _problem(42, B=3, Hq=8, Hkv=8, S=200)
    lens = np.array([200, 1000, 77], np.int32)               # 1000 is clamped to 200
    scale = 0.1
    y = _run(bf16_dev(q), bf16_dev(k), bf16_dev(v), torch.from_numpy(lens).to(DEV), scale)
    K = workloads.bf16_bits_to_f32(k).astype(np.float64)
    V = workloads.bf16_bits_to_f32(v).astype(np.float64)
    y_ref, T = oracle.attention_decode(q, K, V, lens, scale)
    bound = _bound(q, K, lens, scale, T)
    yv = y.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(yv - y_ref) <= bound)


def test_heads_sharing_a_kv_head_and_query_agree():
    q, k, v, lens = _problem(43, B=2, Hq=16, Hkv=1, S=260)
    q[:, 5] = q[:, 0]
    kc = torch.empty((2, 1, 260, D), dtype=torch.int8, device=DEV)
    vc = torch.empty_like(kc)
    ks = torch.empty((2, 1, 260), dtype=torch.float32, device=DEV)
    vs = torch.empty_like(ks)
    w8.kv_quant(bf16_dev(k.reshape(-1, D)), kc, ks)
    w8.kv_quant(bf16_dev(v.reshape(-1, D)), vc, vs)
    y = _run(bf16_dev(q), kc, vc, torch.from_numpy(lens[:2]).to(DEV), 0.09, ks, vs)
    assert torch.equal(y[:, 0], y[:, 5])


def test_decode_workload_sampled():
    spec = workloads.ATTN["decode"]
    q, k, v = workloads.attn_inputs(spec)
    B, Hkv, S = spec.B, spec.Hkv, spec.S
    kc = torch.empty((B, Hkv, S, D), dtype=torch.int8, device=DEV)
    vc = torch.empty_like(kc)
    ks = torch.empty((B, Hkv, S), dtype=torch.float32, device=DEV)
    vs = torch.empty_like(ks)
    w8.kv_quant(bf16_dev(k.reshape(-1, D)), kc, ks)
    w8.kv_quant(bf16_dev(v.reshape(-1, D)), vc, vs)
    lens = np.full(B, S, np.int32)
    scale = 1 / np.sqrt(D)
    y = _run(bf16_dev(q), kc, vc, torch.from_numpy(lens).to(DEV), scale, ks, vs,
             torch.bfloat16)
    for b in (0, 13, 31):
        qk, sk = oracle.kv_quant(k[b:b + 1])
        qv, sv = oracle.kv_quant(v[b:b + 1])
        np.testing.assert_array_equal(kc[b:b + 1].cpu().numpy(), qk)
        K, V = oracle.kv_dequant(qk, sk), oracle.kv_dequant(qv, sv)
        y_ref, T = oracle.attention_decode(q[b:b + 1], K, V, lens[b:b + 1], scale)
        bound = _bound(q[b:b + 1], K, lens[b:b + 1], scale, T)
        bound = bound + 0.5 * oracle.bf16_ulp(oracle.bf16_round(y_ref))
        yv = y[b:b + 1].float().cpu().numpy().astype(np.float64)
        assert np.all(np.abs(yv - y_ref) <= bound)
    assert w8.device_error() == 0
