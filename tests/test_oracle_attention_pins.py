"""Pins of the oracle's INT8 KV cache and decode attention (CPU only): the
per-vector KV quantization is the per-token quantizer; attention against a
numpy softmax brute force, one position (output = the value), equal keys
(output = mean of the values), a dominant key, grouped-query head sharing,
position permutation invariance and empty sequences.

Source: "Deploying Hunyuan 770B in INT8 on domestic accelerators" §3.4
(per-token dynamic scales of the INT8 KV cache, dequantized inside the
attention kernel) and §2.2 (the cache's shape).
"""
import numpy as np

import oracle
import workloads


def _inputs(seed, B=3, Hq=8, Hkv=2, S=40, D=64):
    rng = np.random.default_rng(seed)
    q = workloads.f32_to_bf16_bits(rng.standard_normal((B, Hq, D)).astype(np.float32))
    k = workloads.f32_to_bf16_bits(rng.standard_normal((B, Hkv, S, D)).astype(np.float32))
    v = workloads.f32_to_bf16_bits(rng.standard_normal((B, Hkv, S, D)).astype(np.float32))
    return q, k, v


def test_kv_quant_is_the_per_token_quantizer():
    _, k, _ = _inputs(0)
    qk, sk = oracle.kv_quant(k)
    qa, sa = oracle.quant_act(k.reshape(-1, k.shape[-1]))
    np.testing.assert_array_equal(qk.reshape(qa.shape), qa)
    np.testing.assert_array_equal(sk.reshape(-1), sa)
    deq = oracle.kv_dequant(qk, sk)
    np.testing.assert_array_equal(deq, qk.astype(np.float64) * sk[..., None].astype(np.float64))


def test_attention_matches_numpy_softmax():
    q, k, v = _inputs(1)
    K = workloads.bf16_bits_to_f32(k).astype(np.float64)
    V = workloads.bf16_bits_to_f32(v).astype(np.float64)
    lens = np.array([40, 17, 1], np.int32)
    scale = 1 / np.sqrt(64)
    out, T = oracle.attention_decode(q, K, V, lens, scale)
    qf = workloads.bf16_bits_to_f32(q).astype(np.float64)
    B, Hq, D = q.shape
    G = Hq // K.shape[1]
    for b in range(B):
        for h in range(Hq):
            L = lens[b]
            s = (K[b, h // G, :L] @ qf[b, h]) * scale
            p = np.exp(s - s.max())
            p /= p.sum()
            np.testing.assert_allclose(out[b, h], p @ V[b, h // G, :L], rtol=1e-12, atol=1e-14)
            np.testing.assert_allclose(T[b, h], p @ np.abs(V[b, h // G, :L]), rtol=1e-12, atol=1e-14)


def test_attention_special_cases():
    q, k, v = _inputs(2, B=1, Hq=4, Hkv=1, S=30, D=32)
    V = workloads.bf16_bits_to_f32(v).astype(np.float64)
    K = workloads.bf16_bits_to_f32(k).astype(np.float64)
    # one position: the output is that value
    out, _ = oracle.attention_decode(q, K, V, np.array([1], np.int32), 0.3)
    np.testing.assert_array_equal(out[0, 0], V[0, 0, 0])
    # equal keys: uniform weights, the mean of the values
    Ke = np.repeat(K[:, :, :1], 30, axis=2)
    out, _ = oracle.attention_decode(q, Ke, V, np.array([30], np.int32), 0.3)
    np.testing.assert_allclose(out[0, 2], V[0, 0].mean(axis=0), rtol=1e-12, atol=1e-14)
    # a dominant key: the output is its value
    Kd = K.copy()
    qf = workloads.bf16_bits_to_f32(q).astype(np.float64)
    Kd[0, 0, 7] = 1e4 * qf[0, 1]
    out, _ = oracle.attention_decode(q, Kd, V, np.array([30], np.int32), 1.0)
    np.testing.assert_allclose(out[0, 1], V[0, 0, 7], rtol=1e-12)
    # an empty sequence gives zeros
    out, T = oracle.attention_decode(q, K, V, np.array([0], np.int32), 0.3)
    assert (out == 0).all() and (T == 0).all()


def test_attention_heads_share_kv_and_positions_commute():
    q, k, v = _inputs(3, B=2, Hq=6, Hkv=2, S=25, D=16)
    q[:, 1] = q[:, 0]                                  # heads 0, 1 and 2 share kv head 0
    K = workloads.bf16_bits_to_f32(k).astype(np.float64)
    V = workloads.bf16_bits_to_f32(v).astype(np.float64)
    lens = np.array([25, 25], np.int32)
    out, _ = oracle.attention_decode(q, K, V, lens, 0.25)
    np.testing.assert_array_equal(out[:, 0], out[:, 1])
    perm = np.random.default_rng(4).permutation(25)
    out_p, _ = oracle.attention_decode(q, K[:, :, perm], V[:, :, perm], lens, 0.25)
    np.testing.assert_allclose(out_p, out, rtol=1e-12, atol=1e-14)
