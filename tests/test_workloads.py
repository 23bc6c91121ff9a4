"""CPU tests of the seeded synthetic input recipe (no method arithmetic)."""
import numpy as np
import pytest

import workloads


def test_bf16_encoding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(5000) * 10.0 ** rng.uniform(-10, 10, 5000)).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(workloads.f32_to_bf16_bits(x), ref)


def test_row_subsets_are_stable():
    spec = workloads.DENSE["decode_m32"]
    full = workloads.activations(spec)
    sub = workloads.activations(spec, rows=[31, 3, 0])
    np.testing.assert_array_equal(sub, full[[31, 3, 0]])
    w = workloads.weights(spec, rows=[5, 70, 200])
    w2 = workloads.weights(spec, rows=np.arange(64, 128))
    np.testing.assert_array_equal(w[1], w2[6])


def test_outlier_channels_counts_and_scale():
    d = workloads.DENSE["decode_m8"]
    p = workloads.DENSE["prefill"]
    assert workloads.outlier_channels(d).size == 82
    assert workloads.outlier_channels(p).size == 41
    ch = workloads.outlier_channels(d)
    x = workloads.bf16_bits_to_f32(workloads.activations(d)).astype(np.float64)
    mask = np.zeros(d.K, bool)
    mask[ch] = True
    ratio = np.abs(x[:, mask]).mean() / np.abs(x[:, ~mask]).mean()
    assert 20 < ratio < 40


def test_stress_activation_magnitudes_span_four_decades():
    s = workloads.DENSE["stress"]
    x = workloads.bf16_bits_to_f32(workloads.activations(s, rows=np.arange(128)))
    med = np.median(np.abs(x), axis=1)
    assert med.min() < 0.1 and med.max() > 10


def test_moe_routing_recipe():
    spec = workloads.MOE["moe"]
    r = workloads.routing(spec)
    assert r.offsets[0] == 0 and r.offsets[-1] == spec.R == 4096
    assert np.all(np.diff(r.offsets) >= 0)
    # each token routed to topk distinct experts
    pairs = set(zip(r.token_of_row.tolist(), r.expert_of_row.tolist()))
    assert len(pairs) == spec.R
    counts = np.bincount(r.token_of_row, minlength=spec.T)
    assert np.all(counts == spec.topk)
    # sorted by expert then token; zero-weight experts are empty
    assert np.all(np.diff(r.expert_of_row) >= 0)
    for e in range(spec.E):
        seg = r.token_of_row[r.offsets[e]:r.offsets[e + 1]]
        assert np.all(np.diff(seg) > 0)
    p = workloads.expert_probabilities(spec)
    assert np.all(r.counts[p == 0] == 0) and (p == 0).sum() == 4
    assert r.counts.max() > 4 * r.counts[r.counts > 0].min()   # ragged


def test_moe_t16_has_many_empty_segments():
    r = workloads.routing(workloads.MOE["moe_t16"])
    assert (r.counts == 0).sum() >= 20 and r.offsets[-1] == 128


def test_moe_up_rows_duplicate_token_vectors():
    spec = workloads.MOE["moe_t16"]
    r = workloads.routing(spec)
    a = workloads.moe_activations(spec, "up", r)
    i, j = np.nonzero(r.token_of_row[:, None] == r.token_of_row[None, :])
    k = i != j
    np.testing.assert_array_equal(a[i[k][:5]], a[j[k][:5]])
