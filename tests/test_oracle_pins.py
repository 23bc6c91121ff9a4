"""Pins for the CPU oracle (CPU only).

Each oracle function is checked against something other than itself:
exact rational arithmetic (tests/exact.py), closed forms, numpy integer
matmul as a library primitive, and invariants of the method ("Deploying
Hunyuan 770B in INT8 on domestic accelerators" §3.1: per-group-128 weights,
per-token dynamic activations, round(x/scale), INT8 x INT8 -> INT32, FP32
scales applied at the end). A plausible mistake (reciprocal instead of
division, round-half-away, 128 instead of 127, a transposed operand, a wrong
group index, a dropped scale) fails at least one test here.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads
from tests.exact import f32_value, quantize_exact, round_to_f32, round_half_even

G = 128


def _bf16(x):
    return workloads.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


# ------------------------------------------------------------ quantizer pins
def _exact_quant_rows(a_bits):
    """Per-token quantization from first principles (exact rationals)."""
    vals = workloads.bf16_bits_to_f32(a_bits)
    q = np.zeros(a_bits.shape, dtype=np.int64)
    s_out = []
    for m in range(a_bits.shape[0]):
        row = [f32_value(v) for v in vals[m]]
        amax = max(abs(v) for v in row)
        s = round_to_f32(amax / 127)
        s_out.append(s)
        for k, v in enumerate(row):
            q[m, k] = quantize_exact(v, s)
    return q, s_out


def test_quant_act_matches_exact_rationals():
    rng = np.random.default_rng(123)
    rows = [
        rng.standard_normal(96),
        rng.standard_normal(96) * 1e-3,
        np.concatenate([rng.standard_normal(95), [-37.5]]),      # negative amax
        rng.standard_t(3, 96) * 50,
        rng.uniform(-1, 1, 96) * 2.0 ** -128,                    # BF16 subnormal range
        np.linspace(-3, 3, 96),
    ]
    a = _bf16(np.stack(rows))
    qa, sa = oracle.quant_act(a)
    q_exp, s_exp = _exact_quant_rows(a)
    for m in range(a.shape[0]):
        assert f32_value(sa[m]) == s_exp[m], f"scale row {m}"
    np.testing.assert_array_equal(qa.astype(np.int64), q_exp)


def test_quant_act_ties_round_to_even():
    # amax = 127 gives s = 127/127 = 1 exactly, so x/s = x and the codes are
    # round-half-even of x: 2.5->2, 3.5->4, -2.5->-2, 0.5->0, 1.5->2, 126.5->126.
    row = [127.0, 2.5, 3.5, -2.5, 0.5, 1.5, 126.5, -126.5, -0.5, 5.5]
    qa, sa = oracle.quant_act(_bf16([row]))
    assert sa[0] == 1.0
    assert qa[0].tolist() == [127, 2, 4, -2, 0, 2, 126, -126, 0, 6]
    # amax = 254 gives s = 2 exactly: x = 5 -> 2.5 -> 2, x = 7 -> 3.5 -> 4, x = -3 -> -1.5 -> -2.
    qa, sa = oracle.quant_act(_bf16([[254.0, 5.0, 7.0, -3.0, 1.0]]))
    assert sa[0] == 2.0
    assert qa[0].tolist() == [127, 2, 4, -2, 0]


def test_quant_act_zero_row_and_negative_amax():
    qa, sa = oracle.quant_act(_bf16([[0.0] * 16, [-0.0] * 16]))
    assert sa.tolist() == [0.0, 0.0] and not qa.any()
    qa, sa = oracle.quant_act(_bf16([[1.0, -8.0, 2.0, 0.0]]))
    assert qa[0, 1] == -127 and sa[0] == np.float32(8.0) / np.float32(127.0)


def test_quant_act_invariants_on_workload_rows():
    spec = workloads.DENSE["decode_m32"]
    a = workloads.activations(spec, rows=np.arange(32))[:, :2048]
    a2 = workloads.activations(workloads.DENSE["stress"], rows=np.arange(16))[:, :2048]
    for bits in (a, a2):
        qa, sa = oracle.quant_act(bits)
        x = workloads.bf16_bits_to_f32(bits).astype(np.float64)
        s = sa.astype(np.float64)[:, None]
        # |q*s - x| <= s/2 * (1 + 2^-16): "within scale/2" plus the FP32 rounding of x/s.
        assert np.all(np.abs(qa * s - x) <= s / 2 * (1 + 2.0 ** -16))
        # the amax element maps to +-127 with its sign
        am = np.argmax(np.abs(x), axis=1)
        assert np.all(np.abs(qa[np.arange(len(am)), am]) == 127)
        assert np.all(np.sign(qa[np.arange(len(am)), am]) == np.sign(x[np.arange(len(am)), am]))
        # sign preserved, monotone within a row
        assert np.all((np.sign(qa) == np.sign(x)) | (qa == 0))
        for m in range(4):
            o = np.argsort(x[m], kind="stable")
            assert np.all(np.diff(qa[m, o].astype(np.int64)) >= 0)
        assert qa.min() >= -127


def test_quant_act_power_of_two_scaling():
    rng = np.random.default_rng(7)
    a = _bf16(rng.standard_normal((4, 256)))
    qa, sa = oracle.quant_act(a)
    x = workloads.bf16_bits_to_f32(a)
    qa2, sa2 = oracle.quant_act(_bf16(x * np.float32(2.0 ** 20)))
    np.testing.assert_array_equal(qa, qa2)
    np.testing.assert_array_equal(sa2, sa * np.float32(2.0 ** 20))


def test_quant_act_is_not_reciprocal_multiply():
    # Find a value where round(x * (1/s)) differs from round(x / s) and check
    # the oracle follows division (the page's round(x / scale)).
    rng = np.random.default_rng(3)
    found = 0
    for _ in range(200):
        x = _bf16(rng.standard_normal(512))
        vals = workloads.bf16_bits_to_f32(x)
        amax = np.float32(np.max(np.abs(vals)))
        s = np.float32(amax / np.float32(127.0))
        div = np.rint(vals / s)
        rec = np.rint(vals * (np.float32(1.0) / s))
        diff = np.nonzero(div != rec)[0]
        if diff.size:
            qa, _ = oracle.quant_act(x[None, :])
            assert np.all(qa[0, diff] == np.clip(div[diff], -127, 127))
            found += 1
            if found >= 3:
                break
    assert found >= 1


# ------------------------------------------------------ weight quantizer pins
def test_quant_weight_matches_exact_rationals():
    rng = np.random.default_rng(11)
    w = (rng.standard_normal((3, 256)) * 0.02).astype(np.float32)
    w[1, 128:] = 0.0                                      # an all-zero group
    w[2, 5] = -0.5                                        # negative amax in group 0
    qw, sw = oracle.quant_weight(w)
    assert sw.shape == (3, 2)
    for n in range(3):
        for g in range(2):
            grp = [f32_value(v) for v in w[n, g * G:(g + 1) * G]]
            s = round_to_f32(max(abs(v) for v in grp) / 127)
            assert f32_value(sw[n, g]) == s
            exp = [quantize_exact(v, s) for v in grp]
            assert qw[n, g * G:(g + 1) * G].tolist() == exp
    assert sw[1, 1] == 0.0 and not qw[1, 128:].any()
    assert qw[2, 5] == -127


def test_quant_weight_groups_are_independent():
    rng = np.random.default_rng(5)
    w = (rng.standard_normal((4, 512)) * 0.02).astype(np.float32)
    qw, sw = oracle.quant_weight(w)
    w2 = w.copy()
    w2[:, 256:384] *= np.float32(8.0)                     # only group 2 changes
    qw2, sw2 = oracle.quant_weight(w2)
    np.testing.assert_array_equal(np.delete(sw2, 2, axis=1), np.delete(sw, 2, axis=1))
    np.testing.assert_array_equal(sw2[:, 2], sw[:, 2] * np.float32(8.0))
    np.testing.assert_array_equal(qw2, qw)


# ------------------------------------------------------------ partial pins
def _numpy_partials(qa, qw):
    M, K = qa.shape
    N = qw.shape[0]
    a = qa.astype(np.int64).reshape(M, K // G, G)
    b = qw.astype(np.int64).reshape(N, K // G, G)
    return np.einsum("mgk,ngk->mng", a, b)


def test_partials_match_numpy_integer_matmul():
    rng = np.random.default_rng(1)
    qa = rng.integers(-127, 128, (5, 384), dtype=np.int8)
    qw = rng.integers(-127, 128, (7, 384), dtype=np.int8)
    P = oracle.group_partials(qa, qw)
    np.testing.assert_array_equal(P.astype(np.int64), _numpy_partials(qa, qw))


def test_partials_extremes():
    a = np.full((2, 256), 127, dtype=np.int8)
    b = np.full((3, 256), 127, dtype=np.int8)
    b[1] = -127
    P = oracle.group_partials(a, b)
    assert P[0, 0, 0] == 127 * 127 * 128 == 2064512
    assert P[1, 1, 1] == -2064512


def test_partials_one_hot_selects_transposed_index():
    # qa[m] = e_{k_m}: P[m, n, g] = qw[n, k_m] if k_m is in group g, else 0.
    rng = np.random.default_rng(2)
    K = 512
    ks = np.array([0, 127, 128, 300, 511])
    qa = np.zeros((len(ks), K), dtype=np.int8)
    qa[np.arange(len(ks)), ks] = 1
    qw = rng.integers(-127, 128, (6, K), dtype=np.int8)
    P = oracle.group_partials(qa, qw)
    for m, k in enumerate(ks):
        for n in range(6):
            exp = np.zeros(K // G, dtype=np.int64)
            exp[k // G] = qw[n, k]
            np.testing.assert_array_equal(P[m, n], exp)


# ------------------------------------------------------------ epilogue pins
def test_unit_scales_reproduce_integer_matmul():
    rng = np.random.default_rng(4)
    qa = rng.integers(-127, 128, (6, 1024), dtype=np.int8)
    qw = rng.integers(-127, 128, (9, 1024), dtype=np.int8)
    sa = np.ones(6, dtype=np.float32)
    sw = np.ones((9, 8), dtype=np.float32)
    y, T = oracle.gemm(qa, sa, qw, sw)
    exact = qa.astype(np.int64) @ qw.astype(np.int64).T
    np.testing.assert_array_equal(y, exact.astype(np.float64))
    np.testing.assert_array_equal(T, np.abs(_numpy_partials(qa, qw)).sum(-1).astype(np.float64))


def test_per_tensor_scale_special_case():
    # All group scales equal c: y = sa * c * sum_k qa*qw (bring-up order of
    # the page: per-tensor first, then per-group 128).
    rng = np.random.default_rng(6)
    qa = rng.integers(-127, 128, (4, 512), dtype=np.int8)
    qw = rng.integers(-127, 128, (5, 512), dtype=np.int8)
    sa = rng.random(4).astype(np.float32)
    c = np.float32(0.013)
    sw = np.full((5, 4), c, dtype=np.float32)
    y, T = oracle.gemm(qa, sa, qw, sw)
    exact = qa.astype(np.int64) @ qw.astype(np.int64).T
    ref = sa.astype(np.float64)[:, None] * float(c) * exact
    assert np.all(np.abs(y - ref) <= 1e-14 * T)


def test_gemm_matches_exact_rationals():
    rng = np.random.default_rng(8)
    qa = rng.integers(-127, 128, (3, 384), dtype=np.int8)
    qw = rng.integers(-127, 128, (4, 384), dtype=np.int8)
    sa = (rng.random(3) * 0.1).astype(np.float32)
    sw = (rng.random((4, 3)) * 1e-3).astype(np.float32)
    sw[2, 1] = -sw[2, 1]                                   # negative scale: sign must carry
    y, T = oracle.gemm(qa, sa, qw, sw)
    P = _numpy_partials(qa, qw)
    for m in range(3):
        for n in range(4):
            terms = [f32_value(sa[m]) * f32_value(sw[n, g]) * int(P[m, n, g]) for g in range(3)]
            ye = sum(terms)
            te = sum(abs(t) for t in terms)
            assert abs(Fraction(y[m, n]) - ye) <= Fraction(1, 10 ** 14) * te
            assert abs(Fraction(T[m, n]) - te) <= Fraction(1, 10 ** 14) * te


def test_gemm_one_hot_picks_group_scale():
    K = 512
    qa = np.zeros((2, K), dtype=np.int8)
    qa[0, 130] = 1                                        # group 1
    qa[1, 511] = -3                                       # group 3
    rng = np.random.default_rng(9)
    qw = rng.integers(-127, 128, (5, K), dtype=np.int8)
    sw = rng.random((5, 4)).astype(np.float32)
    sa = np.array([1.0, 0.5], dtype=np.float32)
    y, _ = oracle.gemm(qa, sa, qw, sw)
    np.testing.assert_array_equal(y[0], sw[:, 1].astype(np.float64) * qw[:, 130])
    np.testing.assert_array_equal(y[1], 0.5 * -3 * sw[:, 3].astype(np.float64) * qw[:, 511])


def test_gemm_linear_in_group_scale():
    rng = np.random.default_rng(10)
    qa = rng.integers(-127, 128, (3, 256), dtype=np.int8)
    qw = rng.integers(-127, 128, (4, 256), dtype=np.int8)
    sa = rng.random(3).astype(np.float32)
    sw = rng.random((4, 2)).astype(np.float32)
    y1, T = oracle.gemm(qa, sa, qw, sw)
    sw2 = sw.copy()
    sw2[:, 1] *= 2
    y2, _ = oracle.gemm(qa, sa, qw, sw2)
    P = _numpy_partials(qa, qw)
    delta = sa.astype(np.float64)[:, None] * sw[:, 1].astype(np.float64)[None, :] * P[:, :, 1]
    assert np.all(np.abs((y2 - y1) - delta) <= 1e-14 * (T + np.abs(delta)))


def test_gemm_matches_numpy_on_workload_slice():
    spec = workloads.DENSE["tiny"]
    a = workloads.activations(spec)
    w = workloads.weights(spec, rows=np.arange(64))
    qa, sa = oracle.quant_act(a)
    qw, sw = oracle.quant_weight(w)
    y, T = oracle.gemm(qa, sa, qw, sw)
    P = _numpy_partials(qa, qw).astype(np.float64)
    ref = np.einsum("mng,m,ng->mn", P, sa.astype(np.float64), sw.astype(np.float64))
    assert np.all(np.abs(y - ref) <= 1e-13 * T)
    # quantization quality sanity: close to the unquantized product
    x = workloads.bf16_bits_to_f32(a).astype(np.float64)
    yf = x @ w.astype(np.float64).T
    rel = np.linalg.norm(y - yf) / np.linalg.norm(yf)
    assert rel < 0.05


# ------------------------------------------------------------- grouped pins
def test_grouped_matches_numpy_by_row_expert():
    rng = np.random.default_rng(12)
    E, N, K, R = 5, 6, 256, 23
    off = np.array([0, 4, 4, 15, 15, 23], dtype=np.int32)   # experts 1 and 3 empty
    qa = rng.integers(-127, 128, (R, K), dtype=np.int8)
    sa = rng.random(R).astype(np.float32)
    qw = rng.integers(-127, 128, (E, N, K), dtype=np.int8)
    sw = rng.random((E, N, K // G)).astype(np.float32)
    y, T = oracle.grouped_gemm(qa, sa, off, qw, sw)
    expert = np.searchsorted(off, np.arange(R), side="right") - 1
    for r in range(R):
        e = expert[r]
        P = _numpy_partials(qa[r:r + 1], qw[e])[0].astype(np.float64)   # [N, G]
        ref = (float(sa[r]) * sw[e].astype(np.float64) * P).sum(-1)
        assert np.all(np.abs(y[r] - ref) <= 1e-13 * T[r])


def test_grouped_leaves_uncovered_rows_untouched():
    rng = np.random.default_rng(13)
    E, N, K, R = 3, 4, 128, 10
    off = np.array([2, 5, 5, 8], dtype=np.int32)            # rows 0,1,8,9 uncovered
    qa = rng.integers(-127, 128, (R, K), dtype=np.int8)
    sa = rng.random(R).astype(np.float32)
    qw = rng.integers(-127, 128, (E, N, K), dtype=np.int8)
    sw = rng.random((E, N, 1)).astype(np.float32)
    y, _ = oracle.grouped_gemm(qa, sa, off, qw, sw)
    assert np.isnan(y[[0, 1, 8, 9]]).all() and not np.isnan(y[2:8]).any()


def test_grouped_single_expert_equals_dense():
    rng = np.random.default_rng(14)
    qa = rng.integers(-127, 128, (9, 256), dtype=np.int8)
    sa = rng.random(9).astype(np.float32)
    qw = rng.integers(-127, 128, (1, 5, 256), dtype=np.int8)
    sw = rng.random((1, 5, 2)).astype(np.float32)
    y, _ = oracle.grouped_gemm(qa, sa, np.array([0, 9], np.int32), qw, sw)
    P = _numpy_partials(qa, qw[0]).astype(np.float64)
    ref = np.einsum("mng,m,ng->mn", P, sa.astype(np.float64), sw[0].astype(np.float64))
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=0)


# ---------------------------------------------------------------- BF16 pins
def test_bf16_round_known_values():
    one = 1.0
    cases = {
        1.0: 0x3F80,
        one + 2 ** -8: 0x3F80,                 # tie -> even (1.0)
        one + 3 * 2 ** -8: 0x3F82,             # tie between 0x3F81 and 0x3F82 -> even
        one + 2 ** -8 + 2 ** -30: 0x3F81,      # just above the tie
        -2.0: 0xC000,
        2.0 ** -133: 0x0001,                   # smallest subnormal
        2.0 ** -134: 0x0000,                   # tie with zero -> even (0)
        3 * 2.0 ** -135: 0x0001,               # 0.75 quantum of 2^-133 -> 1 quantum
        3 * 2.0 ** -134: 0x0002,               # 1.5 quanta -> tie -> even (2 quanta)
        3.0e38: 0x7F62,
        3.5e38: 0x7F80,                        # overflows to +inf
    }
    got = oracle.bf16_round(np.array(list(cases.keys())))
    assert [int(g) for g in got] == list(cases.values())


def test_bf16_round_is_nearest_even_among_neighbours():
    rng = np.random.default_rng(15)
    v = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.uniform(-30, 30, 2000),
                        (rng.integers(1, 1 << 20, 500) + 0.5) * 2.0 ** -12])
    h = oracle.bf16_round(v)
    for x, hb in zip(v, h):
        hb = int(hb)
        xv = Fraction(abs(float(x)))
        mag = hb & 0x7FFF
        def val(b):
            return Fraction(oracle.bf16_to_float(np.array([b], np.uint16))[0])
        d0 = abs(xv - val(mag))
        d_lo = abs(xv - val(mag - 1)) if mag > 0 else None
        d_hi = abs(xv - val(mag + 1))
        assert d_lo is None or d0 <= d_lo
        assert d0 <= d_hi
        if (d_lo is not None and d0 == d_lo) or d0 == d_hi:
            assert mag % 2 == 0
        assert (hb >> 15) == (1 if x < 0 else 0)


def test_bf16_round_agrees_with_torch_for_f32_inputs():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(16)
    v32 = (rng.standard_normal(10000) * 10.0 ** rng.uniform(-20, 20, 10000)).astype(np.float32)
    h = oracle.bf16_round(v32.astype(np.float64))
    t = torch.from_numpy(v32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(h, t)
