/*
 * CPU oracle for the W8A8 group-scaled quantized linear layer.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this library. It shares no code with
 * the CUDA library and is written to be checked against the source text by
 * eye: plain loops, no blocking, no fusion, no reordering.
 *
 * Source of the method: "Deploying Hunyuan 770B in INT8 on domestic
 * accelerators (FlagOS Hy4 preview 5)", §3.1 (quantization granularity):
 *   - weights are quantized in groups of 128 elements, one scale per group;
 *   - activations are quantized per token, dynamically, with a scale computed
 *     from the current token's range at every call;
 *   - quantization is round(x / scale);
 *   - each MatMul multiplies INT8 by INT8 into an INT32 accumulator and only
 *     at the end multiplies the FP32 scales back in.
 * MoE grouping: same page §1.3 (only some experts are active per token) and
 * §4.4 (tokens are sent to the experts chosen by the router).
 *
 * Readings where the page is silent (each is listed with its reason in the
 * design notes):
 *   - the weight group runs along K within one output row n;
 *   - symmetric scale s = amax / 127 (no zero point), FP32 IEEE division;
 *   - round() is round-to-nearest-even, then clamped to [-127, 127];
 *   - amax == 0 gives s = 0 and all codes 0;
 *   - the scales are applied once per 128-group partial (weight scale) and once
 *     per output (token scale); the oracle evaluates the sum in FP64 and also
 *     returns T = sum over groups of |term| for the error bound.
 *
 * Parity pins: every function here is pinned by the CPU tests against exact
 * rational arithmetic, closed forms and invariants (see tests/test_oracle_pins.py).
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fopenmp -shared -fPIC
 * (no fast-math: IEEE division and round-to-nearest-even are required).
 */
#include <fenv.h>
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define W8A8_ORACLE_GROUP 128

static float bf16_bits_to_float(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* round(x / s) with round-to-nearest-even, clamped to the symmetric range.
 * Hunyuan-770B page §3.1 ("quantization is round(x / scale)"). */
static int8_t quantize_value(float x, float s) {
    if (s == 0.0f) return 0;
    float r = x / s;            /* IEEE binary32 division, round to nearest */
    float q = nearbyintf(r);    /* ties to even under the default rounding mode */
    if (q > 127.0f) q = 127.0f;
    if (q < -127.0f) q = -127.0f;
    return (int8_t)q;
}

int oracle_group_size(void) { return W8A8_ORACLE_GROUP; }

void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Per-token dynamic activation quantization (Hunyuan-770B page §3.1:
 * "activations are quantized per token, dynamically").
 * a: BF16 bit patterns [M, lda]; qa: int8 [M, ldq]; sa: float [M]. */
void oracle_quant_act(const uint16_t *a, int64_t M, int64_t K, int64_t lda,
                      int8_t *qa, int64_t ldq, float *sa) {
    fesetround(FE_TONEAREST);
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; m++) {
        float amax = 0.0f;
        for (int64_t k = 0; k < K; k++) {
            float x = fabsf(bf16_bits_to_float(a[m * lda + k]));
            if (x > amax) amax = x;
        }
        float s = amax / 127.0f;
        sa[m] = s;
        for (int64_t k = 0; k < K; k++)
            qa[m * ldq + k] = quantize_value(bf16_bits_to_float(a[m * lda + k]), s);
    }
}

/* Per-group-128 weight quantization along K (Hunyuan-770B page §3.1:
 * "weights in groups of 128 elements, each group with its own scale").
 * w: float [N, K]; qw: int8 [N, K]; sw: float [N, K/128]. */
void oracle_quant_weight(const float *w, int64_t N, int64_t K, int8_t *qw, float *sw) {
    const int64_t G = K / W8A8_ORACLE_GROUP;
    fesetround(FE_TONEAREST);
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; n++) {
        for (int64_t g = 0; g < G; g++) {
            const float *src = w + n * K + g * W8A8_ORACLE_GROUP;
            float amax = 0.0f;
            for (int64_t j = 0; j < W8A8_ORACLE_GROUP; j++) {
                float x = fabsf(src[j]);
                if (x > amax) amax = x;
            }
            float s = amax / 127.0f;
            sw[n * G + g] = s;
            for (int64_t j = 0; j < W8A8_ORACLE_GROUP; j++)
                qw[n * K + g * W8A8_ORACLE_GROUP + j] = quantize_value(src[j], s);
        }
    }
}

/* Exact INT32 partial of one 128-wide K group: P = sum_k qa[m,k] * qw[n,k]
 * (Hunyuan-770B page §3.1: INT8 multiply-accumulate into an INT32
 * accumulator). */
static int32_t group_partial(const int8_t *qa_row, const int8_t *qw_row, int64_t g) {
    int32_t acc = 0;
    for (int64_t j = 0; j < W8A8_ORACLE_GROUP; j++) {
        int64_t k = g * W8A8_ORACLE_GROUP + j;
        acc += (int32_t)qa_row[k] * (int32_t)qw_row[k];
    }
    return acc;
}

/* All group partials P[m, n, g], int32 [M, N, K/128]. */
void oracle_group_partials(const int8_t *qa, const int8_t *qw, int64_t M, int64_t N,
                           int64_t K, int32_t *P) {
    const int64_t G = K / W8A8_ORACLE_GROUP;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; m++)
        for (int64_t n = 0; n < N; n++)
            for (int64_t g = 0; g < G; g++)
                P[(m * N + n) * G + g] = group_partial(qa + m * K, qw + n * K, g);
}

/* y[m, n] = sum_g sa[m] * sw[n, g] * P[m, n, g] in FP64, and
 * T[m, n] = sum_g |sa[m] * sw[n, g] * P[m, n, g]| (Hunyuan-770B page §3.1:
 * the FP32 scales are multiplied back only at the end of the INT32
 * accumulation). qa [M,K], sa [M], qw [N,K], sw [N,K/128]; y, T [M,N]. */
void oracle_gemm(const int8_t *qa, const float *sa, const int8_t *qw, const float *sw,
                 int64_t M, int64_t N, int64_t K, double *y, double *T) {
    const int64_t G = K / W8A8_ORACLE_GROUP;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; m++) {
        for (int64_t n = 0; n < N; n++) {
            double ysum = 0.0, tsum = 0.0;
            for (int64_t g = 0; g < G; g++) {
                int32_t p = group_partial(qa + m * K, qw + n * K, g);
                double term = (double)sa[m] * (double)sw[n * G + g] * (double)p;
                ysum += term;
                tsum += fabs(term);
            }
            y[m * N + n] = ysum;
            if (T) T[m * N + n] = tsum;
        }
    }
}

/* MoE expert-grouped GEMM: rows [off[e], off[e+1]) of qa use expert e's
 * weights qw[e] [N,K] and scales sw[e] [N,K/128] (Hunyuan-770B page §1.3 and
 * §4.4: each token is processed by the experts the router picked). Rows not
 * covered by any segment are left untouched. */
void oracle_grouped_gemm(const int8_t *qa, const float *sa, const int32_t *offsets,
                         const int8_t *qw, const float *sw, int64_t R, int64_t E,
                         int64_t N, int64_t K, double *y, double *T) {
    const int64_t G = K / W8A8_ORACLE_GROUP;
    for (int64_t e = 0; e < E; e++) {
        int64_t lo = offsets[e], hi = offsets[e + 1];
        if (lo < 0) lo = 0;
        if (hi > R) hi = R;
        if (hi <= lo) continue;
        oracle_gemm(qa + lo * K, sa + lo, qw + e * N * K, sw + e * N * G, hi - lo, N, K,
                    y + lo * N, T ? T + lo * N : 0);
    }
}

/* Correctly rounded (ties-to-even) conversion of a finite double to the
 * bfloat16 bit pattern: the BF16 output format of the layer. */
uint16_t oracle_bf16_from_double(double v) {
    if (v == 0.0) return signbit(v) ? 0x8000u : 0x0000u;
    const uint16_t sign = signbit(v) ? 0x8000u : 0x0000u;
    double av = fabs(v);
    int e;
    (void)frexp(av, &e);                 /* av = f * 2^e, f in [0.5, 1) */
    int qexp = e - 8;                    /* 8 significant bits */
    if (qexp < -133) qexp = -133;        /* subnormal spacing 2^-133 */
    double m = ldexp(av, -qexp);         /* exact scaling */
    double mr = nearbyint(m);            /* ties to even */
    double r = ldexp(mr, qexp);
    if (r >= 0x1p128) return sign | 0x7F80u;  /* rounds to infinity */
    float f = (float)r;                  /* exact: <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)(u >> 16);
}

void oracle_bf16_round(const double *v, int64_t n, uint16_t *out) {
    fesetround(FE_TONEAREST);
    for (int64_t i = 0; i < n; i++) out[i] = oracle_bf16_from_double(v[i]);
}
