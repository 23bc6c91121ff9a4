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

/* ======================================================================
 * MoE expert FFN: the steps either side of the two grouped GEMMs
 * ("Deploying Hunyuan 770B in INT8 on domestic accelerators", §4.4: a
 * global count of tokens per destination expert is staged first, then the
 * tokens are transferred in bulk; §4.1 operator table: SwiGLU next to the
 * INT8 GEMMs; §3.1: every INT8 GEMM input is quantized per token,
 * dynamically, so the gate_up output is re-quantized before the down GEMM).
 * ====================================================================== */

/* Routing: ids [T*k] holds the k experts of each token (flattened in (t, j)
 * order). Entries whose id lies outside [0, E) are not routed (row_of = -1).
 * counts per expert -> offsets [E+1] (exclusive prefix sum); each routed
 * entry i gets row row_of[i] = offsets[e] + (number of earlier entries with
 * the same expert), so rows are sorted by expert and, within an expert, by
 * flattened index (token order). token_of_row[r] = i / k and pair_of_row[r]
 * = i for the R = offsets[E] routed rows; rows >= R are set to -1. */
void oracle_moe_route(const int32_t *ids, int64_t T, int64_t k, int64_t E, int32_t *offsets,
                      int32_t *row_of, int32_t *token_of_row, int32_t *pair_of_row) {
    const int64_t n = T * k;
    for (int64_t e = 0; e <= E; e++) offsets[e] = 0;
    for (int64_t i = 0; i < n; i++)
        if (ids[i] >= 0 && ids[i] < E) offsets[ids[i] + 1] += 1;   /* histogram */
    for (int64_t e = 0; e < E; e++) offsets[e + 1] += offsets[e];  /* prefix sum */
    for (int64_t r = 0; r < n; r++) {
        token_of_row[r] = -1;
        pair_of_row[r] = -1;
    }
    for (int64_t e = 0; e < E; e++) {
        int32_t fill = offsets[e];
        for (int64_t i = 0; i < n; i++) {
            if (ids[i] != e) continue;
            row_of[i] = fill;
            token_of_row[fill] = (int32_t)(i / k);
            pair_of_row[fill] = (int32_t)i;
            fill++;
        }
    }
    for (int64_t i = 0; i < n; i++)
        if (ids[i] < 0 || ids[i] >= E) row_of[i] = -1;
}

/* 2^n as a binary32 number, -126 <= n <= 127 (exact). */
static float pow2_f32(int n) {
    uint32_t u = (uint32_t)(n + 127) << 23;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* e^x in binary32 (the SwiGLU's exponential), by the textbook method of
 * Cody and Waite: x is clamped to [-87, 88] (where e^x and e^-x stay normal
 * binary32 numbers), n = round-to-nearest-even(x * log2(e)), the reduced
 * argument r = x - n*ln2 is formed with ln2 split into a 15-bit head and a
 * tail (so n*head is exact), e^r (|r| <= 0.35) is the Taylor series of degree
 * 7 evaluated by Horner's rule, and the result is scaled by 2^n. Every step is
 * one separately rounded binary32 operation (no fused multiply-add), so any
 * implementation of these steps produces the same bits. */
float oracle_exp_f32(float x) {
    if (x > 88.0f) x = 88.0f;
    if (x < -87.0f) x = -87.0f;
    const float log2e = 1.44269502163f;
    const float ln2_hi = 0.693145751953125f;        /* 0x3F317200 */
    const float ln2_lo = 1.42860676533018e-06f;     /* ln2 - ln2_hi */
    float t = x * log2e;
    float n = nearbyintf(t);
    float r = x - n * ln2_hi;
    r = r - n * ln2_lo;
    float p = 1.0f / 5040.0f;                       /* 1/7! */
    p = p * r + 1.0f / 720.0f;
    p = p * r + 1.0f / 120.0f;
    p = p * r + 1.0f / 24.0f;
    p = p * r + 1.0f / 6.0f;
    p = p * r + 0.5f;
    p = p * r + 1.0f;
    p = p * r + 1.0f;
    return p * pow2_f32((int)n);
}

/* silu(g) = g / (1 + e^-g) in binary32 with IEEE division. */
float oracle_silu_f32(float g) {
    float e = oracle_exp_f32(-g);
    float d = 1.0f + e;
    return g / d;
}

/* SwiGLU of the gate_up output followed by per-token quantization of the
 * result for the down GEMM. U [R, 2I] FP32: gate in columns [0, I), up in
 * [I, 2I). h = silu(gate) * up (binary32), then per row s = amax|h| / 127
 * and q = clamp(round-half-even(h / s)) as in oracle_quant_act. Rows >= nrows
 * (the routed rows) are left untouched. qh [R, I] int8, sh [R] float. */
void oracle_swiglu_quant(const float *U, int64_t nrows, int64_t I, int8_t *qh, float *sh) {
    fesetround(FE_TONEAREST);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < nrows; r++) {
        const float *g = U + r * 2 * I;
        const float *u = g + I;
        float amax = 0.0f;
        for (int64_t i = 0; i < I; i++) {
            float h = oracle_silu_f32(g[i]) * u[i];
            if (fabsf(h) > amax) amax = fabsf(h);
        }
        float s = amax / 127.0f;
        sh[r] = s;
        for (int64_t i = 0; i < I; i++) {
            float h = oracle_silu_f32(g[i]) * u[i];
            qh[r * I + i] = quantize_value(h, s);
        }
    }
}

/* Weighted un-permute: Y[t, n] = sum_j w[t*k+j] * D[row_of[t*k+j], n] over the
 * routed entries of token t (FP64; unrouted entries contribute nothing).
 * D [R, H] double, Y [T, H] double. */
void oracle_moe_unpermute(const double *D, const int32_t *row_of, const float *w, int64_t T,
                          int64_t k, int64_t H, double *Y) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; t++) {
        for (int64_t n = 0; n < H; n++) {
            double acc = 0.0;
            for (int64_t j = 0; j < k; j++) {
                int32_t r = row_of[t * k + j];
                if (r < 0) continue;
                acc += (double)w[t * k + j] * D[(int64_t)r * H + n];
            }
            Y[t * H + n] = acc;
        }
    }
}

/* Element-wise array forms of the two functions above (for the tests). */
void oracle_exp_f32_n(const float *x, int64_t n, float *out) {
    for (int64_t i = 0; i < n; i++) out[i] = oracle_exp_f32(x[i]);
}

void oracle_silu_f32_n(const float *x, int64_t n, float *out) {
    for (int64_t i = 0; i < n; i++) out[i] = oracle_silu_f32(x[i]);
}

/* ======================================================================
 * Scale formats of the DeepSeek-V4 checkpoints ("Running DeepSeek-V4-Flash-
 * Vision on 4xA800", §一: weights in [128, 128] blocks with power-of-two
 * UE8M0 scales), applied to INT8 codes.
 * ====================================================================== */

/* The UE8M0 (power-of-two) scale of a group with the given amax: the
 * smallest 2^e >= amax / 127 (compared exactly), e clamped to [-127, 127];
 * an all-zero group gets 2^-127. The division x / 2^e is then exact, so the
 * codes are round-half-even(x * 2^-e), |code| <= 127. */
static float pow2_scale(float amax) {
    int e = -127;
    if (amax > 0.0f) {
        int ex;
        (void)frexp((double)amax / 127.0, &ex);   /* amax/127 in [2^(ex-1), 2^ex) approx */
        e = ex - 2;
        while ((double)amax > 127.0 * ldexp(1.0, e)) e++;          /* exact comparisons */
        while (e > -127 && (double)amax <= 127.0 * ldexp(1.0, e - 1)) e--;
        if (e < -127) e = -127;
        if (e > 127) e = 127;
    }
    return (float)ldexp(1.0, e);
}

/* Per-token activation quantization with UE8M0 scales (the amax mode is
 * oracle_quant_act): s_m = pow2_scale(amax_m), qa = rne(a / s_m). */
void oracle_quant_act_pow2(const uint16_t *a, int64_t M, int64_t K, int64_t lda, int8_t *qa,
                           int64_t ldq, float *sa) {
    fesetround(FE_TONEAREST);
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; m++) {
        float amax = 0.0f;
        for (int64_t k = 0; k < K; k++) {
            float x = fabsf(bf16_bits_to_float(a[m * lda + k]));
            if (x > amax) amax = x;
        }
        float s = pow2_scale(amax);
        sa[m] = s;
        for (int64_t k = 0; k < K; k++)
            qa[m * ldq + k] = quantize_value(bf16_bits_to_float(a[m * lda + k]), s);
    }
}

/* Weight quantization over blocks of block_rows rows x 128 K (block_rows 1:
 * the per-row groups of oracle_quant_weight; 128: the [128, 128] blocks),
 * scale amax / 127 (pow2 == 0) or UE8M0 (pow2 != 0).
 * w [N, K]; qw [N, K]; sw [ceil(N / block_rows), K / 128]. */
void oracle_quant_weight_blocks(const float *w, int64_t N, int64_t K, int64_t block_rows,
                                int pow2, int8_t *qw, float *sw) {
    const int64_t G = K / W8A8_ORACLE_GROUP;
    const int64_t NB = (N + block_rows - 1) / block_rows;
    fesetround(FE_TONEAREST);
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < NB; b++) {
        const int64_t n0 = b * block_rows;
        const int64_t n1 = n0 + block_rows < N ? n0 + block_rows : N;
        for (int64_t g = 0; g < G; g++) {
            float amax = 0.0f;
            for (int64_t n = n0; n < n1; n++)
                for (int64_t j = 0; j < W8A8_ORACLE_GROUP; j++) {
                    float x = fabsf(w[n * K + g * W8A8_ORACLE_GROUP + j]);
                    if (x > amax) amax = x;
                }
            float s = pow2 ? pow2_scale(amax) : amax / 127.0f;
            sw[b * G + g] = s;
            for (int64_t n = n0; n < n1; n++)
                for (int64_t j = 0; j < W8A8_ORACLE_GROUP; j++) {
                    const int64_t i = n * K + g * W8A8_ORACLE_GROUP + j;
                    qw[i] = quantize_value(w[i], s);
                }
        }
    }
}

/* The group-scaled GEMM with one weight scale per block of block_rows output
 * rows: y[m, n] = sum_g sa[m] * sw[n / block_rows, g] * P[m, n, g] (FP64),
 * T = sum_g |...|. */
void oracle_gemm_blocks(const int8_t *qa, const float *sa, const int8_t *qw, const float *sw,
                        int64_t M, int64_t N, int64_t K, int64_t block_rows, double *y,
                        double *T) {
    const int64_t G = K / W8A8_ORACLE_GROUP;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; m++) {
        for (int64_t n = 0; n < N; n++) {
            double ysum = 0.0, tsum = 0.0;
            for (int64_t g = 0; g < G; g++) {
                int32_t p = group_partial(qa + m * K, qw + n * K, g);
                double term = (double)sa[m] * (double)sw[(n / block_rows) * G + g] * (double)p;
                ysum += term;
                tsum += fabs(term);
            }
            y[m * N + n] = ysum;
            if (T) T[m * N + n] = tsum;
        }
    }
}

/* Weight-only INT8 with BF16 activations (the "WNA16" reading of the MoE
 * runner on the same page, §二): y[m, n] = sum_g sw[n / block_rows, g] *
 * sum_{k in g} a[m, k] * qw[n, k] (FP64; the products of a BF16 value and an
 * integer of at most 7 bits are exact), T = sum_g |sw| * sum_k |a * qw|. */
void oracle_w8a16_gemm(const uint16_t *a, const int8_t *qw, const float *sw, int64_t M, int64_t N,
                       int64_t K, int64_t block_rows, double *y, double *T) {
    const int64_t G = K / W8A8_ORACLE_GROUP;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; m++) {
        for (int64_t n = 0; n < N; n++) {
            double ysum = 0.0, tsum = 0.0;
            for (int64_t g = 0; g < G; g++) {
                double ps = 0.0, pa = 0.0;
                for (int64_t j = 0; j < W8A8_ORACLE_GROUP; j++) {
                    const int64_t k = g * W8A8_ORACLE_GROUP + j;
                    double prod = (double)bf16_bits_to_float(a[m * K + k]) * (double)qw[n * K + k];
                    ps += prod;
                    pa += fabs(prod);
                }
                const double s = (double)sw[(n / block_rows) * G + g];
                ysum += s * ps;
                tsum += fabs(s) * pa;
            }
            y[m * N + n] = ysum;
            if (T) T[m * N + n] = tsum;
        }
    }
}

/* ======================================================================
 * INT8 KV cache with per-token dynamic scales, dequantized inside attention
 * ("Deploying Hunyuan 770B in INT8 on domestic accelerators", §3.4: one
 * scale per key/value vector, computed when the vector is written; the
 * attention kernel reads the INT8 data and applies the scales itself; §2.2:
 * the cache is 2 x layers x kv_heads x head_dim x seq_len x batch elements).
 * The quantization of one K or V vector is oracle_quant_act on a row of
 * head_dim values.
 * ====================================================================== */

/* Dequantized vectors: out[i, d] = q[i, d] * s[i] (exact in FP64). */
void oracle_kv_dequant(const int8_t *q, const float *s, int64_t n, int64_t D, double *out) {
    for (int64_t i = 0; i < n; i++)
        for (int64_t d = 0; d < D; d++) out[i * D + d] = (double)q[i * D + d] * (double)s[i];
}

/* Decode attention of one query token per sequence, grouped-query: query
 * head hq reads kv head hq / (Hq / Hkv). K, V [B, Hkv, S_max, D] (FP64
 * values), lens [B] valid positions, q [B, Hq, D] BF16 bit patterns:
 *   s_j = scale * sum_d q_d k_{j,d},  p_j = exp(s_j - max_j s_j),
 *   out_d = sum_j p_j v_{j,d} / sum_j p_j   over j < lens[b]   (FP64),
 * and T_d = sum_j p_j |v_{j,d}| / sum_j p_j (the magnitude the error of an
 * implementation is measured against). lens[b] == 0 gives 0. */
void oracle_attention_decode(const uint16_t *q, const double *K, const double *V,
                             const int32_t *lens, int64_t B, int64_t Hq, int64_t Hkv,
                             int64_t S_max, int64_t D, double scale, double *out, double *T) {
    const int64_t G = Hq / Hkv;
#pragma omp parallel for schedule(static)
    for (int64_t bh = 0; bh < B * Hq; bh++) {
        const int64_t b = bh / Hq, hq = bh % Hq, h = hq / G;
        const int64_t L = lens[b] < 0 ? 0 : (lens[b] > S_max ? S_max : lens[b]);
        const uint16_t *qv = q + bh * D;
        const double *Kb = K + (b * Hkv + h) * S_max * D;
        const double *Vb = V + (b * Hkv + h) * S_max * D;
        double *o = out + bh * D;
        double *t = T + bh * D;
        for (int64_t d = 0; d < D; d++) o[d] = t[d] = 0.0;
        if (L == 0) continue;
        double m = -INFINITY;
        for (int64_t j = 0; j < L; j++) {
            double sj = 0.0;
            for (int64_t d = 0; d < D; d++) sj += (double)bf16_bits_to_float(qv[d]) * Kb[j * D + d];
            sj *= scale;
            if (sj > m) m = sj;
        }
        double l = 0.0;
        for (int64_t j = 0; j < L; j++) {
            double sj = 0.0;
            for (int64_t d = 0; d < D; d++) sj += (double)bf16_bits_to_float(qv[d]) * Kb[j * D + d];
            const double pj = exp(sj * scale - m);
            l += pj;
            for (int64_t d = 0; d < D; d++) {
                o[d] += pj * Vb[j * D + d];
                t[d] += pj * fabs(Vb[j * D + d]);
            }
        }
        for (int64_t d = 0; d < D; d++) {
            o[d] /= l;
            t[d] /= l;
        }
    }
}

/* ------------------------------------------------------------------------
 * RMSNorm in front of the per-token quantizer ("Deploying Hunyuan 770B in
 * INT8 on domestic accelerators", §4.1 operator table: RMSNorm runs in high
 * precision beside the INT8 GEMMs, whose activations §3.1 quantizes per
 * token). The definition, in FP64 from the BF16 inputs:
 *   y[m, k] = x[m, k] / sqrt(mean_k(x[m, k]^2) + eps) * gamma[k].
 * The BF16 rounding of y and the quantization of the rounded rows are the
 * existing oracle functions (oracle_bf16_round, oracle_quant_act). */
void oracle_rmsnorm(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, const uint16_t *gamma,
                    double eps, double *y) {
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        const uint16_t *row = x + m * ldx;
        double ss = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double v = (double)bf16_bits_to_float(row[k]);
            ss += v * v;   /* exact: a BF16 square has at most 16 significant bits */
        }
        const double r = sqrt(ss / (double)K + eps);
        for (int64_t k = 0; k < K; ++k)
            y[m * K + k] = (double)bf16_bits_to_float(row[k]) / r *
                           (double)bf16_bits_to_float(gamma[k]);
    }
}
