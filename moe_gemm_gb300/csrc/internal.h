// Internal declarations shared by the translation units of libw8a8 (host side).
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace w8a8 {

cudaError_t launch_quant_act(const uint16_t *a, int64_t M, int64_t K, int64_t lda, int8_t *qa,
                             int64_t ldq, float *sa, cudaStream_t stream);

// The same codes as launch_quant_act, written as fp16 (row stride K) into
// x16 for the tensor-core GEMM, which then needs no staging kernel; also
// zeroes n_cnt split counters at cnt (if not null) for that GEMM.
cudaError_t launch_quant_act_f16(const uint16_t *a, int64_t M, int64_t K, int64_t lda, void *x16,
                                 float *sa, int *cnt, int n_cnt, cudaStream_t stream);

cudaError_t launch_quant_weight(const float *w, int64_t N, int64_t K, int8_t *qw, float *sw,
                                cudaStream_t stream);

// Scale-format variants: activations with power-of-two (UE8M0) scales
// (int8 codes, or fp16 codes into a GEMM workspace), and weights over
// [block_rows x 128] blocks (block_rows 1 or 128) with amax/127 or
// power-of-two scales, sw [ceil(N / block_rows), K / 128].
cudaError_t launch_quant_act_ex(const uint16_t *a, int64_t M, int64_t K, int64_t lda, int8_t *qa,
                                int64_t ldq, float *sa, bool pow2, cudaStream_t stream);
cudaError_t launch_quant_act_f16_ex(const uint16_t *a, int64_t M, int64_t K, int64_t lda,
                                    void *x16, float *sa, int *cnt, int n_cnt, bool pow2,
                                    cudaStream_t stream);
cudaError_t launch_quant_weight_blocks(const float *w, int64_t N, int64_t K, int block_rows,
                                       bool pow2, int8_t *qw, float *sw, cudaStream_t stream);

// Per-token quantization with a row gather: output row r (row stride K)
// quantizes input row src_rows[r] of a (row stride lda); rows whose entry is
// negative are skipped. Codes as fp16 (f16) or int8.
cudaError_t launch_quant_act_rows(const uint16_t *a, int64_t rows, int64_t K, int64_t lda,
                                  const int32_t *src_rows, void *out, bool f16, float *sa,
                                  cudaStream_t stream);

// MoE expert FFN steps (moe.cu).
constexpr int kMoeMaxTopK = 64;
constexpr int64_t kSwigluMaxI = 8192;
cudaError_t launch_moe_route(const int32_t *ids, int64_t T, int64_t k, int64_t E, int32_t *offsets,
                             int32_t *row_of, int32_t *token_of_row, int32_t *pair_of_row,
                             cudaStream_t stream);
// out_kind: 0 int8 codes, 1 fp16 codes (+ scales sh), 2 h itself (FP32)
cudaError_t launch_swiglu_quant(const float *U, int64_t rows, int64_t I, const int32_t *offsets,
                                int64_t E, void *out, int out_kind, float *sh,
                                cudaStream_t stream);
cudaError_t launch_moe_unpermute(const float *D, const int32_t *row_of, const float *w, int64_t T,
                                 int64_t k, int64_t H, void *y, bool out_fp32,
                                 cudaStream_t stream);

// int8 codes [rows, K] (row stride ldq) -> fp16 codes [rows, K] in `out`;
// also zeroes n_cnt split-tile counters at cnt (if not null) for the GEMM
// launched after it.
cudaError_t launch_widen_codes(const int8_t *q, int64_t rows, int64_t K, int64_t ldq, void *out,
                               int num_sms, cudaStream_t stream, int *cnt = nullptr,
                               int n_cnt = 0);

struct GemmProblem {
    const int8_t *qa;         // [R, K] int8 activation codes
    const float *sa;          // [R]
    const float *sw;          // [E*N, G]
    const int8_t *qw;         // [E*N, K]
    const void *x16;          // [R, K] fp16 copy of the int8 activation codes (staging)
    const int32_t *offsets;   // [E+1] device, or nullptr for one dense segment [0, R)
    void *y;                  // [R, N]
    int32_t *debug_partials;  // nullable [R, N, G]
    int64_t R, E, N, K;
    bool out_fp32;
    // Dense calls of <= kGemvMaxTokens rows only: BF16 activations [R, lda]
    // that the GEMV quantizes itself (then qa and sa are not read).
    const uint16_t *act = nullptr;
    int64_t lda = 0;
    // Stream-K split of dense calls; null sk_cnt: whole tiles only.
    // Weight scales per [sw_block_rows x 128] block: 1 (per row) or 128.
    int sw_block_rows = 1;
    // Weight-only path: x16 holds the caller's BF16 activations (row stride
    // ldx elements), sa is null (no token scale).
    bool a16 = false;
    int64_t ldx = 0;
    int *sk_cnt = nullptr;        // [2 * kSkMaxCtas] counters, zeroed before the GEMM
    float *sk_part = nullptr;     // [kSkMaxCtas][2][sk_ld][128] FP32 partials
    int sk_ld = 0;
};

// Dense calls with at most kGemvMaxTokens token rows run on the CUDA cores
// (batched GEMV over the int8 codes; no fp16 staging copy is made).
constexpr int kGemvMaxTokens = 4;
inline bool uses_gemv(int64_t R, bool grouped) { return !grouped && R <= kGemvMaxTokens; }

// The GEMV can quantize its token rows itself when their codes for all of K
// (K * MR bytes, MR = R rounded up to 1, 2 or 4) fit beside its weight
// stages, and the activation rows allow 16-byte vector loads.
inline bool gemv_can_fuse_quant(int64_t R, int64_t K, int64_t lda, const void *a) {
    const int64_t mr = R <= 1 ? 1 : (R <= 2 ? 2 : 4);
    return R >= 1 && R <= kGemvMaxTokens && K * mr <= 96 * 1024 && lda % 8 == 0 &&
           (reinterpret_cast<uintptr_t>(a) % 16) == 0;
}

// Dense calls of 5..64 token rows (narrow tensor-core tiles) split tiles
// across CTAs (stream-K) when the workspace holds the split area: arrival
// counters and two FP32 partial slots per CTA (token rows x 128 weight rows),
// for at most kSkMaxCtas CTAs. A narrow tile is bound by its MMA issue, not
// by the weight stream, so the steps of a partial last wave are worth
// spreading over all SMs.
constexpr int kSkMaxCtas = 160;
constexpr int kNarrowSplitMaxRows = 64;
inline bool uses_split(int64_t R, bool grouped) {
    return !grouped && R > kGemvMaxTokens && R <= kNarrowSplitMaxRows;
}
inline size_t sk_counter_bytes() { return 2 * kSkMaxCtas * sizeof(int); }
inline size_t sk_area_bytes(int64_t R, bool grouped) {
    if (R <= 0 || !uses_split(R, grouped)) return 0;
    return sk_counter_bytes() +
           static_cast<size_t>(kSkMaxCtas) * 2 * static_cast<size_t>(R) * 128 * sizeof(float);
}

// Dense calls of at least this many token rows run tiles of 128 weight rows x
// 192 token rows (one 192-column MMA per 16 K, two partial buffers in TMEM).
constexpr int kWide256MinRows = 256;
// RMSNorm + per-token quantization (quant.cu): out_kind 0 int8 codes, 1 fp16
// codes (dense rows of K; zeroes n_cnt split counters), 2 the BF16 rows.
// K a multiple of 8, at most kRmsNormMaxK; x, gamma 16-byte aligned, out 16
// (8 for int8 codes); row strides multiples of 8 elements.
constexpr int64_t kRmsNormMaxK = 32768;
cudaError_t launch_rmsnorm_quant(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                                 const uint16_t *gamma, float eps, int out_kind, void *out,
                                 int64_t ldo, float *sa, int *cnt, int n_cnt, bool pow2,
                                 cudaStream_t stream);

inline bool uses_wide256(int64_t R, bool grouped) { return !grouped && R >= kWide256MinRows; }

// Decode attention over a KV cache [B, Hkv, S_max, 128] (attention.cu): INT8
// codes with one scale per vector (ks, vs [B, Hkv, S_max]), or BF16 values.
struct AttnProblem {
    const uint16_t *q;      // [B, Hq, 128] BF16
    const void *kc, *vc;    // caches
    const float *ks, *vs;   // INT8 caches: per-vector scales
    const int32_t *lens;    // [B] device
    int64_t B, Hq, Hkv, S_max;
    float scale;
    bool int8;
    void *out;              // [B, Hq, 128]
    bool out_fp32;
    float *part_o, *part_ml;   // workspace: per-chunk partial outputs and statistics
};
constexpr int kAttnHeadDim = 128;
size_t attn_workspace_bytes(int64_t B, int64_t Hq, int64_t S_max);
cudaError_t launch_attention_decode(const AttnProblem &p, cudaStream_t stream);
// Quantizes n vectors of 128 BF16 values into rows dst_rows[i] (or i) of an
// INT8 cache [rows, 128] with one scale per row.
cudaError_t launch_kv_quant(const uint16_t *x, int64_t n, const int32_t *dst_rows, int8_t *cache,
                            float *scales, cudaStream_t stream);

// Maximum number of experts a grouped call may have.
constexpr int kMaxExperts = 1024;

cudaError_t launch_gemm(const GemmProblem &p, int num_sms, cudaStream_t stream);

// Launches the bounded-wait diagnostic (see gemm.cu): its wait gives up after
// limit_ns and records a code in the device error word.
cudaError_t launch_selftest_wait(unsigned long long limit_ns, cudaStream_t stream);

// Device error word of the GEMM kernel (read/clear; synchronising).
cudaError_t read_device_error(unsigned long long *value, bool clear);

// Device address of the error word (for kernels of other translation units).
cudaError_t device_error_word(unsigned long long **out);

// Rate probes of the MMA paths (probe.cu): tcgen05.mma kind::f16, M = 128,
// N = n, K = 16, A in tensor memory, `chains` accumulators taking turns (on
// the same operands, or each on its own when distinct),
// 8 * chains * steps instructions per CTA on num_sms CTAs; and dp4a,
// 16 * iters per thread on 4 * num_sms CTAs of 512 threads.
cudaError_t launch_probe_tc(int n, int chains, int distinct, long long steps, int num_sms,
                            cudaStream_t stream);
cudaError_t launch_probe_dp4a(long long iters, int num_sms, cudaStream_t stream);

// Per-device properties cached on first use.
struct DeviceInfo {
    int device = -1;
    int cc_major = 0, cc_minor = 0;
    int num_sms = 0;
};
cudaError_t current_device_info(DeviceInfo *out);

}  // namespace w8a8
