// Quantizer kernels for sm_103a:
//  * per-token dynamic activation quantization ("Deploying Hunyuan 770B in
//    INT8 on domestic accelerators", §3.1: activations quantized per token,
//    dynamically; codes = round(x / scale));
//  * per-row, per-128-K-group weight quantization (same section: weights in
//    groups of 128 elements, one scale per group);
//  * the fp16 staging copy of int8 activation codes that the tensor-core
//    GEMM consumes as its B operand (exact: every int8 is an fp16 integer).
//
// All three are HBM-bound streaming kernels: 16-byte vector loads, one CTA
// (activation) or one warp (weight group) per reduction, warp-shuffle amax.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "quant_math.cuh"
#include "internal.h"

namespace w8a8 {
namespace {

constexpr int kQuantThreads = 256;
constexpr int64_t kQuantFewRows = 64;   // up to this many rows: 1024 threads per row

// Block-wide max of non-negative 32-bit integers (all threads get the result).
__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, uint32_t *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    v = lane < (kQuantThreads / 32) ? red[lane] : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// Block-wide sum of floats in a fixed order (all threads get the same result):
// a butterfly over each warp's 32 values, then one over the NT / 32 warp sums.
template <int NT>
__device__ __forceinline__ float block_sum_f32(float v, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    v = lane < (NT / 32) ? red[lane] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Block-wide max of non-negative 32-bit integers over NT threads.
template <int NT>
__device__ __forceinline__ uint32_t block_max_u32_n(uint32_t v, uint32_t *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    v = lane < (NT / 32) ? red[lane] : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// kF16: the codes are written as fp16 (exact integers; the tensor-core GEMM's
// operand) instead of int8, and block 0 also zeroes n_cnt split counters of
// the GEMM that follows (after the wait below, so the GEMM before it, which
// may share them, has finished).
// src_rows (nullable): output row r quantizes input row src_rows[r] (a
// gather, e.g. tokens into expert-sorted order); rows whose entry is
// negative are skipped.
// pow2: power-of-two (UE8M0) scales instead of amax / 127.
// NT threads per row (256; 1024 for a few rows, where the latency of each
// thread's chain of work, not bandwidth, sets the time), VPT vectors each.
template <int NT, int VPT, bool kF16>
__global__ void __launch_bounds__(NT) quant_act_vec_kernel(
    const uint16_t *__restrict__ a, int K, int64_t lda, const int32_t *__restrict__ src_rows,
    void *__restrict__ out, int64_t ldq, float *__restrict__ sa, int *__restrict__ cnt,
    int n_cnt, int pow2) {
    // A GEMM launched after this kernel as a programmatic dependent may start
    // its set-up and weight stream now; it waits for this grid (and so for qa
    // and sa) before it reads the codes. This kernel is itself launched as a
    // programmatic dependent of the kernel before it (which may have written
    // the activations, or still read qa/sa): it waits for that grid before
    // touching either.
    griddep_launch_dependents();
    griddep_wait();
    if (kF16 && blockIdx.x == 0)
        for (int i = threadIdx.x; i < n_cnt; i += blockDim.x) cnt[i] = 0;
    __shared__ uint32_t red[NT / 32];
    const int64_t row = blockIdx.x;
    const int64_t in_row = src_rows != nullptr ? static_cast<int64_t>(src_rows[row]) : row;
    if (in_row < 0) return;
    const uint4 *src = reinterpret_cast<const uint4 *>(a + in_row * lda);
    const int nvec = K >> 3;
    uint4 v[VPT];
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int idx = threadIdx.x + i * NT;
        v[i] = idx < nvec ? __ldcs(src + idx) : make_uint4(0, 0, 0, 0);
        m = max(m, amax_bits8(v[i]));
    }
    m = block_max_u32_n<NT>(m, red);
    const float amax = bf16_bits_to_f32(m);
    const float s = pow2 ? pow2_scale(amax) : __fdiv_rn(amax, 127.0f);
    const bool fast = s >= 1.17549435e-38f;  // normal scale: 1/s is finite
    const float r = fast ? __frcp_rn(s) : 0.0f;
    if (threadIdx.x == 0) sa[row] = s;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int idx = threadIdx.x + i * NT;
        if (idx >= nvec) continue;
        if constexpr (kF16) {
            reinterpret_cast<uint4 *>(static_cast<__half *>(out) + row * ldq)[idx] =
                quantize8_f16(v[i], s, r, fast);
        } else {
            __stcs(reinterpret_cast<uint2 *>(static_cast<int8_t *>(out) + row * ldq) + idx,
                   quantize8(v[i], s, r, fast));
        }
    }
}

// RMSNorm of 8 BF16 values (one 16-byte vector) with their 8 BF16 weights:
// bf16_rn((x * inv) * gamma), two IEEE fp32 products.
__device__ __forceinline__ uint4 rmsnorm8(const uint4 v, const uint4 g, float inv) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
    uint32_t o[4];
    const unsigned long long inv2 = f2_bits(inv, inv);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        // (x * inv) * gamma for both halves, two IEEE products each (f32x2)
        float lo, hi;
        f2_split(f2_mul(f2_mul(f2_bits(bf16_bits_to_f32(w[i] & 0xFFFFu),
                                       bf16_bits_to_f32(w[i] >> 16)),
                               inv2),
                        f2_bits(bf16_bits_to_f32(gw[i] & 0xFFFFu), bf16_bits_to_f32(gw[i] >> 16))),
                 lo, hi);
        const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);   // one conversion for both
        o[i] = *reinterpret_cast<const uint32_t *>(&b);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// RMSNorm of each token row followed by its per-token quantization, one CTA
// of NT threads per row with the row in registers (at most 4 vectors of 8
// values per thread): y = bf16_rn((x * inv) * gamma) with
// inv = 1 / sqrt(sum(x^2) / K + eps) in IEEE fp32 (the sum of squares: one
// fma per element in K order within a thread, then block_sum_f32). The codes
// and scale are those quant_act_vec_kernel gives for the BF16 rows y, so the
// fused kernel equals a BF16 RMSNorm followed by the quantizer, with one HBM
// pass fewer. kOut: 0 int8 codes, 1 fp16 codes (the tensor-core GEMM's
// operand; block 0 also zeroes the n_cnt split counters, as quant_act does),
// 2 the BF16 rows y themselves (no quantization; sa unused).
template <int NT, int kOut>
__global__ void __launch_bounds__(NT) rmsnorm_quant_kernel(
    const uint16_t *__restrict__ x, int K, int64_t ldx, const uint16_t *__restrict__ gamma,
    float eps, void *__restrict__ out, int64_t ldo, float *__restrict__ sa, int *__restrict__ cnt,
    int n_cnt, int pow2) {
    griddep_launch_dependents();   // as in quant_act_vec_kernel
    griddep_wait();
    if (kOut == 1 && blockIdx.x == 0)
        for (int i = threadIdx.x; i < n_cnt; i += blockDim.x) cnt[i] = 0;
    constexpr int VPT = 4;
    __shared__ float redf[NT / 32];
    __shared__ uint32_t red[NT / 32];
    const int64_t row = blockIdx.x;
    const uint4 *src = reinterpret_cast<const uint4 *>(x + row * ldx);
    const int nvec = K >> 3;
    uint4 v[VPT];
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int idx = threadIdx.x + i * NT;
        v[i] = idx < nvec ? __ldcs(src + idx) : make_uint4(0, 0, 0, 0);
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float lo = bf16_bits_to_f32(w[j] & 0xFFFFu);
            const float hi = bf16_bits_to_f32(w[j] >> 16);
            ss = __fmaf_rn(lo, lo, ss);
            ss = __fmaf_rn(hi, hi, ss);
        }
    }
    ss = block_sum_f32<NT>(ss, redf);
    const float inv =
        __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(K)), eps)));
    const uint4 *gv = reinterpret_cast<const uint4 *>(gamma);
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int idx = threadIdx.x + i * NT;
        if (idx < nvec) v[i] = rmsnorm8(v[i], __ldg(gv + idx), inv);
        m = max(m, amax_bits8(v[i]));
    }
    if constexpr (kOut == 2) {
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int idx = threadIdx.x + i * NT;
            if (idx < nvec)
                __stcs(reinterpret_cast<uint4 *>(static_cast<uint16_t *>(out) + row * ldo) + idx,
                       v[i]);
        }
        return;
    }
    m = block_max_u32_n<NT>(m, red);
    const float amax = bf16_bits_to_f32(m);
    const float s = pow2 ? pow2_scale(amax) : __fdiv_rn(amax, 127.0f);
    const bool fast = s >= 1.17549435e-38f;  // normal scale: 1/s is finite
    const float r = fast ? __frcp_rn(s) : 0.0f;
    if (threadIdx.x == 0) sa[row] = s;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int idx = threadIdx.x + i * NT;
        if (idx >= nvec) continue;
        if constexpr (kOut == 1) {
            reinterpret_cast<uint4 *>(static_cast<__half *>(out) + row * ldo)[idx] =
                quantize8_f16(v[i], s, r, fast);
        } else {
            __stcs(reinterpret_cast<uint2 *>(static_cast<int8_t *>(out) + row * ldo) + idx,
                   quantize8(v[i], s, r, fast));
        }
    }
}

// ---- Row stream for many rows (persistent CTAs)
// Each CTA takes rows blockIdx.x + i * grid. One thread keeps kRowRing rows in
// flight: a bulk copy (cp.async.bulk) of each whole row into its own
// shared-memory buffer, issued kRowRing rows ahead, so the copies of the next
// rows run while the block reduces, quantizes and stores the current one. The
// arithmetic per row is that of quant_act_vec_kernel, value for value, so the
// codes and scales are the same. Every wait is bounded: a wait that gives up
// records the error word (kernel 3) and the CTA waits for its copies and
// stops. (Prefill rows, 4096 x 8192: 20.7 -> 18.1 us back to back; a ring of
// 4 rows, or the same stream for RMSNorm + quantization, measured slower than
// one CTA per row.)
// NT threads per CTA and VPT vectors of 8 values per thread: 256 x <= 4 for
// K <= 8192, 512 x 4 up to 16384.
constexpr int kRowRing = 2;
constexpr int64_t kRowRingMaxBytes = 64 * 1024;
// Rows above this count (16-byte aligned, K <= 16384) take the stream.
constexpr int64_t kRowStreamMinRows = kQuantFewRows;
constexpr int64_t kRowStreamMaxK = 16384;

// kOut: 0 int8 codes, 1 fp16 codes (block 0 zeroes n_cnt split counters).
template <int NT, int VPT, int kOut>
__global__ void __launch_bounds__(NT) quant_act_stream_kernel(
    const uint16_t *__restrict__ x, int64_t M, int K, int64_t ldx, void *__restrict__ out,
    int64_t ldo, float *__restrict__ sa, int *__restrict__ cnt, int n_cnt, int pow2,
    unsigned long long *__restrict__ err) {
    griddep_launch_dependents();   // as in quant_act_vec_kernel
    griddep_wait();
    if (kOut == 1 && blockIdx.x == 0)
        for (int i = threadIdx.x; i < n_cnt; i += blockDim.x) cnt[i] = 0;
    extern __shared__ __align__(16) uint8_t ring[];
    __shared__ __align__(8) uint64_t bars[kRowRing];
    __shared__ uint32_t red[NT / 32];
    __shared__ int abort_flag;
    const uint32_t row_bytes = static_cast<uint32_t>(K) * 2u;
    const int64_t grid = gridDim.x;
    const int nvec = K >> 3;
    if (threadIdx.x == 0) {
        for (int b = 0; b < kRowRing; ++b) mbar_init(smem_u32(&bars[b]), 1);
        abort_flag = 0;
        fence_mbarrier_init();
    }
    __syncthreads();
    // local row i: global row blockIdx.x + i * grid, in buffer i % kRowRing
    auto issue = [&](int64_t i) {
        const int64_t row = blockIdx.x + i * grid;
        if (row >= M) return;
        const int b = static_cast<int>(i % kRowRing);
        mbar_arrive_expect_tx(smem_u32(&bars[b]), row_bytes);
        bulk_g2s(smem_u32(ring + b * row_bytes), x + row * ldx, row_bytes, smem_u32(&bars[b]));
    };
    if (threadIdx.x == 0)
        for (int i = 0; i < kRowRing; ++i) issue(i);
    int64_t i = 0;
    for (;; ++i) {
        const int64_t row = blockIdx.x + i * grid;
        if (row >= M) break;
        const int b = static_cast<int>(i % kRowRing);
        const bool ok = mbar_wait(smem_u32(&bars[b]), static_cast<uint32_t>((i / kRowRing) & 1),
                                  &abort_flag, err, ROLE_PRODUCER, 1, kWaitLimitNs, KID_QUANT);
        if (!__syncthreads_and(ok)) break;   // the block stops as one
        const uint4 *src = reinterpret_cast<const uint4 *>(ring + b * row_bytes);
        uint4 v[VPT];
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int idx = threadIdx.x + j * NT;
            v[j] = idx < nvec ? src[idx] : make_uint4(0, 0, 0, 0);
        }
        uint32_t m = 0;
#pragma unroll
        for (int j = 0; j < VPT; ++j) m = max(m, amax_bits8(v[j]));
        m = block_max_u32_n<NT>(m, red);
        // every thread has read buffer b: it takes the row kRowRing ahead
        if (threadIdx.x == 0) issue(i + kRowRing);
        const float amax = bf16_bits_to_f32(m);
        const float s = pow2 ? pow2_scale(amax) : __fdiv_rn(amax, 127.0f);
        const bool fast = s >= 1.17549435e-38f;  // normal scale: 1/s is finite
        const float r = fast ? __frcp_rn(s) : 0.0f;
        if (threadIdx.x == 0) sa[row] = s;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int idx = threadIdx.x + j * NT;
            if (idx >= nvec) continue;
            if constexpr (kOut == 1) {
                reinterpret_cast<uint4 *>(static_cast<__half *>(out) + row * ldo)[idx] =
                    quantize8_f16(v[j], s, r, fast);
            } else {
                __stcs(reinterpret_cast<uint2 *>(static_cast<int8_t *>(out) + row * ldo) + idx,
                       quantize8(v[j], s, r, fast));
            }
        }
    }
    // after a failed wait: the copies still in flight land before the CTA
    // exits (bounded waits that ignore the abort flag)
    if (threadIdx.x == 0 && blockIdx.x + i * grid < M) {
        for (int64_t k = i; k < i + kRowRing; ++k) {
            if (blockIdx.x + k * grid >= M) break;
            const uint32_t bar = smem_u32(&bars[k % kRowRing]);
            const uint32_t par = static_cast<uint32_t>((k / kRowRing) & 1);
            const unsigned long long t0 = globaltimer_ns();
            while (!mbar_try_wait(bar, par) && globaltimer_ns() - t0 < kWaitLimitNs) {
            }
        }
    }
}

// Any K / stride / alignment: scalar two-pass version (re-reads the row).
template <bool kF16>
__global__ void __launch_bounds__(kQuantThreads) quant_act_generic_kernel(
    const uint16_t *__restrict__ a, int K, int64_t lda, const int32_t *__restrict__ src_rows,
    void *__restrict__ out, int64_t ldq, float *__restrict__ sa, int *__restrict__ cnt,
    int n_cnt, int pow2) {
    griddep_launch_dependents();   // as in quant_act_vec_kernel
    griddep_wait();
    if (kF16 && blockIdx.x == 0)
        for (int i = threadIdx.x; i < n_cnt; i += blockDim.x) cnt[i] = 0;
    __shared__ uint32_t red[kQuantThreads / 32];
    const int64_t row = blockIdx.x;
    const int64_t in_row = src_rows != nullptr ? static_cast<int64_t>(src_rows[row]) : row;
    if (in_row < 0) return;
    const uint16_t *src = a + in_row * lda;
    uint32_t m = 0;
    for (int k = threadIdx.x; k < K; k += kQuantThreads) m = max(m, (uint32_t)src[k] & 0x7FFFu);
    m = block_max_u32(m, red);
    const float s = pow2 ? pow2_scale(bf16_bits_to_f32(m)) : __fdiv_rn(bf16_bits_to_f32(m), 127.0f);
    if (threadIdx.x == 0) sa[row] = s;
    for (int k = threadIdx.x; k < K; k += kQuantThreads) {
        const int q = s == 0.0f ? 0 : quantize_exact(bf16_bits_to_f32(src[k]), s);
        if constexpr (kF16)
            static_cast<__half *>(out)[row * ldq + k] = __int2half_rn(q);
        else
            static_cast<int8_t *>(out)[row * ldq + k] = static_cast<int8_t>(q);
    }
}

// One warp per (row n, group g): 128 floats, 4 per lane.
__global__ void __launch_bounds__(256) quant_weight_kernel(const float *__restrict__ w, int64_t N,
                                                           int K, int8_t *__restrict__ qw,
                                                           float *__restrict__ sw) {
    const int G = K / 128;
    const int64_t item = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (item >= N * G) return;
    const int lane = threadIdx.x & 31;
    const int64_t n = item / G;
    const int g = static_cast<int>(item % G);
    const float4 x = *reinterpret_cast<const float4 *>(w + n * K + g * 128 + lane * 4);
    float m = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    const float s = __fdiv_rn(m, 127.0f);
    if (lane == 0) sw[n * G + g] = s;
    uint32_t packed = 0;
    if (s != 0.0f)
        packed = pack4(quantize_exact(x.x, s), quantize_exact(x.y, s), quantize_exact(x.z, s),
                       quantize_exact(x.w, s));
    *reinterpret_cast<uint32_t *>(qw + n * K + g * 128 + lane * 4) = packed;
}

// One CTA per block of `rows` weight rows x 128 K (grid: blocks x groups):
// amax over the block, scale amax / 127 or power of two, codes (second pass
// re-reads the block). Offline input preparation.
__global__ void __launch_bounds__(256) quant_weight_block_kernel(const float *__restrict__ w,
                                                                 int64_t N, int K, int rows,
                                                                 int pow2, int8_t *__restrict__ qw,
                                                                 float *__restrict__ sw) {
    __shared__ float red[8];
    const int G = K / 128;
    const int64_t b = blockIdx.x;
    const int g = blockIdx.y;
    const int64_t n0 = b * rows;
    const int nr = static_cast<int>(min(static_cast<int64_t>(rows), N - n0));
    float m = 0.0f;
    for (int i = threadIdx.x; i < nr * 32; i += 256) {
        const float4 x = *reinterpret_cast<const float4 *>(w + (n0 + i / 32) * K + g * 128 +
                                                           (i % 32) * 4);
        m = fmaxf(m, fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    m = red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) m = fmaxf(m, red[i]);
    const float s = pow2 ? pow2_scale(m) : __fdiv_rn(m, 127.0f);
    if (threadIdx.x == 0) sw[b * G + g] = s;
    for (int i = threadIdx.x; i < nr * 32; i += 256) {
        const int64_t off = (n0 + i / 32) * K + g * 128 + (i % 32) * 4;
        const float4 x = *reinterpret_cast<const float4 *>(w + off);
        uint32_t packed = 0;
        if (s != 0.0f)
            packed = pack4(quantize_exact(x.x, s), quantize_exact(x.y, s), quantize_exact(x.z, s),
                           quantize_exact(x.w, s));
        *reinterpret_cast<uint32_t *>(qw + off) = packed;
    }
}

// int8 codes [rows, K] (row stride ldq) -> fp16 codes [rows, K] (dense).
__global__ void __launch_bounds__(256) widen_codes_kernel(const int8_t *__restrict__ q,
                                                          int64_t rows, int K, int64_t ldq,
                                                          __half *__restrict__ out,
                                                          int *__restrict__ cnt, int n_cnt) {
    // The GEMM that consumes this copy is launched as a programmatic
    // dependent: let it start its set-up and weight stream right away. This
    // kernel is itself a programmatic dependent of the quantizer: wait for
    // its codes (and so, through the quantizer's own wait, for any GEMM
    // before it, which may still use the split counters and the staging
    // copy), before it resets or writes either.
    griddep_launch_dependents();
    griddep_wait();
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < n_cnt; i += blockDim.x) cnt[i] = 0;
    const int vec_per_row = K >> 4;  // 16 codes per vector
    const int64_t total = rows * vec_per_row;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / vec_per_row;
        const int c = static_cast<int>(i % vec_per_row);
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(q + r * ldq) + c);
        uint4 o0, o1;
        i8x4_to_f16x4(v.x, o0.x, o0.y);
        i8x4_to_f16x4(v.y, o0.z, o0.w);
        i8x4_to_f16x4(v.z, o1.x, o1.y);
        i8x4_to_f16x4(v.w, o1.z, o1.w);
        uint4 *d = reinterpret_cast<uint4 *>(out + r * K) + 2 * c;
        d[0] = o0;
        d[1] = o1;
    }
}

// Launch as a programmatic dependent of the previous kernel in the stream.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, cudaStream_t stream,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Row stream: a persistent grid of as many CTAs as fit on the device (by
// shared memory), at most one per row; launched as a programmatic dependent.
template <int NT, int VPT, int kOut>
cudaError_t launch_quant_stream(const uint16_t *x, int64_t M, int K, int64_t ldx, void *out,
                               int64_t ldo, float *sa, int *cnt, int n_cnt, int pow2,
                               cudaStream_t stream) {
    auto kernel = quant_act_stream_kernel<NT, VPT, kOut>;
    const int smem = kRowRing * K * 2;
    DeviceInfo info;
    cudaError_t e = current_device_info(&info);
    if (e != cudaSuccess) return e;
    static int attr_done[64] = {0};   // per device, per kernel instance
    if (info.device >= 0 && info.device < 64 && !attr_done[info.device]) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kRowRingMaxBytes));
        if (e != cudaSuccess) return e;
        attr_done[info.device] = 1;
    }
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, NT, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const int64_t cap = static_cast<int64_t>(per_sm) * info.num_sms;
    unsigned long long *err = nullptr;
    e = device_error_word(&err);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(M < cap ? M : cap));
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, x, M, K, ldx, out, ldo, sa, cnt, n_cnt, pow2, err);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int kOut>
cudaError_t launch_quant_stream_k(const uint16_t *x, int64_t M, int K, int64_t ldx, void *out,
                                 int64_t ldo, float *sa, int *cnt, int n_cnt, int pow2,
                                 cudaStream_t stream) {
    if (K <= 2048)
        return launch_quant_stream<256, 1, kOut>(x, M, K, ldx, out, ldo, sa, cnt, n_cnt, pow2, stream);
    if (K <= 4096)
        return launch_quant_stream<256, 2, kOut>(x, M, K, ldx, out, ldo, sa, cnt, n_cnt, pow2, stream);
    if (K <= 8192)
        return launch_quant_stream<256, 4, kOut>(x, M, K, ldx, out, ldo, sa, cnt, n_cnt, pow2, stream);
    return launch_quant_stream<512, 4, kOut>(x, M, K, ldx, out, ldo, sa, cnt, n_cnt, pow2, stream);
}

template <bool kF16>
cudaError_t launch_quant(const uint16_t *a, int64_t M, int64_t K, int64_t lda, void *out,
                         int64_t ldq, float *sa, int *cnt, int n_cnt, cudaStream_t stream,
                         const int32_t *src_rows = nullptr, int pow2 = 0) {
    const int align = kF16 ? 16 : 8;   // one 8-code vector per store
    const bool vec_ok = (K % 8 == 0) && (lda % 8 == 0) && (ldq % 8 == 0) &&
                        (reinterpret_cast<uintptr_t>(a) % 16 == 0) &&
                        (reinterpret_cast<uintptr_t>(out) % align == 0);
    const int k = static_cast<int>(K);
    const dim3 grid(static_cast<unsigned>(M));
    const dim3 block(kQuantThreads);
    if (cnt == nullptr) n_cnt = 0;
    // many rows: the persistent row stream
    if (vec_ok && src_rows == nullptr && M > kRowStreamMinRows && K <= kRowStreamMaxK)
        return launch_quant_stream_k<kF16 ? 1 : 0>(a, M, k, lda, out, ldq, sa, cnt, n_cnt, pow2,
                                                  stream);
    // a few rows: 1024 threads per row (one or two vectors each)
    if (vec_ok && M <= kQuantFewRows && K <= 1024 * 8 * 1)
        return launch_pdl(quant_act_vec_kernel<1024, 1, kF16>, grid, dim3(1024), stream, a, k, lda,
                          src_rows, out, ldq, sa, cnt, n_cnt, pow2);
    if (vec_ok && M <= kQuantFewRows && K <= 1024 * 8 * 2)
        return launch_pdl(quant_act_vec_kernel<1024, 2, kF16>, grid, dim3(1024), stream, a, k, lda,
                          src_rows, out, ldq, sa, cnt, n_cnt, pow2);
    if (vec_ok && K <= 256 * 8 * 1)
        return launch_pdl(quant_act_vec_kernel<256, 1, kF16>, grid, block, stream, a, k, lda,
                          src_rows, out, ldq, sa, cnt, n_cnt, pow2);
    if (vec_ok && K <= 256 * 8 * 2)
        return launch_pdl(quant_act_vec_kernel<256, 2, kF16>, grid, block, stream, a, k, lda,
                          src_rows, out, ldq, sa, cnt, n_cnt, pow2);
    if (vec_ok && K <= 256 * 8 * 4)
        return launch_pdl(quant_act_vec_kernel<256, 4, kF16>, grid, block, stream, a, k, lda,
                          src_rows, out, ldq, sa, cnt, n_cnt, pow2);
    if (vec_ok && K <= 256 * 8 * 8)
        return launch_pdl(quant_act_vec_kernel<256, 8, kF16>, grid, block, stream, a, k, lda,
                          src_rows, out, ldq, sa, cnt, n_cnt, pow2);
    return launch_pdl(quant_act_generic_kernel<kF16>, grid, block, stream, a, k, lda, src_rows,
                      out, ldq, sa, cnt, n_cnt, pow2);
}

template <int kOut>
cudaError_t launch_rmsnorm_k(const uint16_t *x, int64_t M, int K, int64_t ldx,
                             const uint16_t *gamma, float eps, void *out, int64_t ldo, float *sa,
                             int *cnt, int n_cnt, int pow2, cudaStream_t stream) {
    const dim3 grid(static_cast<unsigned>(M));
    if (K <= 128 * 32)
        return launch_pdl(rmsnorm_quant_kernel<128, kOut>, grid, dim3(128), stream, x, K, ldx,
                          gamma, eps, out, ldo, sa, cnt, n_cnt, pow2);
    if (K <= 256 * 32)
        return launch_pdl(rmsnorm_quant_kernel<256, kOut>, grid, dim3(256), stream, x, K, ldx,
                          gamma, eps, out, ldo, sa, cnt, n_cnt, pow2);
    if (K <= 512 * 32)
        return launch_pdl(rmsnorm_quant_kernel<512, kOut>, grid, dim3(512), stream, x, K, ldx,
                          gamma, eps, out, ldo, sa, cnt, n_cnt, pow2);
    return launch_pdl(rmsnorm_quant_kernel<1024, kOut>, grid, dim3(1024), stream, x, K, ldx,
                      gamma, eps, out, ldo, sa, cnt, n_cnt, pow2);
}

}  // namespace

cudaError_t launch_rmsnorm_quant(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                                 const uint16_t *gamma, float eps, int out_kind, void *out,
                                 int64_t ldo, float *sa, int *cnt, int n_cnt, bool pow2,
                                 cudaStream_t stream) {
    const uintptr_t out_align = out_kind == 0 ? 8 : 16;   // one 8-value vector per store
    if (K <= 0 || K % 8 != 0 || K > kRmsNormMaxK || ldx % 8 != 0 || ldo % 8 != 0 ||
        reinterpret_cast<uintptr_t>(x) % 16 != 0 || reinterpret_cast<uintptr_t>(gamma) % 16 != 0 ||
        reinterpret_cast<uintptr_t>(out) % out_align != 0)
        return cudaErrorInvalidValue;
    if (cnt == nullptr) n_cnt = 0;
    const int k = static_cast<int>(K);
    const int p2 = pow2 ? 1 : 0;
    switch (out_kind) {
    case 0: return launch_rmsnorm_k<0>(x, M, k, ldx, gamma, eps, out, ldo, sa, cnt, n_cnt, p2, stream);
    case 1: return launch_rmsnorm_k<1>(x, M, k, ldx, gamma, eps, out, ldo, sa, cnt, n_cnt, p2, stream);
    case 2: return launch_rmsnorm_k<2>(x, M, k, ldx, gamma, eps, out, ldo, sa, cnt, n_cnt, p2, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_quant_act(const uint16_t *a, int64_t M, int64_t K, int64_t lda, int8_t *qa,
                             int64_t ldq, float *sa, cudaStream_t stream) {
    return launch_quant<false>(a, M, K, lda, qa, ldq, sa, nullptr, 0, stream);
}

cudaError_t launch_quant_act_f16(const uint16_t *a, int64_t M, int64_t K, int64_t lda, void *x16,
                                 float *sa, int *cnt, int n_cnt, cudaStream_t stream) {
    return launch_quant<true>(a, M, K, lda, x16, K, sa, cnt, n_cnt, stream);
}

cudaError_t launch_quant_act_ex(const uint16_t *a, int64_t M, int64_t K, int64_t lda, int8_t *qa,
                                int64_t ldq, float *sa, bool pow2, cudaStream_t stream) {
    return launch_quant<false>(a, M, K, lda, qa, ldq, sa, nullptr, 0, stream, nullptr,
                               pow2 ? 1 : 0);
}

cudaError_t launch_quant_act_f16_ex(const uint16_t *a, int64_t M, int64_t K, int64_t lda,
                                    void *x16, float *sa, int *cnt, int n_cnt, bool pow2,
                                    cudaStream_t stream) {
    return launch_quant<true>(a, M, K, lda, x16, K, sa, cnt, n_cnt, stream, nullptr, pow2 ? 1 : 0);
}

cudaError_t launch_quant_weight_blocks(const float *w, int64_t N, int64_t K, int block_rows,
                                       bool pow2, int8_t *qw, float *sw, cudaStream_t stream) {
    const int64_t nb = (N + block_rows - 1) / block_rows;
    const dim3 grid(static_cast<unsigned>(nb), static_cast<unsigned>(K / 128));
    quant_weight_block_kernel<<<grid, 256, 0, stream>>>(w, N, static_cast<int>(K), block_rows,
                                                         pow2 ? 1 : 0, qw, sw);
    return cudaGetLastError();
}

cudaError_t launch_quant_act_rows(const uint16_t *a, int64_t rows, int64_t K, int64_t lda,
                                  const int32_t *src_rows, void *out, bool f16, float *sa,
                                  cudaStream_t stream) {
    return f16 ? launch_quant<true>(a, rows, K, lda, out, K, sa, nullptr, 0, stream, src_rows)
               : launch_quant<false>(a, rows, K, lda, out, K, sa, nullptr, 0, stream, src_rows);
}

cudaError_t launch_quant_weight(const float *w, int64_t N, int64_t K, int8_t *qw, float *sw,
                                cudaStream_t stream) {
    const int64_t items = N * (K / 128);
    const unsigned blocks = static_cast<unsigned>((items + 7) / 8);
    quant_weight_kernel<<<blocks, 256, 0, stream>>>(w, N, static_cast<int>(K), qw, sw);
    return cudaGetLastError();
}

cudaError_t launch_widen_codes(const int8_t *q, int64_t rows, int64_t K, int64_t ldq, void *out,
                               int num_sms, cudaStream_t stream, int *cnt, int n_cnt) {
    if (cnt == nullptr) n_cnt = 0;
    const int64_t total = rows * (K / 16);
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, widen_codes_kernel, q, rows, static_cast<int>(K),
                                             ldq, static_cast<__half *>(out), cnt, n_cnt);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace w8a8
