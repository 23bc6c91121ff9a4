// INT8 KV cache with per-vector dynamic scales, dequantized inside the
// attention kernel, on sm_103a ("Deploying Hunyuan 770B in INT8 on domestic
// accelerators", §3.4: every key/value vector gets its own scale when it is
// written; the attention kernel reads the INT8 data and applies the scales
// itself instead of running a separate dequantization pass; §2.2: the cache
// holds K and V for every layer, kv head, position and sequence).
//  * kv_quant_kernel: one warp per K or V vector of 128 BF16 values: amax,
//    scale amax / 127, round-half-even codes (the activation quantizer's
//    arithmetic), written to its row of the cache.
//  * attn_decode_kernel: one query token per sequence, grouped-query heads
//    (G query heads per kv head). A CTA takes 128 positions of one (sequence,
//    kv head): it stages the chunk's K and V in shared memory, forms the G x
//    128 scores (K codes widened exactly, the vector's scale applied to the
//    dot product), the chunk's softmax statistics and its unnormalised
//    output; attn_combine_kernel merges the chunks (max / sum rescaling).
// Both kernels are HBM-bound streams of the cache; the BF16-cache form of the
// same kernel (kInt8 = false) is the baseline the fused dequantization is
// measured against.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "quant_math.cuh"
#include "internal.h"

namespace w8a8 {
namespace {

constexpr int kHeadDim = 128;
constexpr int kChunk = 128;          // positions per CTA
constexpr int kAttnThreads = 128;

// ------------------------------------------------------------------ KV write
__global__ void __launch_bounds__(256)
kv_quant_kernel(const uint16_t *__restrict__ x, int64_t n, const int32_t *__restrict__ dst_rows,
                int8_t *__restrict__ cache, float *__restrict__ scales) {
    griddep_launch_dependents();
    griddep_wait();
    const int64_t i = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (i >= n) return;
    const int lane = threadIdx.x & 31;
    const int64_t row = dst_rows != nullptr ? static_cast<int64_t>(dst_rows[i]) : i;
    if (row < 0) return;
    const uint2 v = *reinterpret_cast<const uint2 *>(x + i * kHeadDim + lane * 4);
    uint32_t m = max(max(v.x & 0x7FFFu, (v.x >> 16) & 0x7FFFu),
                     max(v.y & 0x7FFFu, (v.y >> 16) & 0x7FFFu));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    const float s = __fdiv_rn(bf16_bits_to_f32(m), 127.0f);
    const float xs[4] = {bf16_bits_to_f32(v.x & 0xFFFFu), bf16_bits_to_f32(v.x >> 16),
                         bf16_bits_to_f32(v.y & 0xFFFFu), bf16_bits_to_f32(v.y >> 16)};
    int q[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) q[c] = s == 0.0f ? 0 : quantize_exact(xs[c], s);
    *reinterpret_cast<uint32_t *>(cache + row * kHeadDim + lane * 4) = pack4(q[0], q[1], q[2], q[3]);
    if (lane == 0) scales[row] = s;
}

// int8 x4 (one word) -> 4 floats, exact: each byte biased to unsigned is put
// in the low mantissa bits of 2^23 and 2^23 + 128 subtracted.
__device__ __forceinline__ void i8x4_to_f32x4(uint32_t w, float (&f)[4]) {
    const uint32_t u = w ^ 0x80808080u;
#pragma unroll
    for (int c = 0; c < 4; ++c)
        f[c] = __uint_as_float(0x4B000000u | ((u >> (8 * c)) & 0xFFu)) - 8388736.0f;
}

// Shared memory of one CTA (kInt8: codes; else BF16 values).
template <int G, bool kInt8>
struct AttnSmem {
    static constexpr int kRowWords = kInt8 ? kHeadDim / 4 + 1 : kHeadDim / 2 + 1;  // padded
    float q[G][kHeadDim];
    uint32_t k[kChunk][kRowWords];
    uint32_t v[kChunk][kInt8 ? kHeadDim / 4 : kHeadDim / 2];
    float p[kChunk][G];              // scores, then probabilities times the V scale
    float ks[kChunk], vs[kChunk];
    float red[kAttnThreads / 32][G];
    float stat[2][G];                // max, sum
};

// grid (chunks, Hkv, B). Writes, per query head, the chunk's max score,
// sum of exp(score - max) and unnormalised output sum_j exp(s_j - max) v_j.
// Chunks at or past the sequence's length write nothing (the combine reads
// only the first ceil(len / 128)).
template <int G, bool kInt8>
__global__ void __launch_bounds__(kAttnThreads)
attn_decode_kernel(const uint16_t *__restrict__ q, const void *__restrict__ kc,
                   const float *__restrict__ ksc, const void *__restrict__ vc,
                   const float *__restrict__ vsc, const int32_t *__restrict__ lens, int Hkv,
                   int S_max, float scale, float *__restrict__ part_o,
                   float *__restrict__ part_ml) {
    griddep_launch_dependents();
    griddep_wait();   // the cache may have been written by the kernel before
    extern __shared__ __align__(16) uint8_t smem_raw[];
    AttnSmem<G, kInt8> &sm = *reinterpret_cast<AttnSmem<G, kInt8> *>(smem_raw);
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int Hq = Hkv * G;
    const int nch = gridDim.x;
    const int L = min(max(lens[b], 0), S_max);
    const int j0 = c * kChunk;
    if (j0 >= L) return;
    const int n = min(kChunk, L - j0);
    const int64_t vec0 = (static_cast<int64_t>(b) * Hkv + h) * S_max + j0;   // first cache row

    // ---- stage q (FP32), the chunk's K and V rows and their scales
#pragma unroll
    for (int g = 0; g < G; ++g)
        sm.q[g][tid] = bf16_bits_to_f32(q[(static_cast<int64_t>(b) * Hq + h * G + g) * kHeadDim + tid]);
    constexpr int kWords = kInt8 ? kHeadDim / 4 : kHeadDim / 2;   // 32-bit words per row
    const uint4 *kg = reinterpret_cast<const uint4 *>(
        static_cast<const uint8_t *>(kc) + vec0 * kWords * 4);
    const uint4 *vg = reinterpret_cast<const uint4 *>(
        static_cast<const uint8_t *>(vc) + vec0 * kWords * 4);
    for (int idx = tid; idx < n * (kWords / 4); idx += kAttnThreads) {
        const int r = idx / (kWords / 4), w4 = idx % (kWords / 4);
        const uint4 kv = __ldcs(kg + idx);
        const uint4 vv = __ldcs(vg + idx);
        sm.k[r][4 * w4 + 0] = kv.x;
        sm.k[r][4 * w4 + 1] = kv.y;
        sm.k[r][4 * w4 + 2] = kv.z;
        sm.k[r][4 * w4 + 3] = kv.w;
        *reinterpret_cast<uint4 *>(&sm.v[r][4 * w4]) = vv;
    }
    if (kInt8 && tid < n) {
        sm.ks[tid] = ksc[vec0 + tid];
        sm.vs[tid] = vsc[vec0 + tid];
    }
    __syncthreads();

    // ---- scores: thread = position
    float acc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) acc[g] = 0.0f;
    if (tid < n) {
#pragma unroll 4
        for (int w = 0; w < kWords; ++w) {
            const uint32_t kw = sm.k[tid][w];
            if constexpr (kInt8) {
                float f[4];
                i8x4_to_f32x4(kw, f);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float4 qv = *reinterpret_cast<const float4 *>(&sm.q[g][4 * w]);
                    acc[g] = fmaf(qv.x, f[0], fmaf(qv.y, f[1], fmaf(qv.z, f[2], fmaf(qv.w, f[3], acc[g]))));
                }
            } else {
                const float f0 = __uint_as_float(kw << 16), f1 = __uint_as_float(kw & 0xFFFF0000u);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float2 qv = *reinterpret_cast<const float2 *>(&sm.q[g][2 * w]);
                    acc[g] = fmaf(qv.x, f0, fmaf(qv.y, f1, acc[g]));
                }
            }
        }
    }
    const float kscale = (kInt8 && tid < n) ? sm.ks[tid] * scale : scale;
    float s[G];
#pragma unroll
    for (int g = 0; g < G; ++g) s[g] = tid < n ? acc[g] * kscale : -INFINITY;
    // ---- softmax statistics of the chunk, per head
#pragma unroll
    for (int g = 0; g < G; ++g) {
        float m = s[g];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        if (lane == 0) sm.red[warp][g] = m;
    }
    __syncthreads();
    if (tid < G) {
        float m = sm.red[0][tid];
        for (int w = 1; w < kAttnThreads / 32; ++w) m = fmaxf(m, sm.red[w][tid]);
        sm.stat[0][tid] = m;
    }
    __syncthreads();
    float pr[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        pr[g] = tid < n ? expf(s[g] - sm.stat[0][g]) : 0.0f;
        float l = pr[g];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xFFFFFFFFu, l, o);
        if (lane == 0) sm.red[warp][g] = l;
        // probability times the V vector's scale (applied to the PV products)
        sm.p[tid][g] = pr[g] * ((kInt8 && tid < n) ? sm.vs[tid] : 1.0f);
    }
    __syncthreads();
    if (tid < G) {
        float l = 0.0f;
        for (int w = 0; w < kAttnThreads / 32; ++w) l += sm.red[w][tid];
        sm.stat[1][tid] = l;
    }
    // ---- unnormalised output: warp = a quarter of the positions, lane = a
    // word of V (4 int8 or 2 BF16 dimensions); then a sum over the warps
    constexpr int kDimsPerLane = kInt8 ? 4 : 2;
    constexpr int kLaneGroups = kHeadDim / (32 * kDimsPerLane);   // 1 (int8) or 2 (bf16)
    float o[kLaneGroups][G][kDimsPerLane];
#pragma unroll
    for (int a = 0; a < kLaneGroups; ++a)
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int d = 0; d < kDimsPerLane; ++d) o[a][g][d] = 0.0f;
    const int r0 = warp * (kChunk / 4), r1 = min(r0 + kChunk / 4, n);
    for (int r = r0; r < r1; ++r) {
#pragma unroll
        for (int a = 0; a < kLaneGroups; ++a) {
            const uint32_t vw = sm.v[r][lane + 32 * a];
            float f[kDimsPerLane];
            if constexpr (kInt8) {
                float t[4];
                i8x4_to_f32x4(vw, t);
#pragma unroll
                for (int d = 0; d < 4; ++d) f[d] = t[d];
            } else {
                f[0] = __uint_as_float(vw << 16);
                f[1] = __uint_as_float(vw & 0xFFFF0000u);
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float pg = sm.p[r][g];
#pragma unroll
                for (int d = 0; d < kDimsPerLane; ++d) o[a][g][d] = fmaf(pg, f[d], o[a][g][d]);
            }
        }
    }
    __syncthreads();   // sm.k and sm.v (contiguous) hold the cross-warp sum below
    float *red_o = reinterpret_cast<float *>(&sm.k[0][0]);   // [4 warps][G][128]
    static_assert(sizeof(AttnSmem<G, kInt8>::k) + sizeof(AttnSmem<G, kInt8>::v) >=
                      4 * G * kHeadDim * sizeof(float),
                  "cross-warp sum area");
#pragma unroll
    for (int a = 0; a < kLaneGroups; ++a)
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int d = 0; d < kDimsPerLane; ++d)
                red_o[(warp * G + g) * kHeadDim + (lane + 32 * a) * kDimsPerLane + d] = o[a][g][d];
    __syncthreads();
#pragma unroll
    for (int g = 0; g < G; ++g) {
        float sum = 0.0f;
#pragma unroll
        for (int w = 0; w < kAttnThreads / 32; ++w) sum += red_o[(w * G + g) * kHeadDim + tid];
        const int64_t hq = static_cast<int64_t>(b) * Hq + h * G + g;
        part_o[(hq * nch + c) * kHeadDim + tid] = sum;
        if (tid == 0) {
            part_ml[(hq * nch + c) * 2 + 0] = sm.stat[0][g];
            part_ml[(hq * nch + c) * 2 + 1] = sm.stat[1][g];
        }
    }
}

// One CTA per (sequence, query head): merges the chunks of the sequence.
__global__ void __launch_bounds__(kAttnThreads)
attn_combine_kernel(const float *__restrict__ part_o, const float *__restrict__ part_ml,
                    const int32_t *__restrict__ lens, int Hq, int S_max, int nch, void *out,
                    int out_fp32) {
    griddep_launch_dependents();
    griddep_wait();
    const int64_t hq = blockIdx.x;
    const int b = static_cast<int>(hq / Hq);
    const int L = min(max(lens[b], 0), S_max);
    const int nc = (L + kChunk - 1) / kChunk;
    const int d = threadIdx.x;
    float m = -INFINITY;
    for (int c = 0; c < nc; ++c) m = fmaxf(m, part_ml[(hq * nch + c) * 2]);
    float l = 0.0f, acc = 0.0f;
    for (int c = 0; c < nc; ++c) {
        const float w = expf(part_ml[(hq * nch + c) * 2] - m);
        l = fmaf(w, part_ml[(hq * nch + c) * 2 + 1], l);
        acc = fmaf(w, part_o[(hq * nch + c) * kHeadDim + d], acc);
    }
    const float r = nc > 0 ? acc / l : 0.0f;
    if (out_fp32)
        static_cast<float *>(out)[hq * kHeadDim + d] = r;
    else
        static_cast<__nv_bfloat16 *>(out)[hq * kHeadDim + d] = __float2bfloat16_rn(r);
}

template <typename... Params, typename... Args>
cudaError_t launch_pdl_attn(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
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

template <int G, bool kInt8>
cudaError_t launch_attn_g(const AttnProblem &p, cudaStream_t stream) {
    auto kernel = attn_decode_kernel<G, kInt8>;
    const size_t smem = sizeof(AttnSmem<G, kInt8>);
    static int attr_done[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        attr_done[dev] = 1;
    }
    const int nch = static_cast<int>((p.S_max + kChunk - 1) / kChunk);
    e = launch_pdl_attn(kernel, dim3(nch, static_cast<unsigned>(p.Hkv), static_cast<unsigned>(p.B)),
                        dim3(kAttnThreads), smem, stream, p.q, p.kc, p.ks, p.vc, p.vs, p.lens,
                        static_cast<int>(p.Hkv), static_cast<int>(p.S_max), p.scale, p.part_o,
                        p.part_ml);
    if (e != cudaSuccess) return e;
    return launch_pdl_attn(attn_combine_kernel, dim3(static_cast<unsigned>(p.B * p.Hkv * G)),
                           dim3(kAttnThreads), 0, stream, p.part_o, p.part_ml, p.lens,
                           static_cast<int>(p.Hkv * G), static_cast<int>(p.S_max), nch, p.out,
                           p.out_fp32 ? 1 : 0);
}

template <bool kInt8>
cudaError_t launch_attn_kind(const AttnProblem &p, cudaStream_t stream) {
    switch (p.Hq / p.Hkv) {
        case 1: return launch_attn_g<1, kInt8>(p, stream);
        case 2: return launch_attn_g<2, kInt8>(p, stream);
        case 4: return launch_attn_g<4, kInt8>(p, stream);
        case 8: return launch_attn_g<8, kInt8>(p, stream);
        case 16: return launch_attn_g<16, kInt8>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

size_t attn_workspace_bytes(int64_t B, int64_t Hq, int64_t S_max) {
    const int64_t nch = (S_max + kChunk - 1) / kChunk;
    return static_cast<size_t>(B * Hq * nch) * (kHeadDim + 2) * sizeof(float);
}

cudaError_t launch_attention_decode(const AttnProblem &p, cudaStream_t stream) {
    return p.int8 ? launch_attn_kind<true>(p, stream) : launch_attn_kind<false>(p, stream);
}

cudaError_t launch_kv_quant(const uint16_t *x, int64_t n, const int32_t *dst_rows, int8_t *cache,
                            float *scales, cudaStream_t stream) {
    const unsigned blocks = static_cast<unsigned>((n + 7) / 8);
    return launch_pdl_attn(kv_quant_kernel, dim3(blocks), dim3(256), 0, stream, x, n, dst_rows,
                           cache, scales);
}

}  // namespace w8a8
