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
//    kv head): its lanes load their K and V pieces straight into tensor-core
//    fragments, form the 128 x G scores (K codes widened exactly, the
//    vector's scale applied to the dot product), the chunk's softmax
//    statistics and its unnormalised output; attn_combine_kernel merges the
//    chunks (max / sum rescaling).
// Both kernels are HBM-bound streams of the cache; the BF16-cache form of the
// same kernel (kInt8 = false) is the baseline the fused dequantization is
// measured against.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
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

// ------------------------------------------------------- tensor-core helpers
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Transpose of an 8 x 8 matrix of 16-bit values held one 32-bit pair per lane.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ float2 unpack_f16x2(uint32_t x) {
    return __half22float2(*reinterpret_cast<const __half2 *>(&x));
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t x) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&x));
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int i) {
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// Shared memory of one CTA (defined below, after the pipeline stage).
template <int G, bool kInt8>
struct AttnSmem;

// One chunk's operands in registers: K rows pw + 16 mt + gid (+ 8), dims
// [32 t, 32 t + 32); V rows pw + 16 mt + 2 t + {0, 1, 8, 9}, dims [16 gid,
// 16 gid + 16); the K and V scales of the K rows (zero past the sequence).
template <bool kInt8>
struct ChunkRegs {
    static constexpr int kRowBytes = kInt8 ? kHeadDim : 2 * kHeadDim;
    static constexpr int KV = kRowBytes / 4 / 16;   // 16-byte vectors of a lane's 32 K dims
    static constexpr int VV = kRowBytes / 8 / 16;   // 16-byte vectors of a lane's 16 V dims
    uint4 k[2][2][KV];
    uint4 v[2][4][VV];
    float ks[2][2], vs[2][2];
};

// A pipeline stage: one chunk's K and V rows and their scales. Within a row,
// 16-byte piece c is stored at piece c ^ (row & 7), so that the fragment
// reads below (8 rows at the same piece, or 8 pieces spread over rows) fall
// in distinct banks.
template <bool kInt8>
struct ChunkStage {
    static constexpr int kRowBytes = kInt8 ? kHeadDim : 2 * kHeadDim;
    static constexpr int kPieces = kRowBytes / 16;
    uint4 k[kChunk * kPieces];
    uint4 v[kChunk * kPieces];
    float ks[kChunk], vs[kChunk];
};

constexpr int kAttnStages = 2;

// The chunk pipeline's stages, then per-warp softmax statistics; the warps'
// unnormalised outputs are merged through the first stage once the pipeline
// has drained.
template <int G, bool kInt8>
struct AttnSmem {
    static constexpr int kHeads = ((G + 7) / 8) * 8;
    ChunkStage<kInt8> stage[kAttnStages];
    float red_m[kAttnThreads / 32][kHeads];
    float red_l[kAttnThreads / 32][kHeads];
    __device__ float *red_o() { return reinterpret_cast<float *>(&stage[0]); }   // [4][G][128]
};
static_assert(sizeof(ChunkStage<true>) >= 4 * 16 * kHeadDim * sizeof(float), "merge area");

__device__ __forceinline__ int swz(int row, int piece, int pieces) {
    return row * pieces + (piece ^ (row & 7));
}

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// All threads of the CTA copy one chunk of n valid rows starting at cache row
// vec0 into a stage (rows >= n are zero-filled and not read).
template <bool kInt8>
__device__ __forceinline__ void issue_chunk(ChunkStage<kInt8> &sg, const void *kc, const void *vc,
                                            const float *ksc, const float *vsc, int64_t vec0,
                                            int n) {
    using S = ChunkStage<kInt8>;
    const uint4 *kg = reinterpret_cast<const uint4 *>(kc) + vec0 * S::kPieces;
    const uint4 *vg = reinterpret_cast<const uint4 *>(vc) + vec0 * S::kPieces;
#pragma unroll
    for (int i = threadIdx.x; i < kChunk * S::kPieces; i += kAttnThreads) {
        const int row = i / S::kPieces, piece = i % S::kPieces;
        const uint32_t bytes = row < n ? 16u : 0u;
        const int src = row < n ? i : 0;
        const int dst = swz(row, piece, S::kPieces);
        cp_async_16(smem_u32(&sg.k[dst]), kg + src, bytes);
        cp_async_16(smem_u32(&sg.v[dst]), vg + src, bytes);
    }
    if constexpr (kInt8) {
        const int row = threadIdx.x;   // kAttnThreads == kChunk
        const int64_t src = vec0 + (row < n ? row : 0);
        cp_async_4(smem_u32(&sg.ks[row]), ksc + src, row < n ? 4u : 0u);
        cp_async_4(smem_u32(&sg.vs[row]), vsc + src, row < n ? 4u : 0u);
    }
}

// The lane's fragments of a landed stage.
template <bool kInt8>
__device__ __forceinline__ void frags_of_stage(ChunkRegs<kInt8> &r, const ChunkStage<kInt8> &sg,
                                               int n, int pw, int gid, int t) {
    using S = ChunkStage<kInt8>;
    using R = ChunkRegs<kInt8>;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const int row = pw + 16 * mt + gid + 8 * hf;
#pragma unroll
            for (int v = 0; v < R::KV; ++v) r.k[mt][hf][v] = sg.k[swz(row, t * R::KV + v, S::kPieces)];
            if constexpr (kInt8) {
                r.ks[mt][hf] = sg.ks[row];
                r.vs[mt][hf] = sg.vs[row];
            } else {
                r.ks[mt][hf] = 1.0f;
                r.vs[mt][hf] = row < n ? 1.0f : 0.0f;
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int row = pw + 16 * mt + 2 * t + (j < 2 ? j : j + 6);
#pragma unroll
            for (int v = 0; v < R::VV; ++v)
                r.v[mt][j][v] = sg.v[swz(row, gid * R::VV + v, S::kPieces)];
        }
    }
}

// Running state of one warp over the chunks it has seen: per head its max
// score, the lane's share of sum exp(s - max), and the unnormalised output
// (in units of 2^-se: the fp16 range scaling of the INT8 cache).
template <int NT>
struct WarpState {
    float m[NT][2];
    float l[NT][2];
    float o[8][NT][4];
    int se;
};

// One chunk of n valid rows into the warp's running state (online softmax:
// the state is rescaled by exp(m_old - m_new) when a larger score arrives).
template <int G, bool kInt8>
__device__ __forceinline__ void attend_chunk(WarpState<(G + 7) / 8> &st, const ChunkRegs<kInt8> &r,
                                             const uint32_t (&qf)[(G + 7) / 8][16], int n,
                                             float scale, float qinv, int pw, int gid, int t) {
    constexpr int NT = (G + 7) / 8;
    // ---- scores: k-step kb covers dims 32 t + 4 kb + {0..3} of each lane
    float sacc[2][NT][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) sacc[mt][nt][i] = 0.0f;
#pragma unroll
    for (int kb = 0; kb < 8; ++kb) {
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
            uint32_t a[4];
            if constexpr (kInt8) {
                // codes widened exactly to fp16; q is in fp16 too (scaled)
                i8x4_to_f16x4(word_of(r.k[mt][0][kb >> 2], kb & 3), a[0], a[2]);
                i8x4_to_f16x4(word_of(r.k[mt][1][kb >> 2], kb & 3), a[1], a[3]);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    mma_f16(sacc[mt][nt], a, qf[nt][2 * kb], qf[nt][2 * kb + 1]);
            } else {
                a[0] = word_of(r.k[mt][0][kb >> 1], (2 * kb) & 3);
                a[2] = word_of(r.k[mt][0][kb >> 1], (2 * kb + 1) & 3);
                a[1] = word_of(r.k[mt][1][kb >> 1], (2 * kb) & 3);
                a[3] = word_of(r.k[mt][1][kb >> 1], (2 * kb + 1) & 3);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    mma_bf16(sacc[mt][nt], a, qf[nt][2 * kb], qf[nt][2 * kb + 1]);
            }
        }
    }
    // scaled scores (fragment i: row gid + 8 (i >> 1), head 8 nt + 2 t + (i & 1))
    // and the chunk's max per head over the warp
    float mc[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) mc[nt][0] = mc[nt][1] = -INFINITY;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int hf = i >> 1;
                const int row = pw + 16 * mt + gid + 8 * hf;
                // (the fp16 q carries the power of two 1/qinv: scaling back is exact)
                const float sv =
                    row < n ? (sacc[mt][nt][i] * (r.ks[mt][hf] * scale)) * qinv : -INFINITY;
                sacc[mt][nt][i] = sv;
                mc[nt][i & 1] = fmaxf(mc[nt][i & 1], sv);
            }
    float mu[NT][2], alpha[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float m = mc[nt][j];
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
            const float m_new = fmaxf(st.m[nt][j], m);
            mu[nt][j] = m_new == -INFINITY ? 0.0f : m_new;   // no valid score yet
            alpha[nt][j] = expf(st.m[nt][j] - mu[nt][j]);    // 0 while the state is empty
            st.m[nt][j] = m_new;
            st.l[nt][j] *= alpha[nt][j];
        }
    // the warp's largest V scale of the chunk sets the power of two that keeps
    // P' in fp16's normal range (INT8 cache); rows of other lanes t are the same
    int se = st.se;
    if constexpr (kInt8) {
        float vmax = fmaxf(fmaxf(r.vs[0][0], r.vs[0][1]), fmaxf(r.vs[1][0], r.vs[1][1]));
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xFFFFFFFFu, vmax, o));
        const int bexp = static_cast<int>((__float_as_uint(vmax) >> 23) & 0xFFu);
        if (bexp != 0) se = max(-100, min(100, 14 - (bexp - 127)));
    }
    // rescale the state's output: exp(m_old - m_new) and the change of units
    const float ratio = __uint_as_float(static_cast<uint32_t>(se - st.se + 127) << 23);
    st.se = se;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int k = 0; k < 4; ++k) st.o[i][nt][k] *= alpha[nt][k & 1] * ratio;
    const float pscale = __uint_as_float(static_cast<uint32_t>(se + 127) << 23);
    // probabilities, their sums, and the B fragments of the output product
    constexpr int NS = kInt8 ? 2 : 3;   // hi, lo (fp16) or hi, mid, lo (bf16)
    uint32_t bp[2][NT][NS][2];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            float pp[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float pr = expf(sacc[mt][nt][i] - mu[nt][i & 1]);
                st.l[nt][i & 1] += pr;
                pp[i] = (pr * r.vs[mt][i >> 1]) * pscale;
            }
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const float x0 = pp[2 * hf], x1 = pp[2 * hf + 1];
                if constexpr (kInt8) {
                    const uint32_t hi = pack_f16x2(x0, x1);
                    const float2 hv = unpack_f16x2(hi);
                    const uint32_t lo = pack_f16x2(x0 - hv.x, x1 - hv.y);
                    bp[mt][nt][0][hf] = movmatrix_trans(hi);
                    bp[mt][nt][1][hf] = movmatrix_trans(lo);
                } else {
                    const uint32_t hi = pack_bf16x2(x0, x1);
                    const float2 hv = unpack_bf16x2(hi);
                    const float r0 = x0 - hv.x, r1 = x1 - hv.y;
                    const uint32_t mid = pack_bf16x2(r0, r1);
                    const float2 mv = unpack_bf16x2(mid);
                    const uint32_t lo = pack_bf16x2(r0 - mv.x, r1 - mv.y);
                    bp[mt][nt][0][hf] = movmatrix_trans(hi);
                    bp[mt][nt][1][hf] = movmatrix_trans(mid);
                    bp[mt][nt][2][hf] = movmatrix_trans(lo);
                }
            }
        }
    // ---- unnormalised output: m-tile i holds dims 16 gid + 2 i (row gid) and
    // 16 gid + 2 i + 1 (row gid + 8)
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint32_t a[4];
            if constexpr (kInt8) {
                // bytes 2i, 2i + 1 of the four positions' 16-byte vectors, as
                // fp16 pairs over positions (1024 + biased byte, minus 1152)
                const int w = i >> 1;
                const uint32_t sel = (i & 1) ? 0x7362u : 0x5140u;
                const uint32_t g01 = prmt(word_of(r.v[mt][0][0], w) ^ 0x80808080u,
                                          word_of(r.v[mt][1][0], w) ^ 0x80808080u, sel);
                const uint32_t g23 = prmt(word_of(r.v[mt][2][0], w) ^ 0x80808080u,
                                          word_of(r.v[mt][3][0], w) ^ 0x80808080u, sel);
                const uint32_t x[4] = {prmt(g01, 0x64646464u, 0x4140u),
                                       prmt(g01, 0x64646464u, 0x4342u),
                                       prmt(g23, 0x64646464u, 0x4140u),
                                       prmt(g23, 0x64646464u, 0x4342u)};
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(a[k]) : "r"(x[k]), "r"(0x64806480u));
            } else {
                const uint32_t w0 = word_of(r.v[mt][0][i >> 2], i & 3);
                const uint32_t w1 = word_of(r.v[mt][1][i >> 2], i & 3);
                const uint32_t w2 = word_of(r.v[mt][2][i >> 2], i & 3);
                const uint32_t w3 = word_of(r.v[mt][3][i >> 2], i & 3);
                a[0] = prmt(w0, w1, 0x5410u);
                a[1] = prmt(w0, w1, 0x7632u);
                a[2] = prmt(w2, w3, 0x5410u);
                a[3] = prmt(w2, w3, 0x7632u);
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int sp = 0; sp < NS; ++sp) {
                    if constexpr (kInt8)
                        mma_f16(st.o[i][nt], a, bp[mt][nt][sp][0], bp[mt][nt][sp][1]);
                    else
                        mma_bf16(st.o[i][nt], a, bp[mt][nt][sp][0], bp[mt][nt][sp][1]);
                }
        }
    }
}

// grid (splits, Hkv, B), 4 warps. A CTA takes `span` consecutive 128-position
// chunks of one (sequence, kv head). The chunks stream through a two-stage
// shared-memory pipeline (cp.async, one chunk ahead of the one being read);
// warp w works on positions [32 w, 32 w + 32) of each chunk from registers
// and keeps its own running softmax state. At the end the four warps' states
// are merged and the CTA writes, per query head, the split's max score, sum
// of exp(score - max) and unnormalised output sum_j exp(s_j - max) v_j.
// Splits at or past the sequence's length write nothing (the combine reads
// only the first ceil(ceil(len / 128) / span)).
//
// Both products run on the tensor cores (mma.sync m16n8k16, FP32
// accumulation):
//  * scores S^T[p, g] = sum_d K[p, d] q[g, d]: A = the K rows (int8 codes
//    widened exactly to bf16, or the BF16 values), B = q (BF16). The
//    reduction index d is permuted identically in A and B (a lane reads 32
//    contiguous dimensions of its rows), which leaves every sum unchanged.
//    Then s = S^T * (k_scale * softmax scale);
//  * output O^T[d, g] = sum_p V[p, d] P'[p, g] with P' = exp(s - m) * v_scale:
//    A = V^T (codes widened exactly to fp16, or BF16 values; output rows d
//    permuted so that a lane reads 16 contiguous dimensions), B = P' moved
//    from the score fragments by an in-register transpose (movmatrix). P' is
//    split into fp16 hi + lo (bf16 hi + mid + lo for the BF16 cache), so the
//    products keep 22 (24) significant bits of P': the same accuracy class as
//    FP32 products. For the INT8 cache, P' is first scaled by the power of two
//    2^(14 - e) (e the exponent of the warp's largest v_scale in the chunk),
//    keeping it in fp16's normal range; the sums are scaled back exactly.
template <int G, bool kInt8, bool kQVec>
__global__ void __launch_bounds__(kAttnThreads)
attn_decode_kernel(const uint16_t *__restrict__ q, const void *__restrict__ kc,
                   const float *__restrict__ ksc, const void *__restrict__ vc,
                   const float *__restrict__ vsc, const int32_t *__restrict__ lens, int Hkv,
                   int S_max, int span, float scale, float *__restrict__ part_o,
                   float *__restrict__ part_ml) {
    constexpr int NT = (G + 7) / 8;                 // n-tiles of 8 query heads
    griddep_launch_dependents();
    griddep_wait();   // the cache may have been written by the kernel before
    extern __shared__ __align__(16) uint8_t smem_raw[];
    AttnSmem<G, kInt8> &sm = *reinterpret_cast<AttnSmem<G, kInt8> *>(smem_raw);
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gid = lane >> 2, t = lane & 3;
    const int Hq = Hkv * G;
    const int nsplit = gridDim.x;
    const int L = min(max(lens[b], 0), S_max);
    const int nc = (L + kChunk - 1) / kChunk;
    const int c_begin = split * span;
    const int c_end = min(c_begin + span, nc);
    if (c_begin >= c_end) return;
    const int64_t row0 = (static_cast<int64_t>(b) * Hkv + h) * S_max;   // the pair's cache rows
    const int pw = warp * 32;
    auto rows_of = [&](int cc) { return min(kChunk, L - cc * kChunk); };
    auto issue = [&](int cc) {
        issue_chunk(sm.stage[(cc - c_begin) % kAttnStages], kc, vc, ksc, vsc,
                    row0 + static_cast<int64_t>(cc) * kChunk, rows_of(cc));
    };
    // the first two chunks in flight (one commit group per chunk, empty past
    // the split's end, so that the group count stays uniform)
    issue(c_begin);
    cp_async_commit();
    if (c_begin + 1 < c_end) issue(c_begin + 1);
    cp_async_commit();

    // q rows 8 nt + gid, dims [32 t, 32 t + 32), as bf16 pairs
    uint32_t qf[NT][16];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int g = 8 * nt + gid;
        const uint16_t *qrow =
            q + (static_cast<int64_t>(b) * Hq + h * G + (g < G ? g : 0)) * kHeadDim + 32 * t;
        if constexpr (kQVec) {   // q 16-byte aligned, else 2-byte loads
            const uint4 *src = reinterpret_cast<const uint4 *>(qrow);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const uint4 x = g < G ? __ldg(src + v) : make_uint4(0, 0, 0, 0);
                qf[nt][4 * v + 0] = x.x;
                qf[nt][4 * v + 1] = x.y;
                qf[nt][4 * v + 2] = x.z;
                qf[nt][4 * v + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int w = 0; w < 16; ++w)
                qf[nt][w] = g < G ? (static_cast<uint32_t>(__ldg(qrow + 2 * w)) |
                                     (static_cast<uint32_t>(__ldg(qrow + 2 * w + 1)) << 16))
                                  : 0u;
        }
    }
    // INT8 cache: the score product runs in fp16 (the codes widen to fp16 in
    // half the instructions bf16 takes). q goes to fp16 scaled by the power of
    // two 2^(14 - e), e the exponent of the largest |q| of the CTA's heads (the
    // warp holds all of them), so the largest value sits in [2^14, 2^15) and
    // every value of at least 2^-14 of the scaled range converts exactly; the
    // scores are scaled back by qinv exactly.
    float qinv = 1.0f;
    if constexpr (kInt8) {
        uint32_t mq = 0;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int w = 0; w < 16; ++w) mq = __vmaxu2(mq, qf[nt][w] & 0x7FFF7FFFu);
        mq = max(mq & 0xFFFFu, mq >> 16);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) mq = max(mq, __shfl_xor_sync(0xFFFFFFFFu, mq, o));
        const int bexp = static_cast<int>((mq >> 7) & 0xFFu);   // bf16 exponent field
        const int se = bexp == 0 ? 0 : max(-100, min(100, 14 - (bexp - 127)));
        const float qs = __uint_as_float(static_cast<uint32_t>(se + 127) << 23);
        qinv = __uint_as_float(static_cast<uint32_t>(127 - se) << 23);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int w = 0; w < 16; ++w) {
                const __half2 hq = __floats2half2_rn(__uint_as_float(qf[nt][w] << 16) * qs,
                                                     __uint_as_float(qf[nt][w] & 0xFFFF0000u) * qs);
                qf[nt][w] = *reinterpret_cast<const uint32_t *>(&hq);
            }
    }
    WarpState<NT> st;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            st.m[nt][j] = -INFINITY;
            st.l[nt][j] = 0.0f;
        }
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int k = 0; k < 4; ++k) st.o[i][nt][k] = 0.0f;
    st.se = 0;

    for (int cc = c_begin; cc < c_end; ++cc) {
        cp_async_wait_group<1>();   // this chunk's group has landed (the next may be in flight)
        __syncthreads();
        ChunkRegs<kInt8> r;
        frags_of_stage(r, sm.stage[(cc - c_begin) % kAttnStages], rows_of(cc), pw, gid, t);
        __syncthreads();            // every warp has its fragments: the stage is free
        if (cc + 2 < c_end) issue(cc + 2);
        cp_async_commit();
        attend_chunk<G, kInt8>(st, r, qf, rows_of(cc), scale, qinv, pw, gid, t);
    }
    cp_async_wait_group<0>();
    __syncthreads();   // the stages are free for the merge below

    // ---- merge the four warps: the lanes' sums over the warp, then every
    // warp's state rescaled to the CTA's max
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float l = st.l[nt][j];
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) l += __shfl_xor_sync(0xFFFFFFFFu, l, o);
            if (gid == 0) {
                sm.red_m[warp][8 * nt + 2 * t + j] = st.m[nt][j];
                sm.red_l[warp][8 * nt + 2 * t + j] = l;
            }
        }
    __syncthreads();
    float wf[NT][2];   // this warp's weight exp(m_warp - m_cta) per head
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int g = 8 * nt + 2 * t + j;
            float m = sm.red_m[0][g];
#pragma unroll
            for (int w = 1; w < kAttnThreads / 32; ++w) m = fmaxf(m, sm.red_m[w][g]);
            wf[nt][j] = expf(st.m[nt][j] - m);   // 0 for a warp without valid rows
        }
    const float unit = __uint_as_float(static_cast<uint32_t>(127 - st.se) << 23);   // 2^-se
    float *red_o = sm.red_o();
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int g = 8 * nt + 2 * t + (k & 1);
                const int d = 16 * gid + 2 * i + (k >> 1);
                if (g < G)
                    red_o[(warp * G + g) * kHeadDim + d] = (st.o[i][nt][k] * unit) * wf[nt][k & 1];
            }
    __syncthreads();
#pragma unroll
    for (int g = 0; g < G; ++g) {
        float sum = 0.0f;
#pragma unroll
        for (int w = 0; w < kAttnThreads / 32; ++w) sum += red_o[(w * G + g) * kHeadDim + tid];
        const int64_t hq = static_cast<int64_t>(b) * Hq + h * G + g;
        part_o[(hq * nsplit + split) * kHeadDim + tid] = sum;
    }
    if (tid < G) {
        float m = sm.red_m[0][tid];
#pragma unroll
        for (int w = 1; w < kAttnThreads / 32; ++w) m = fmaxf(m, sm.red_m[w][tid]);
        float l = 0.0f;
#pragma unroll
        for (int w = 0; w < kAttnThreads / 32; ++w)
            l += sm.red_l[w][tid] * expf(sm.red_m[w][tid] - m);
        const int64_t hq = static_cast<int64_t>(b) * Hq + h * G + tid;
        part_ml[(hq * nsplit + split) * 2 + 0] = m;
        part_ml[(hq * nsplit + split) * 2 + 1] = l;
    }
}

// One CTA per (sequence, query head): merges the splits of the sequence.
__global__ void __launch_bounds__(kAttnThreads)
attn_combine_kernel(const float *__restrict__ part_o, const float *__restrict__ part_ml,
                    const int32_t *__restrict__ lens, int Hq, int S_max, int nch, int span, void *out,
                    int out_fp32) {
    griddep_launch_dependents();
    griddep_wait();
    const int64_t hq = blockIdx.x;
    const int b = static_cast<int>(hq / Hq);
    const int L = min(max(lens[b], 0), S_max);
    const int nc = ((L + kChunk - 1) / kChunk + span - 1) / span;   // splits with rows
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

template <int G, bool kInt8, bool kQVec>
cudaError_t launch_attn_q(const AttnProblem &p, cudaStream_t stream) {
    auto kernel = attn_decode_kernel<G, kInt8, kQVec>;
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
    // Splits of `span` chunks per (sequence, kv head): as many splits as make
    // about two waves of resident CTAs (B=32, 8 kv heads, 4096 positions: 4
    // splits of 8 chunks, 54.7 us, against 61.0 us with 8 splits of 4, 57.6
    // with 3 of 11 and 59.3 with 2 of 16). Longer splits pay each CTA's start
    // (q, pipeline fill, merge) over more positions and leave fewer partials
    // to combine.
    const int64_t nch = (p.S_max + kChunk - 1) / kChunk;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kAttnThreads, smem);
    if (e != cudaSuccess) return e;
    DeviceInfo info;
    e = current_device_info(&info);
    if (e != cudaSuccess) return e;
    const int64_t slots = static_cast<int64_t>(per_sm > 0 ? per_sm : 1) * info.num_sms;
    const int64_t pairs = p.B * p.Hkv;
    int64_t want = (2 * slots + pairs - 1) / pairs;                 // splits per pair
    want = want < 1 ? 1 : (want > nch ? nch : want);
    const int span = static_cast<int>((nch + want - 1) / want);
    const int nsplit = static_cast<int>((nch + span - 1) / span);
    e = launch_pdl_attn(kernel,
                        dim3(static_cast<unsigned>(nsplit), static_cast<unsigned>(p.Hkv),
                             static_cast<unsigned>(p.B)),
                        dim3(kAttnThreads), smem, stream, p.q, p.kc, p.ks, p.vc, p.vs, p.lens,
                        static_cast<int>(p.Hkv), static_cast<int>(p.S_max), span, p.scale,
                        p.part_o, p.part_ml);
    if (e != cudaSuccess) return e;
    return launch_pdl_attn(attn_combine_kernel, dim3(static_cast<unsigned>(p.B * p.Hkv * G)),
                           dim3(kAttnThreads), 0, stream, p.part_o, p.part_ml, p.lens,
                           static_cast<int>(p.Hkv * G), static_cast<int>(p.S_max), nsplit, span,
                           p.out, p.out_fp32 ? 1 : 0);
}

template <int G, bool kInt8>
cudaError_t launch_attn_g(const AttnProblem &p, cudaStream_t stream) {
    return (reinterpret_cast<uintptr_t>(p.q) & 15u) == 0 ? launch_attn_q<G, kInt8, true>(p, stream)
                                                        : launch_attn_q<G, kInt8, false>(p, stream);
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
