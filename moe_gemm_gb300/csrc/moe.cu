// The MoE expert FFN steps around the two grouped W8A8 GEMMs, on sm_103a
// ("Deploying Hunyuan 770B in INT8 on domestic accelerators": §4.4, tokens
// are counted per destination expert first and then transferred in bulk;
// §4.1, SwiGLU sits between the INT8 expert GEMMs; §3.1, every INT8 GEMM
// input is quantized per token, dynamically):
//  * routing: histogram of the top-k expert ids, exclusive prefix sum into
//    segment offsets, and a stable permutation (rows sorted by expert, then by
//    (token, slot) order), in one CTA;
//  * SwiGLU of the gate_up output, h = silu(gate) * up in binary32, followed
//    by the per-token quantization of h that the down GEMM consumes;
//  * the weighted un-permute, y[t] = sum_j w[t, j] * D[row(t, j)].
// The permuted token rows are quantized by the activation quantizer with a
// row gather (quant.cu), and the GEMMs are the grouped tensor-core kernels.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "quant_math.cuh"
#include "internal.h"

namespace w8a8 {
namespace {

// ------------------------------------------------------------------ routing
constexpr int kRouteThreads = 1024;
constexpr int kRouteWarps = kRouteThreads / 32;

// One CTA of 32 warps. Warp w owns the entries [w C, (w + 1) C), C = ceil(n /
// 32), and walks them 32 at a time in entry order. Shared memory: cntw[w][e]
// (the warp's count of expert e, then the first row of its expert-e entries)
// and tot[e + 1]. Entries whose id is outside [0, E) are not routed (row_of =
// -1). The rows of an expert keep the entries' order (warps in order, lanes
// in order within a warp), so the permutation is the stable sort by expert.
__global__ void __launch_bounds__(kRouteThreads)
moe_route_kernel(const int32_t *__restrict__ ids, int n, int k, int E, int32_t *__restrict__ offsets,
                 int32_t *__restrict__ row_of, int32_t *__restrict__ token_of_row,
                 int32_t *__restrict__ pair_of_row) {
    extern __shared__ int s_route[];
    int *cntw = s_route;                       // [kRouteWarps][E]
    int *tot = s_route + kRouteWarps * E;      // [E + 1]
    __shared__ int s_part[kRouteWarps];
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const unsigned lt_mask = (1u << lane) - 1u;
    griddep_wait();   // the ids may come from the kernel launched before
    for (int i = tid; i < kRouteWarps * E; i += kRouteThreads) cntw[i] = 0;
    for (int r = tid; r < n; r += kRouteThreads) {
        token_of_row[r] = -1;
        pair_of_row[r] = -1;
    }
    __syncthreads();
    const int C = (n + kRouteWarps - 1) / kRouteWarps;
    const int i0 = warp * C, i1 = min(i0 + C, n);
    int *mine = cntw + warp * E;
    // counts per (warp, expert): one leader per group of equal ids
    for (int b = i0; b < i1; b += 32) {
        const int i = b + lane;
        const int e = i < i1 ? ids[i] : -1;
        const bool valid = e >= 0 && e < E;
        const unsigned peers = __match_any_sync(0xFFFFFFFFu, valid ? e : -1);
        if (valid && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    // per expert: exclusive prefix over the warps, and the expert's total
    for (int e = tid; e < E; e += kRouteThreads) {
        int run = 0;
        for (int w = 0; w < kRouteWarps; ++w) {
            const int c = cntw[w * E + e];
            cntw[w * E + e] = run;
            run += c;
        }
        tot[e] = run;
    }
    __syncthreads();
    // exclusive prefix over the experts: each warp scans a contiguous range
    // of experts, then the warps' sums are scanned
    const int per = (E + kRouteThreads - 1) / kRouteThreads;   // experts per thread
    const int e0 = min(tid * per, E), e1 = min(e0 + per, E);
    int local = 0;
    for (int e = e0; e < e1; ++e) local += tot[e];
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) s_part[warp] = incl;
    __syncthreads();
    int wbase = 0;
    for (int w = 0; w < warp; ++w) wbase += s_part[w];
    int run = wbase + incl - local;
    __syncthreads();   // every thread has read tot[e0, e1) before it is overwritten
    for (int e = e0; e < e1; ++e) {
        const int c = tot[e];
        tot[e] = run;
        offsets[e] = run;
        run += c;
    }
    if (tid == kRouteThreads - 1) {
        int all = 0;
        for (int w = 0; w < kRouteWarps; ++w) all += s_part[w];
        offsets[E] = all;
    }
    __syncthreads();
    for (int i = tid; i < kRouteWarps * E; i += kRouteThreads) cntw[i] += tot[i % E];
    __syncthreads();
    // scatter: the same walk, each group of equal ids taking its rows from
    // the warp's running start for that expert
    for (int b = i0; b < i1; b += 32) {
        const int i = b + lane;
        const int e = i < i1 ? ids[i] : -1;
        const bool valid = e >= 0 && e < E;
        const unsigned peers = __match_any_sync(0xFFFFFFFFu, valid ? e : -1);
        const int leader = __ffs(peers) - 1;
        int start = 0;
        if (valid && lane == leader) {
            start = mine[e];
            mine[e] = start + __popc(peers);
        }
        start = __shfl_sync(0xFFFFFFFFu, start, leader);
        if (valid) {
            const int r = start + __popc(peers & lt_mask);
            row_of[i] = r;
            token_of_row[r] = i / k;
            pair_of_row[r] = i;
        } else if (i < i1) {
            row_of[i] = -1;
        }
        __syncwarp();
    }
}

// ---------------------------------------------------------- SwiGLU + quant
// e^x in binary32 by Cody and Waite's method: x clamped to [-87, 88], n =
// round-half-even(x log2 e), r = x - n ln2 with ln2 split into a 15-bit head
// (n * head exact) and a tail, e^r by its degree-7 Taylor series (Horner),
// scaled by 2^n. Every step is a separately rounded binary32 operation (the
// _rn intrinsics are never fused into multiply-adds), so the result is a fixed
// function of x, the same in any implementation of these steps.
__device__ __forceinline__ float exp_f32_cw(float x) {
    x = fminf(fmaxf(x, -87.0f), 88.0f);
    const float n = rintf(__fmul_rn(x, 1.44269502163f));
    float r = __fsub_rn(x, __fmul_rn(n, 0.693145751953125f));
    r = __fsub_rn(r, __fmul_rn(n, 1.42860676533018e-06f));
    float p = 1.0f / 5040.0f;
    p = __fadd_rn(__fmul_rn(p, r), 1.0f / 720.0f);
    p = __fadd_rn(__fmul_rn(p, r), 1.0f / 120.0f);
    p = __fadd_rn(__fmul_rn(p, r), 1.0f / 24.0f);
    p = __fadd_rn(__fmul_rn(p, r), 1.0f / 6.0f);
    p = __fadd_rn(__fmul_rn(p, r), 0.5f);
    p = __fadd_rn(__fmul_rn(p, r), 1.0f);
    p = __fadd_rn(__fmul_rn(p, r), 1.0f);
    return __fmul_rn(p, __int_as_float((static_cast<int>(n) + 127) << 23));
}

// h = silu(g) * u = (g / (1 + e^-g)) * u, binary32, IEEE division.
__device__ __forceinline__ float swiglu_f32(float g, float u) {
    const float d = __fadd_rn(1.0f, exp_f32_cw(-g));
    return __fmul_rn(__fdiv_rn(g, d), u);
}

constexpr int kSwigluThreads = 256;

__device__ __forceinline__ float block_max_f32(float v, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    v = lane < kSwigluThreads / 32 ? red[lane] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// One CTA per row of U [rows, 2I] (gate in [0, I), up in [I, 2I)); rows at
// or beyond offsets[E] (when offsets is given) are not routed and skipped.
// VPT float4 groups per thread stay in registers between the amax and the
// quantize pass (I <= 1024 * VPT, I % 4 == 0). Output: codes [rows, I] as
// int8, or as fp16 (the tensor-core operand), and the scales sh [rows]; or,
// kHOnly, h itself as FP32 [rows, I].
template <int VPT, int kOut>   // kOut: 0 int8 codes, 1 fp16 codes, 2 h (FP32)
__global__ void __launch_bounds__(kSwigluThreads)
swiglu_quant_kernel(const float *__restrict__ U, int I, const int32_t *__restrict__ offsets,
                    int E, void *__restrict__ out, float *__restrict__ sh) {
    griddep_launch_dependents();
    griddep_wait();   // U comes from the GEMM launched before
    const int64_t row = blockIdx.x;
    if (offsets != nullptr && row >= offsets[E]) return;
    __shared__ float red[kSwigluThreads / 32];
    const float4 *g4 = reinterpret_cast<const float4 *>(U + row * 2 * I);
    const float4 *u4 = reinterpret_cast<const float4 *>(U + row * 2 * I + I);
    const int nv = I >> 2;
    float4 h[VPT];
    float m = 0.0f;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int idx = threadIdx.x + v * kSwigluThreads;
        if (idx < nv) {
            const float4 g = __ldcs(g4 + idx), u = __ldcs(u4 + idx);
            h[v] = make_float4(swiglu_f32(g.x, u.x), swiglu_f32(g.y, u.y), swiglu_f32(g.z, u.z),
                               swiglu_f32(g.w, u.w));
        } else {
            h[v] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
        m = fmaxf(m, fmaxf(fmaxf(fabsf(h[v].x), fabsf(h[v].y)), fmaxf(fabsf(h[v].z), fabsf(h[v].w))));
    }
    if constexpr (kOut == 2) {
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int idx = threadIdx.x + v * kSwigluThreads;
            if (idx < nv) reinterpret_cast<float4 *>(static_cast<float *>(out) + row * I)[idx] = h[v];
        }
        return;
    }
    m = block_max_f32(m, red);
    const float s = __fdiv_rn(m, 127.0f);
    const bool fast = s >= 1.17549435e-38f;   // normal scale: 1/s is finite
    const float rcp = fast ? __frcp_rn(s) : 0.0f;
    if (threadIdx.x == 0) sh[row] = s;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int idx = threadIdx.x + v * kSwigluThreads;
        if (idx >= nv) continue;
        const float x[4] = {h[v].x, h[v].y, h[v].z, h[v].w};
        int q[4];
#pragma unroll
        for (int c = 0; c < 4; ++c)
            q[c] = s == 0.0f ? 0 : (fast ? quantize_fast(x[c], s, rcp) : quantize_exact(x[c], s));
        const uint32_t packed = pack4(q[0], q[1], q[2], q[3]);
        if constexpr (kOut == 1) {
            uint2 hh;
            i8x4_to_f16x4(packed, hh.x, hh.y);
            reinterpret_cast<uint2 *>(static_cast<__half *>(out) + row * I)[idx] = hh;
        } else {
            reinterpret_cast<uint32_t *>(static_cast<int8_t *>(out) + row * I)[idx] = packed;
        }
    }
}

// --------------------------------------------------------- weighted un-permute
constexpr int kUnpermThreads = 256;
constexpr int kMaxTopK = 64;

// One CTA per token t: y[t, n] = sum_j w[t, j] * D[row_of[t, j], n] (FP32, j in
// order, fma), skipping unrouted entries; BF16 (round to nearest even) or
// FP32 output. H % 4 == 0.
__global__ void __launch_bounds__(kUnpermThreads)
moe_unpermute_kernel(const float *__restrict__ D, const int32_t *__restrict__ row_of,
                     const float *__restrict__ w, int k, int H, void *__restrict__ y,
                     int out_fp32) {
    griddep_launch_dependents();
    griddep_wait();   // D comes from the GEMM launched before
    __shared__ int s_row[kMaxTopK];
    __shared__ float s_w[kMaxTopK];
    const int64_t t = blockIdx.x;
    for (int j = threadIdx.x; j < k; j += kUnpermThreads) {
        s_row[j] = row_of[t * k + j];
        s_w[j] = w[t * k + j];
    }
    __syncthreads();
    const int nv = H >> 2;
    for (int v = threadIdx.x; v < nv; v += kUnpermThreads) {
        float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        for (int j = 0; j < k; ++j) {
            const int r = s_row[j];
            if (r < 0) continue;
            const float wj = s_w[j];
            const float4 d = __ldcs(reinterpret_cast<const float4 *>(D + static_cast<int64_t>(r) * H) + v);
            acc.x = fmaf(wj, d.x, acc.x);
            acc.y = fmaf(wj, d.y, acc.y);
            acc.z = fmaf(wj, d.z, acc.z);
            acc.w = fmaf(wj, d.w, acc.w);
        }
        if (out_fp32) {
            reinterpret_cast<float4 *>(static_cast<float *>(y) + t * H)[v] = acc;
        } else {
            const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
            const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
            uint2 o;
            o.x = *reinterpret_cast<const uint32_t *>(&lo);
            o.y = *reinterpret_cast<const uint32_t *>(&hi);
            reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(y) + t * H)[v] = o;
        }
    }
}

template <typename... Params, typename... Args>
cudaError_t launch_pdl_moe(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
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

template <int kOut>
cudaError_t launch_swiglu(const float *U, int64_t rows, int64_t I, const int32_t *offsets,
                          int64_t E, void *out, float *sh, cudaStream_t stream) {
    const dim3 grid(static_cast<unsigned>(rows)), block(kSwigluThreads);
    const int i = static_cast<int>(I), e = static_cast<int>(E);
    const int nv = i / 4;
    if (nv <= kSwigluThreads * 1)
        return launch_pdl_moe(swiglu_quant_kernel<1, kOut>, grid, block, 0, stream, U, i, offsets,
                              e, out, sh);
    if (nv <= kSwigluThreads * 2)
        return launch_pdl_moe(swiglu_quant_kernel<2, kOut>, grid, block, 0, stream, U, i, offsets,
                              e, out, sh);
    if (nv <= kSwigluThreads * 4)
        return launch_pdl_moe(swiglu_quant_kernel<4, kOut>, grid, block, 0, stream, U, i, offsets,
                              e, out, sh);
    return launch_pdl_moe(swiglu_quant_kernel<8, kOut>, grid, block, 0, stream, U, i, offsets, e,
                          out, sh);
}

}  // namespace

cudaError_t launch_moe_route(const int32_t *ids, int64_t T, int64_t k, int64_t E, int32_t *offsets,
                             int32_t *row_of, int32_t *token_of_row, int32_t *pair_of_row,
                             cudaStream_t stream) {
    const size_t smem = static_cast<size_t>(kRouteWarps * E + E + 1) * sizeof(int);
    static int attr_done[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        e = cudaFuncSetAttribute(moe_route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>((kRouteWarps * kMaxExperts + kMaxExperts + 1) *
                                                  sizeof(int)));
        if (e != cudaSuccess) return e;
        attr_done[dev] = 1;
    }
    return launch_pdl_moe(moe_route_kernel, dim3(1), dim3(kRouteThreads), smem, stream, ids,
                          static_cast<int>(T * k), static_cast<int>(k), static_cast<int>(E),
                          offsets, row_of, token_of_row, pair_of_row);
}

cudaError_t launch_swiglu_quant(const float *U, int64_t rows, int64_t I, const int32_t *offsets,
                                int64_t E, void *out, int out_kind, float *sh,
                                cudaStream_t stream) {
    if (out_kind == 0) return launch_swiglu<0>(U, rows, I, offsets, E, out, sh, stream);
    if (out_kind == 1) return launch_swiglu<1>(U, rows, I, offsets, E, out, sh, stream);
    return launch_swiglu<2>(U, rows, I, offsets, E, out, sh, stream);
}

cudaError_t launch_moe_unpermute(const float *D, const int32_t *row_of, const float *w, int64_t T,
                                 int64_t k, int64_t H, void *y, bool out_fp32,
                                 cudaStream_t stream) {
    return launch_pdl_moe(moe_unpermute_kernel, dim3(static_cast<unsigned>(T)),
                          dim3(kUnpermThreads), 0, stream, D, row_of, w, static_cast<int>(k),
                          static_cast<int>(H), y, out_fp32 ? 1 : 0);
}

}  // namespace w8a8
