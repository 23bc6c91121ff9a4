// Rate probes of the integer-exact MMA paths this library uses on sm_103a
// (diagnostics; no counterpart on the source pages). The benchmark times them
// with CUDA events to report the peak of the arithmetic the GEMMs actually
// run, next to the measured dense bf16 peak:
//  * tcgen05.mma kind::f16 (fp16 operands holding exact int8 integers, FP32
//    accumulate), M = 128 weight rows, A from tensor memory, B (tokens) from
//    shared memory with the 128-byte swizzle, N token columns, K = 16 per
//    instruction: the instruction of w8a8_gemm_narrow_kernel. `chains`
//    independent accumulators take turns, reading the same A and B operands
//    (distinct = 0) or each its own (distinct = 1);
//  * dp4a (four int8 products summed into an int32): the CUDA-core GEMV.
// The operands are zeros; timing does not depend on the values.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace w8a8 {
namespace {

// B takes up to 256 rows x 128 B; the rest only keeps a second CTA off the SM
// (one CTA per SM holds all 512 tensor-memory columns).
constexpr int kProbeSmemBytes = 128 * 1024;

__global__ void __launch_bounds__(128, 1)
probe_tc_kernel(int n, int chains, int distinct, long long steps, unsigned long long *err) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sB = (raw + 1023u) & ~1023u;
    uint8_t *b_ptr = smem_raw + (sB - raw);
    for (int i = threadIdx.x; i < 256 * 128 / 16; i += blockDim.x)
        reinterpret_cast<uint4 *>(b_ptr)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        s_abort = 0;
        fence_mbarrier_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&s_tmem), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = s_tmem;
    {
        // each warp zeroes its quarter of the lanes of the A operand columns
        uint32_t z[16] = {0};
        const uint32_t lane_base = tb + ((static_cast<uint32_t>(warp) * 32u) << 16);
#pragma unroll
        for (int c = 0; c < 256; c += 16) tmem_st_16cols(lane_base + 256 + c, z);
        tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0) {
        const uint32_t idesc = idesc_f16_f32(128, static_cast<uint32_t>(n));
        const uint64_t b0 = smem_desc_sw128(sB);
        for (long long s = 0; s < steps; ++s) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                for (int c = 0; c < chains; ++c) {
                    // distinct: chain c reads its own A columns and B rows
                    const uint32_t a_off = distinct ? static_cast<uint32_t>(c * 64) : 0u;
                    const uint64_t b_off = distinct ? static_cast<uint64_t>((c * n * 128) >> 4) : 0u;
                    const uint64_t bdesc = b0 + b_off + static_cast<uint64_t>((kk & 3) * 2);
                    mma_f16_tmemA(tb + static_cast<uint32_t>(c * n), tb + 256 + a_off + kk * 8,
                                  bdesc, idesc, kk > 0 ? 1u : 0u);
                }
            }
        }
        mma_commit(smem_u32(&bar));
        mbar_wait(smem_u32(&bar), 0, &s_abort, err, ROLE_MMA, 9);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tb, 512);
}

__global__ void __launch_bounds__(512) probe_dp4a_kernel(long long iters, int *sink) {
    const int a = static_cast<int>(threadIdx.x * 0x01010101u);
    const int b = static_cast<int>(threadIdx.x ^ 0x12345678u);
    int c[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) c[u] = u;
    for (long long i = 0; i < iters; ++i) {
#pragma unroll
        for (int u = 0; u < 16; ++u) c[u] = __dp4a(a, b + u, c[u]);
    }
    int s = 0;
#pragma unroll
    for (int u = 0; u < 16; ++u) s += c[u];
    if (s == 0x7FFFFFFF) *sink = s;   // keeps the loop; never true in practice
}

__device__ int g_probe_sink;

}  // namespace

cudaError_t launch_probe_tc(int n, int chains, int distinct, long long steps, int num_sms,
                            cudaStream_t stream) {
    static int attr_done[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        e = cudaFuncSetAttribute(probe_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kProbeSmemBytes);
        if (e != cudaSuccess) return e;
        attr_done[dev] = 1;
    }
    unsigned long long *err = nullptr;
    e = device_error_word(&err);
    if (e != cudaSuccess) return e;
    probe_tc_kernel<<<num_sms, 128, kProbeSmemBytes, stream>>>(n, chains, distinct, steps, err);
    return cudaGetLastError();
}

cudaError_t launch_probe_dp4a(long long iters, int num_sms, cudaStream_t stream) {
    int *sink = nullptr;
    cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void **>(&sink), g_probe_sink);
    if (e != cudaSuccess) return e;
    probe_dp4a_kernel<<<num_sms * 4, 512, 0, stream>>>(iters, sink);
    return cudaGetLastError();
}

}  // namespace w8a8
