// C ABI of libw8a8 (declared in include/w8a8.h): argument validation,
// device capability check, workspace sizing and dispatch to the kernels.
// No call allocates device memory, synchronises the host or reads device data.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/w8a8.h"
#include "internal.h"

namespace w8a8 {

cudaError_t current_device_info(DeviceInfo *out) {
    static DeviceInfo cache[64];
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev].device != dev) {
        DeviceInfo d;
        d.device = dev;
        if ((e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) !=
                cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) !=
                cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev)) !=
                cudaSuccess)
            return e;
        cache[dev] = d;
    }
    *out = cache[dev];
    return cudaSuccess;
}

}  // namespace w8a8

namespace {

constexpr int64_t kMaxElems = (int64_t(1) << 31) - 1;
constexpr size_t kWsAlign = 256;

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

w8a8_status check_device(w8a8::DeviceInfo *info) {
    if (w8a8::current_device_info(info) != cudaSuccess) return W8A8_ERR_CUDA;
    if (info->cc_major != 10 || info->cc_minor != 3) return W8A8_ERR_UNSUPPORTED;
    return W8A8_OK;
}

w8a8_status from_cuda(cudaError_t e) { return e == cudaSuccess ? W8A8_OK : W8A8_ERR_CUDA; }

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Workspace: fp16 staging copy of the int8 activation codes [rows, K] (the
// tensor-core operand), rounded up to 256 bytes.
size_t staging_bytes(int64_t rows, int64_t K) {
    if (rows <= 0 || K <= 0) return 0;
    return round_up(static_cast<size_t>(rows) * static_cast<size_t>(K) * 2, kWsAlign);
}

// Shared validation of the GEMM operands; E == 1 with offsets == nullptr is dense.
w8a8_status check_gemm(const int8_t *qa, const float *sa, const void *offsets, const int8_t *qw,
                       const float *sw, const void *y, int64_t R, int64_t E, int64_t N,
                       int64_t K, bool grouped, void *workspace, size_t workspace_bytes) {
    if (R < 0 || N <= 0 || K <= 0 || E <= 0) return W8A8_ERR_INVALID_ARG;
    if (K % W8A8_GROUP != 0) return W8A8_ERR_INVALID_ARG;
    if (grouped && E > w8a8::kMaxExperts) return W8A8_ERR_INVALID_ARG;
    if (R > kMaxElems / K || E * N > kMaxElems / K || R > kMaxElems / N) return W8A8_ERR_INVALID_ARG;
    if (R == 0) return W8A8_OK;
    if (!qa || !sa || !qw || !sw || !y || (grouped && !offsets)) return W8A8_ERR_INVALID_ARG;
    if (!aligned(qa, 16) || !aligned(qw, 16) || !aligned(sa, 4) || !aligned(sw, 4) ||
        !aligned(y, 4) || (offsets && !aligned(offsets, 4)))
        return W8A8_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < staging_bytes(R, K) || !aligned(workspace, kWsAlign))
        return W8A8_ERR_WORKSPACE;
    return W8A8_OK;
}

// Full workspace: the staging copy, then (dense calls of 5..64 token rows)
// the stream-K split area at the next 256-byte boundary.
size_t workspace_bytes_for(int64_t R, int64_t K, bool grouped) {
    if (R <= 0) return 0;
    return staging_bytes(R, K) + round_up(w8a8::sk_area_bytes(R, grouped), kWsAlign);
}

w8a8_status run_gemm(const int8_t *qa, const float *sa, const int32_t *offsets, const int8_t *qw,
                     const float *sw, void *y, w8a8_dtype y_dtype, int64_t R, int64_t E,
                     int64_t N, int64_t K, int32_t *dbg, void *workspace, size_t workspace_bytes,
                     w8a8_stream_t stream, int sw_block_rows = 1) {
    w8a8::DeviceInfo info;
    w8a8_status st = check_device(&info);
    if (st != W8A8_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool grouped = offsets != nullptr;
    w8a8::GemmProblem p;
    // The split area is optional: with a workspace that only holds the
    // staging copy, tiles are never split across CTAs.
    const size_t stage = staging_bytes(R, K);
    if (w8a8::sk_area_bytes(R, grouped) > 0 &&
        workspace_bytes >= workspace_bytes_for(R, K, grouped)) {
        unsigned char *area = static_cast<unsigned char *>(workspace) + stage;
        p.sk_cnt = reinterpret_cast<int *>(area);
        p.sk_part = reinterpret_cast<float *>(area + w8a8::sk_counter_bytes());
        p.sk_ld = static_cast<int>(R);
    }
    cudaError_t e = cudaSuccess;
    if (!w8a8::uses_gemv(R, grouped)) {
        // The tensor-core path reads an fp16 copy of the codes; the kernel that
        // writes it also resets the split counters. (The CUDA-core path reads
        // the int8 codes directly.)
        e = w8a8::launch_widen_codes(qa, R, K, K, workspace, info.num_sms, s, p.sk_cnt,
                                     p.sk_cnt != nullptr ? 2 * w8a8::kSkMaxCtas : 0);
    }
    if (e != cudaSuccess) return W8A8_ERR_CUDA;
    p.qa = qa;
    p.sa = sa;
    p.sw = sw;
    p.qw = qw;
    p.x16 = workspace;
    p.offsets = offsets;
    p.y = y;
    p.debug_partials = dbg;
    p.R = R;
    p.E = E;
    p.N = N;
    p.K = K;
    p.out_fp32 = (y_dtype == W8A8_FP32);
    p.sw_block_rows = sw_block_rows;
    return from_cuda(w8a8::launch_gemm(p, info.num_sms, s));
}

// ---------------------------------------------------------------------------
// Fused quantizer + GEMM (w8a8_linear, w8a8_grouped_linear). Workspace: the
// codes [R, K] (int8 for the CUDA-core GEMV, else fp16 for the tensor-core
// GEMM, M*K*2 bytes either way), the token scales [R], then the optional
// split area. The quantizer writes the operand the GEMM reads, so the
// tensor-core path needs no staging kernel.
size_t linear_scales_offset(int64_t R, int64_t K) { return staging_bytes(R, K); }
size_t linear_required_bytes(int64_t R, int64_t K) {
    if (R <= 0) return 0;
    return staging_bytes(R, K) + round_up(static_cast<size_t>(R) * 4, kWsAlign);
}
size_t linear_bytes_for(int64_t R, int64_t K, bool grouped) {
    if (R <= 0) return 0;
    return linear_required_bytes(R, K) + round_up(w8a8::sk_area_bytes(R, grouped), kWsAlign);
}

w8a8_status check_linear(const void *a, int64_t lda, const void *offsets, const int8_t *qw,
                         const float *sw, const void *y, w8a8_dtype y_dtype, int64_t R, int64_t E,
                         int64_t N, int64_t K, bool grouped, void *workspace,
                         size_t workspace_bytes) {
    if (y_dtype != W8A8_BF16 && y_dtype != W8A8_FP32) return W8A8_ERR_INVALID_ARG;
    if (R < 0 || N <= 0 || K <= 0 || E <= 0 || lda < K) return W8A8_ERR_INVALID_ARG;
    if (K % W8A8_GROUP != 0) return W8A8_ERR_INVALID_ARG;
    if (grouped && E > w8a8::kMaxExperts) return W8A8_ERR_INVALID_ARG;
    if (R > kMaxElems / lda || E * N > kMaxElems / K || R > kMaxElems / N)
        return W8A8_ERR_INVALID_ARG;
    if (R == 0) return W8A8_OK;
    if (!a || !qw || !sw || !y || (grouped && !offsets)) return W8A8_ERR_INVALID_ARG;
    if (!aligned(a, 2) || !aligned(qw, 16) || !aligned(sw, 4) || !aligned(y, 4) ||
        (offsets && !aligned(offsets, 4)))
        return W8A8_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < linear_required_bytes(R, K) ||
        !aligned(workspace, kWsAlign))
        return W8A8_ERR_WORKSPACE;
    return W8A8_OK;
}

// RMSNorm in front of the quantizer of a linear call (null: none).
struct NormArg {
    const uint16_t *gamma;
    float eps;
};

w8a8_status run_linear(const void *a, int64_t lda, const int32_t *offsets, const int8_t *qw,
                       const float *sw, void *y, w8a8_dtype y_dtype, int64_t R, int64_t E,
                       int64_t N, int64_t K, void *workspace, size_t workspace_bytes,
                       w8a8_stream_t stream, int sw_block_rows = 1, bool pow2 = false,
                       const NormArg *norm = nullptr) {
    w8a8::DeviceInfo info;
    w8a8_status st = check_device(&info);
    if (st != W8A8_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool grouped = offsets != nullptr;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    float *sa = reinterpret_cast<float *>(ws + linear_scales_offset(R, K));
    w8a8::GemmProblem p;
    if (w8a8::sk_area_bytes(R, grouped) > 0 &&
        workspace_bytes >= linear_bytes_for(R, K, grouped)) {
        unsigned char *area = ws + linear_required_bytes(R, K);
        p.sk_cnt = reinterpret_cast<int *>(area);
        p.sk_part = reinterpret_cast<float *>(area + w8a8::sk_counter_bytes());
        p.sk_ld = static_cast<int>(R);
    }
    const uint16_t *a16 = static_cast<const uint16_t *>(a);
    cudaError_t e = cudaSuccess;
    if (norm != nullptr) {
        // RMSNorm and quantization in one kernel, then the GEMM
        const bool gemv = w8a8::uses_gemv(R, grouped);
        e = w8a8::launch_rmsnorm_quant(a16, R, K, lda, norm->gamma, norm->eps, gemv ? 0 : 1, ws, K,
                                       sa, gemv ? nullptr : p.sk_cnt,
                                       p.sk_cnt != nullptr ? 2 * w8a8::kSkMaxCtas : 0, pow2, s);
        p.qa = gemv ? reinterpret_cast<const int8_t *>(ws) : nullptr;
    } else if (w8a8::uses_gemv(R, grouped) && !pow2 &&
               w8a8::gemv_can_fuse_quant(R, K, lda, a)) {
        // one kernel: the GEMV quantizes its token rows itself
        p.act = a16;
        p.lda = lda;
        p.qa = nullptr;
    } else if (w8a8::uses_gemv(R, grouped)) {
        e = w8a8::launch_quant_act_ex(a16, R, K, lda, reinterpret_cast<int8_t *>(ws), K, sa, pow2,
                                      s);
        p.qa = reinterpret_cast<const int8_t *>(ws);
    } else {
        e = w8a8::launch_quant_act_f16_ex(a16, R, K, lda, ws, sa, p.sk_cnt,
                                          p.sk_cnt != nullptr ? 2 * w8a8::kSkMaxCtas : 0, pow2, s);
        p.qa = nullptr;   // the tensor-core GEMM reads only the fp16 codes
    }
    if (e != cudaSuccess) return W8A8_ERR_CUDA;
    p.sa = sa;
    p.sw = sw;
    p.qw = qw;
    p.x16 = ws;
    p.offsets = offsets;
    p.y = y;
    p.debug_partials = nullptr;
    p.R = R;
    p.E = E;
    p.N = N;
    p.K = K;
    p.out_fp32 = (y_dtype == W8A8_FP32);
    p.sw_block_rows = sw_block_rows;
    return from_cuda(w8a8::launch_gemm(p, info.num_sms, s));
}

// ---------------------------------------------------------------------------
// Built-in scratch for w8a8_gemm_noalloc: the fp16 staging copy of the
// activation codes lives in this fixed device array instead of a caller
// workspace. Every GPU that loads the library keeps it until the process
// exits; all calls on a device share it.
constexpr size_t kNoallocScratchBytes = W8A8_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of g_noalloc_scratch on the current device, looked up once
// per device (with that device current) and cached. In host code the symbol
// name is only a host-side handle, never a device address.
cudaError_t noalloc_scratch_ptr(void **out) {
    static void *ptrs[64] = {nullptr};
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (ptrs[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        ptrs[dev] = p;
    }
    *out = ptrs[dev];
    return cudaSuccess;
}

// ---------------------------------------------------------------------------
// MoE expert FFN (w8a8_moe_ffn): workspace layout, every part 256-byte aligned,
// n = T * k routed-row slots:
//   offsets [E+1] int32, row_of [n], token_of_row [n], pair_of_row [n] int32,
//   gate_up operand: fp16 codes [n, H] + token scales [n],
//   gate_up output U [n, 2I] FP32,
//   down operand: fp16 codes [n, I] + scales [n],
//   down output D [n, H] FP32.
struct FfnLayout {
    size_t offsets, row_of, tok, pair, x_up, sa_up, u, x_dn, sa_dn, d, total;
};

FfnLayout ffn_layout(int64_t T, int64_t k, int64_t H, int64_t I, int64_t E) {
    const size_t n = static_cast<size_t>(T) * static_cast<size_t>(k);
    FfnLayout L;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off += round_up(bytes, kWsAlign);
        return at;
    };
    L.offsets = take(static_cast<size_t>(E + 1) * 4);
    L.row_of = take(n * 4);
    L.tok = take(n * 4);
    L.pair = take(n * 4);
    L.x_up = take(n * static_cast<size_t>(H) * 2);
    L.sa_up = take(n * 4);
    L.u = take(n * static_cast<size_t>(2 * I) * 4);
    L.x_dn = take(n * static_cast<size_t>(I) * 2);
    L.sa_dn = take(n * 4);
    L.d = take(n * static_cast<size_t>(H) * 4);
    L.total = off;
    return L;
}

w8a8_status check_ffn_shape(int64_t T, int64_t k, int64_t H, int64_t I, int64_t E) {
    if (T < 0 || k < 1 || k > w8a8::kMoeMaxTopK || E < 1 || E > w8a8::kMaxExperts)
        return W8A8_ERR_INVALID_ARG;
    if (H <= 0 || I <= 0 || H % W8A8_GROUP != 0 || I % W8A8_GROUP != 0 || I > w8a8::kSwigluMaxI)
        return W8A8_ERR_INVALID_ARG;
    const int64_t n = T * k;
    if (T > kMaxElems / k || n > kMaxElems / H || n > kMaxElems / (2 * I) ||
        E * 2 * I > kMaxElems / H || E * H > kMaxElems / I)
        return W8A8_ERR_INVALID_ARG;
    return W8A8_OK;
}

}  // namespace

extern "C" {

int w8a8_version(void) { return 100; }

const char *w8a8_status_string(w8a8_status status) {
    switch (status) {
        case W8A8_OK: return "W8A8_OK";
        case W8A8_ERR_INVALID_ARG: return "W8A8_ERR_INVALID_ARG";
        case W8A8_ERR_UNSUPPORTED: return "W8A8_ERR_UNSUPPORTED";
        case W8A8_ERR_CUDA: return "W8A8_ERR_CUDA";
        case W8A8_ERR_WORKSPACE: return "W8A8_ERR_WORKSPACE";
        case W8A8_ERR_DEVICE_TIMEOUT: return "W8A8_ERR_DEVICE_TIMEOUT";
    }
    return "W8A8_UNKNOWN_STATUS";
}

w8a8_status w8a8_quant_act(const void *a_bf16, int64_t M, int64_t K, int64_t lda, int8_t *qa,
                           int64_t ldq, float *sa, w8a8_stream_t stream) {
    if (M < 0 || K <= 0 || lda < K || ldq < K) return W8A8_ERR_INVALID_ARG;
    if (M > kMaxElems / lda || M > kMaxElems / ldq || M > 0x7FFFFFFF) return W8A8_ERR_INVALID_ARG;
    if (M == 0) return W8A8_OK;
    if (!a_bf16 || !qa || !sa || !aligned(a_bf16, 2) || !aligned(sa, 4))
        return W8A8_ERR_INVALID_ARG;
    w8a8::DeviceInfo info;
    w8a8_status st = check_device(&info);
    if (st != W8A8_OK) return st;
    return from_cuda(w8a8::launch_quant_act(static_cast<const uint16_t *>(a_bf16), M, K, lda, qa,
                                            ldq, sa, reinterpret_cast<cudaStream_t>(stream)));
}

w8a8_status w8a8_quant_weight(const float *w, int64_t N, int64_t K, int8_t *qw, float *sw,
                              w8a8_stream_t stream) {
    if (N < 0 || K <= 0 || K % W8A8_GROUP != 0 || N > kMaxElems / K) return W8A8_ERR_INVALID_ARG;
    if (N == 0) return W8A8_OK;
    if (!w || !qw || !sw || !aligned(w, 16) || !aligned(qw, 4) || !aligned(sw, 4))
        return W8A8_ERR_INVALID_ARG;
    w8a8::DeviceInfo info;
    w8a8_status st = check_device(&info);
    if (st != W8A8_OK) return st;
    return from_cuda(
        w8a8::launch_quant_weight(w, N, K, qw, sw, reinterpret_cast<cudaStream_t>(stream)));
}

size_t w8a8_gemm_workspace_size(int64_t M, int64_t N, int64_t K) {
    (void)N;
    if (K <= 0) return 0;
    return workspace_bytes_for(M, K, false);
}

size_t w8a8_grouped_gemm_workspace_size(int64_t R, int64_t E, int64_t N, int64_t K) {
    (void)E;
    (void)N;
    if (K <= 0) return 0;
    return workspace_bytes_for(R, K, true);
}

w8a8_status w8a8_gemm(const int8_t *qa, const float *sa, const int8_t *qw, const float *sw,
                      void *y, w8a8_dtype y_dtype, int64_t M, int64_t N, int64_t K,
                      int32_t *debug_partials, void *workspace, size_t workspace_bytes,
                      w8a8_stream_t stream) {
    if (y_dtype != W8A8_BF16 && y_dtype != W8A8_FP32) return W8A8_ERR_INVALID_ARG;
    w8a8_status st = check_gemm(qa, sa, nullptr, qw, sw, y, M, 1, N, K, false, workspace,
                                workspace_bytes);
    if (st != W8A8_OK || M == 0) return st;
    if (debug_partials && !aligned(debug_partials, 4)) return W8A8_ERR_INVALID_ARG;
    return run_gemm(qa, sa, nullptr, qw, sw, y, y_dtype, M, 1, N, K, debug_partials, workspace,
                    workspace_bytes, stream);
}

w8a8_status w8a8_grouped_gemm(const int8_t *qa, const float *sa, const int32_t *offsets,
                              const int8_t *qw, const float *sw, void *y, w8a8_dtype y_dtype,
                              int64_t R, int64_t E, int64_t N, int64_t K,
                              int32_t *debug_partials, void *workspace, size_t workspace_bytes,
                              w8a8_stream_t stream) {
    if (y_dtype != W8A8_BF16 && y_dtype != W8A8_FP32) return W8A8_ERR_INVALID_ARG;
    w8a8_status st = check_gemm(qa, sa, offsets, qw, sw, y, R, E, N, K, true, workspace,
                                workspace_bytes);
    if (st != W8A8_OK || R == 0) return st;
    if (debug_partials && !aligned(debug_partials, 4)) return W8A8_ERR_INVALID_ARG;
    return run_gemm(qa, sa, offsets, qw, sw, y, y_dtype, R, E, N, K, debug_partials, workspace,
                    workspace_bytes, stream);
}

size_t w8a8_linear_workspace_size(int64_t M, int64_t N, int64_t K) {
    (void)N;
    if (K <= 0) return 0;
    return linear_bytes_for(M, K, false);
}

size_t w8a8_grouped_linear_workspace_size(int64_t R, int64_t E, int64_t N, int64_t K) {
    (void)E;
    (void)N;
    if (K <= 0) return 0;
    return linear_bytes_for(R, K, true);
}

w8a8_status w8a8_linear(const void *a_bf16, int64_t lda, const int8_t *qw, const float *sw,
                        void *y, w8a8_dtype y_dtype, int64_t M, int64_t N, int64_t K,
                        void *workspace, size_t workspace_bytes, w8a8_stream_t stream) {
    w8a8_status st = check_linear(a_bf16, lda, nullptr, qw, sw, y, y_dtype, M, 1, N, K, false,
                                  workspace, workspace_bytes);
    if (st != W8A8_OK || M == 0) return st;
    return run_linear(a_bf16, lda, nullptr, qw, sw, y, y_dtype, M, 1, N, K, workspace,
                      workspace_bytes, stream);
}

w8a8_status w8a8_grouped_linear(const void *a_bf16, int64_t lda, const int32_t *offsets,
                                const int8_t *qw, const float *sw, void *y, w8a8_dtype y_dtype,
                                int64_t R, int64_t E, int64_t N, int64_t K, void *workspace,
                                size_t workspace_bytes, w8a8_stream_t stream) {
    w8a8_status st = check_linear(a_bf16, lda, offsets, qw, sw, y, y_dtype, R, E, N, K, true,
                                  workspace, workspace_bytes);
    if (st != W8A8_OK || R == 0) return st;
    return run_linear(a_bf16, lda, offsets, qw, sw, y, y_dtype, R, E, N, K, workspace,
                      workspace_bytes, stream);
}

w8a8_status w8a8_gemm_noalloc(const int8_t *qa, const float *sa, const int8_t *qw,
                              const float *sw, void *y, w8a8_dtype y_dtype, int64_t M, int64_t N,
                              int64_t K, w8a8_stream_t stream) {
    if (y_dtype != W8A8_BF16 && y_dtype != W8A8_FP32) return W8A8_ERR_INVALID_ARG;
    if (M < 0 || N <= 0 || K <= 0 || K % W8A8_GROUP != 0) return W8A8_ERR_INVALID_ARG;
    if (M == 0) return W8A8_OK;
    // The staging copy needs M*K*2 bytes; larger problems do not fit the
    // built-in scratch and are refused (use w8a8_gemm with a workspace).
    if (M > kMaxElems / K || staging_bytes(M, K) > kNoallocScratchBytes) return W8A8_ERR_WORKSPACE;
    w8a8::DeviceInfo info;
    w8a8_status st = check_device(&info);
    if (st != W8A8_OK) return st;
    void *scratch = nullptr;
    if (noalloc_scratch_ptr(&scratch) != cudaSuccess) return W8A8_ERR_CUDA;
    return w8a8_gemm(qa, sa, qw, sw, y, y_dtype, M, N, K, nullptr, scratch, kNoallocScratchBytes,
                     stream);
}

w8a8_status w8a8_quant_act_ex(const void *a_bf16, int64_t M, int64_t K, int64_t lda,
                              int8_t *qa, int64_t ldq, float *sa, w8a8_scale_mode mode,
                              w8a8_stream_t stream) {
    if (mode != W8A8_SCALE_AMAX && mode != W8A8_SCALE_POW2) return W8A8_ERR_INVALID_ARG;
    if (M < 0 || K <= 0 || lda < K || ldq < K) return W8A8_ERR_INVALID_ARG;
    if (M > kMaxElems / lda || M > kMaxElems / ldq || M > 0x7FFFFFFF) return W8A8_ERR_INVALID_ARG;
    if (M == 0) return W8A8_OK;
    if (!a_bf16 || !qa || !sa || !aligned(a_bf16, 2) || !aligned(sa, 4))
        return W8A8_ERR_INVALID_ARG;
    w8a8::DeviceInfo info;
    w8a8_status st = check_device(&info);
    if (st != W8A8_OK) return st;
    return from_cuda(w8a8::launch_quant_act_ex(static_cast<const uint16_t *>(a_bf16), M, K, lda,
                                               qa, ldq, sa, mode == W8A8_SCALE_POW2,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

w8a8_status w8a8_quant_weight_ex(const float *w, int64_t N, int64_t K, int32_t block_rows,
                                 w8a8_scale_mode mode, int8_t *qw, float *sw,
                                 w8a8_stream_t stream) {
    if (mode != W8A8_SCALE_AMAX && mode != W8A8_SCALE_POW2) return W8A8_ERR_INVALID_ARG;
    if (block_rows != 1 && block_rows != 128) return W8A8_ERR_INVALID_ARG;
    if (N < 0 || K <= 0 || K % W8A8_GROUP != 0 || N > kMaxElems / K) return W8A8_ERR_INVALID_ARG;
    if (N == 0) return W8A8_OK;
    if (!w || !qw || !sw || !aligned(w, 16) || !aligned(qw, 4) || !aligned(sw, 4))
        return W8A8_ERR_INVALID_ARG;
    w8a8::DeviceInfo info;
    w8a8_status st = check_device(&info);
    if (st != W8A8_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (block_rows == 1 && mode == W8A8_SCALE_AMAX)
        return from_cuda(w8a8::launch_quant_weight(w, N, K, qw, sw, s));
    return from_cuda(w8a8::launch_quant_weight_blocks(w, N, K, block_rows,
                                                      mode == W8A8_SCALE_POW2, qw, sw, s));
}

w8a8_status w8a8_gemm_ex(const int8_t *qa, const float *sa, const int8_t *qw, const float *sw,
                         int32_t sw_block_rows, void *y, w8a8_dtype y_dtype, int64_t M, int64_t N,
                         int64_t K, int32_t *debug_partials, void *workspace,
                         size_t workspace_bytes, w8a8_stream_t stream) {
    if (sw_block_rows != 1 && sw_block_rows != 128) return W8A8_ERR_INVALID_ARG;
    if (y_dtype != W8A8_BF16 && y_dtype != W8A8_FP32) return W8A8_ERR_INVALID_ARG;
    w8a8_status st = check_gemm(qa, sa, nullptr, qw, sw, y, M, 1, N, K, false, workspace,
                                workspace_bytes);
    if (st != W8A8_OK || M == 0) return st;
    if (debug_partials && !aligned(debug_partials, 4)) return W8A8_ERR_INVALID_ARG;
    return run_gemm(qa, sa, nullptr, qw, sw, y, y_dtype, M, 1, N, K, debug_partials, workspace,
                    workspace_bytes, stream, sw_block_rows);
}

w8a8_status w8a8_grouped_gemm_ex(const int8_t *qa, const float *sa, const int32_t *offsets,
                                 const int8_t *qw, const float *sw, int32_t sw_block_rows,
                                 void *y, w8a8_dtype y_dtype, int64_t R, int64_t E, int64_t N,
                                 int64_t K, int32_t *debug_partials, void *workspace,
                                 size_t workspace_bytes, w8a8_stream_t stream) {
    if (sw_block_rows != 1 && sw_block_rows != 128) return W8A8_ERR_INVALID_ARG;
    if (y_dtype != W8A8_BF16 && y_dtype != W8A8_FP32) return W8A8_ERR_INVALID_ARG;
    w8a8_status st = check_gemm(qa, sa, offsets, qw, sw, y, R, E, N, K, true, workspace,
                                workspace_bytes);
    if (st != W8A8_OK || R == 0) return st;
    if (debug_partials && !aligned(debug_partials, 4)) return W8A8_ERR_INVALID_ARG;
    return run_gemm(qa, sa, offsets, qw, sw, y, y_dtype, R, E, N, K, debug_partials, workspace,
                    workspace_bytes, stream, sw_block_rows);
}

w8a8_status w8a8_linear_ex(const void *a_bf16, int64_t lda, w8a8_scale_mode act_mode,
                           const int8_t *qw, const float *sw, int32_t sw_block_rows, void *y,
                           w8a8_dtype y_dtype, int64_t M, int64_t N, int64_t K, void *workspace,
                           size_t workspace_bytes, w8a8_stream_t stream) {
    if (act_mode != W8A8_SCALE_AMAX && act_mode != W8A8_SCALE_POW2) return W8A8_ERR_INVALID_ARG;
    if (sw_block_rows != 1 && sw_block_rows != 128) return W8A8_ERR_INVALID_ARG;
    w8a8_status st = check_linear(a_bf16, lda, nullptr, qw, sw, y, y_dtype, M, 1, N, K, false,
                                  workspace, workspace_bytes);
    if (st != W8A8_OK || M == 0) return st;
    return run_linear(a_bf16, lda, nullptr, qw, sw, y, y_dtype, M, 1, N, K, workspace,
                      workspace_bytes, stream, sw_block_rows, act_mode == W8A8_SCALE_POW2);
}

// Weight-only INT8 with BF16 activations (no activation quantizer, no
// workspace): the tensor-core kernels read the activations directly.
static w8a8_status run_w8a16(const void *a_bf16, int64_t lda, const int32_t *offsets,
                             const int8_t *qw, const float *sw, int32_t sw_block_rows, void *y,
                             w8a8_dtype y_dtype, int64_t R, int64_t E, int64_t N, int64_t K,
                             w8a8_stream_t stream) {
    const bool grouped = offsets != nullptr;
    if (y_dtype != W8A8_BF16 && y_dtype != W8A8_FP32) return W8A8_ERR_INVALID_ARG;
    if (sw_block_rows != 1 && sw_block_rows != 128) return W8A8_ERR_INVALID_ARG;
    if (R < 0 || N <= 0 || K <= 0 || E <= 0 || K % W8A8_GROUP != 0 || lda < K || lda % 8 != 0)
        return W8A8_ERR_INVALID_ARG;
    if (grouped && E > w8a8::kMaxExperts) return W8A8_ERR_INVALID_ARG;
    if (R > kMaxElems / lda || E * N > kMaxElems / K || R > kMaxElems / N)
        return W8A8_ERR_INVALID_ARG;
    if (R == 0) return W8A8_OK;
    if (!a_bf16 || !qw || !sw || !y || (grouped && !offsets)) return W8A8_ERR_INVALID_ARG;
    if (!aligned(a_bf16, 16) || !aligned(qw, 16) || !aligned(sw, 4) || !aligned(y, 4) ||
        (offsets && !aligned(offsets, 4)))
        return W8A8_ERR_INVALID_ARG;
    w8a8::DeviceInfo info;
    w8a8_status st = check_device(&info);
    if (st != W8A8_OK) return st;
    w8a8::GemmProblem p;
    p.qa = nullptr;
    p.sa = nullptr;
    p.sw = sw;
    p.qw = qw;
    p.x16 = a_bf16;
    p.offsets = offsets;
    p.y = y;
    p.debug_partials = nullptr;
    p.R = R;
    p.E = E;
    p.N = N;
    p.K = K;
    p.out_fp32 = (y_dtype == W8A8_FP32);
    p.sw_block_rows = sw_block_rows;
    p.a16 = true;
    p.ldx = lda;
    return from_cuda(w8a8::launch_gemm(p, info.num_sms, reinterpret_cast<cudaStream_t>(stream)));
}

w8a8_status w8a8_w8a16_gemm(const void *a_bf16, int64_t lda, const int8_t *qw, const float *sw,
                            int32_t sw_block_rows, void *y, w8a8_dtype y_dtype, int64_t M,
                            int64_t N, int64_t K, w8a8_stream_t stream) {
    return run_w8a16(a_bf16, lda, nullptr, qw, sw, sw_block_rows, y, y_dtype, M, 1, N, K, stream);
}

w8a8_status w8a8_w8a16_grouped_gemm(const void *a_bf16, int64_t lda, const int32_t *offsets,
                                    const int8_t *qw, const float *sw, int32_t sw_block_rows,
                                    void *y, w8a8_dtype y_dtype, int64_t R, int64_t E, int64_t N,
                                    int64_t K, w8a8_stream_t stream) {
    if (!offsets && R > 0) return W8A8_ERR_INVALID_ARG;
    return run_w8a16(a_bf16, lda, offsets, qw, sw, sw_block_rows, y, y_dtype, R, E, N, K, stream);
}

w8a8_status w8a8_kv_quant(const void *x_bf16, int64_t n, int64_t head_dim,
                          const int32_t *dst_rows, int8_t *cache, float *scales,
                          w8a8_stream_t stream) {
    if (n < 0 || head_dim != w8a8::kAttnHeadDim || n > kMaxElems / head_dim)
        return W8A8_ERR_INVALID_ARG;
    if (n == 0) return W8A8_OK;
    if (!x_bf16 || !cache || !scales || !aligned(x_bf16, 8) || !aligned(cache, 4) ||
        !aligned(scales, 4) || !aligned(dst_rows, 4))
        return W8A8_ERR_INVALID_ARG;
    w8a8::DeviceInfo info;
    w8a8_status st = check_device(&info);
    if (st != W8A8_OK) return st;
    return from_cuda(w8a8::launch_kv_quant(static_cast<const uint16_t *>(x_bf16), n, dst_rows,
                                           cache, scales, reinterpret_cast<cudaStream_t>(stream)));
}

size_t w8a8_attention_decode_workspace_size(int64_t B, int64_t Hq, int64_t S_max,
                                            int64_t head_dim) {
    if (B <= 0 || Hq <= 0 || S_max <= 0 || head_dim != w8a8::kAttnHeadDim) return 0;
    return w8a8::attn_workspace_bytes(B, Hq, S_max);
}

static w8a8_status run_attention(const void *q_bf16, const void *kc, const float *ks,
                                 const void *vc, const float *vs, const int32_t *lens, int64_t B,
                                 int64_t Hq, int64_t Hkv, int64_t S_max, int64_t head_dim,
                                 float softmax_scale, void *out, w8a8_dtype out_dtype,
                                 void *workspace, size_t workspace_bytes, bool int8,
                                 w8a8_stream_t stream) {
    if (out_dtype != W8A8_BF16 && out_dtype != W8A8_FP32) return W8A8_ERR_INVALID_ARG;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || S_max <= 0 ||
        head_dim != w8a8::kAttnHeadDim)
        return W8A8_ERR_INVALID_ARG;
    const int64_t G = Hq / Hkv;
    if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return W8A8_ERR_INVALID_ARG;
    if (B > 65535 || Hkv > 65535 || S_max > (int64_t(1) << 24) ||
        B * Hkv > kMaxElems / (S_max * head_dim) || !(softmax_scale > 0.0f))
        return W8A8_ERR_INVALID_ARG;
    if (B == 0) return W8A8_OK;
    if (!q_bf16 || !kc || !vc || !lens || !out || (int8 && (!ks || !vs)))
        return W8A8_ERR_INVALID_ARG;
    if (!aligned(q_bf16, 2) || !aligned(kc, 16) || !aligned(vc, 16) || !aligned(ks, 4) ||
        !aligned(vs, 4) || !aligned(lens, 4) || !aligned(out, 4))
        return W8A8_ERR_INVALID_ARG;
    const size_t need = w8a8::attn_workspace_bytes(B, Hq, S_max);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 16)) return W8A8_ERR_WORKSPACE;
    w8a8::DeviceInfo info;
    w8a8_status st = check_device(&info);
    if (st != W8A8_OK) return st;
    w8a8::AttnProblem p;
    p.q = static_cast<const uint16_t *>(q_bf16);
    p.kc = kc;
    p.vc = vc;
    p.ks = ks;
    p.vs = vs;
    p.lens = lens;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.S_max = S_max;
    p.scale = softmax_scale;
    p.int8 = int8;
    p.out = out;
    p.out_fp32 = (out_dtype == W8A8_FP32);
    const int64_t nch = (S_max + 127) / 128;
    p.part_o = static_cast<float *>(workspace);
    p.part_ml = p.part_o + B * Hq * nch * head_dim;
    return from_cuda(w8a8::launch_attention_decode(p, reinterpret_cast<cudaStream_t>(stream)));
}

w8a8_status w8a8_attention_decode_int8kv(const void *q_bf16, const int8_t *k_cache,
                                         const float *k_scale, const int8_t *v_cache,
                                         const float *v_scale, const int32_t *lens, int64_t B,
                                         int64_t Hq, int64_t Hkv, int64_t S_max,
                                         int64_t head_dim, float softmax_scale, void *out,
                                         w8a8_dtype out_dtype, void *workspace,
                                         size_t workspace_bytes, w8a8_stream_t stream) {
    return run_attention(q_bf16, k_cache, k_scale, v_cache, v_scale, lens, B, Hq, Hkv, S_max,
                         head_dim, softmax_scale, out, out_dtype, workspace, workspace_bytes, true,
                         stream);
}

w8a8_status w8a8_attention_decode_bf16kv(const void *q_bf16, const void *k_cache,
                                         const void *v_cache, const int32_t *lens, int64_t B,
                                         int64_t Hq, int64_t Hkv, int64_t S_max,
                                         int64_t head_dim, float softmax_scale, void *out,
                                         w8a8_dtype out_dtype, void *workspace,
                                         size_t workspace_bytes, w8a8_stream_t stream) {
    return run_attention(q_bf16, k_cache, nullptr, v_cache, nullptr, lens, B, Hq, Hkv, S_max,
                         head_dim, softmax_scale, out, out_dtype, workspace, workspace_bytes,
                         false, stream);
}

namespace {
// Arguments shared by the RMSNorm entry points.
w8a8_status check_rmsnorm(const void *x, int64_t ldx, const void *gamma, float eps, int64_t M,
                          int64_t K) {
    if (M < 0 || K <= 0 || K % 8 != 0 || K > w8a8::kRmsNormMaxK || ldx < K || ldx % 8 != 0)
        return W8A8_ERR_INVALID_ARG;
    if (!(eps > 0.0f) || !std::isfinite(eps)) return W8A8_ERR_INVALID_ARG;
    if (M > kMaxElems / ldx || M > 0x7FFFFFFF) return W8A8_ERR_INVALID_ARG;
    if (M == 0) return W8A8_OK;
    if (!x || !gamma || !aligned(x, 16) || !aligned(gamma, 16)) return W8A8_ERR_INVALID_ARG;
    return W8A8_OK;
}
}  // namespace

w8a8_status w8a8_rmsnorm(const void *x_bf16, int64_t ldx, const void *gamma_bf16, float eps,
                         int64_t M, int64_t K, void *y_bf16, int64_t ldy, w8a8_stream_t stream) {
    w8a8_status st = check_rmsnorm(x_bf16, ldx, gamma_bf16, eps, M, K);
    if (st != W8A8_OK || M == 0) return st;
    if (!y_bf16 || !aligned(y_bf16, 16) || ldy < K || ldy % 8 != 0 || M > kMaxElems / ldy)
        return W8A8_ERR_INVALID_ARG;
    w8a8::DeviceInfo info;
    st = check_device(&info);
    if (st != W8A8_OK) return st;
    return from_cuda(w8a8::launch_rmsnorm_quant(
        static_cast<const uint16_t *>(x_bf16), M, K, ldx, static_cast<const uint16_t *>(gamma_bf16),
        eps, 2, y_bf16, ldy, nullptr, nullptr, 0, false, reinterpret_cast<cudaStream_t>(stream)));
}

w8a8_status w8a8_rmsnorm_quant(const void *x_bf16, int64_t ldx, const void *gamma_bf16, float eps,
                               w8a8_scale_mode mode, int64_t M, int64_t K, int8_t *qa,
                               int64_t ldq, float *sa, w8a8_stream_t stream) {
    if (mode != W8A8_SCALE_AMAX && mode != W8A8_SCALE_POW2) return W8A8_ERR_INVALID_ARG;
    w8a8_status st = check_rmsnorm(x_bf16, ldx, gamma_bf16, eps, M, K);
    if (st != W8A8_OK || M == 0) return st;
    if (!qa || !sa || !aligned(qa, 8) || !aligned(sa, 4) || ldq < K || ldq % 8 != 0 ||
        M > kMaxElems / ldq)
        return W8A8_ERR_INVALID_ARG;
    w8a8::DeviceInfo info;
    st = check_device(&info);
    if (st != W8A8_OK) return st;
    return from_cuda(w8a8::launch_rmsnorm_quant(
        static_cast<const uint16_t *>(x_bf16), M, K, ldx, static_cast<const uint16_t *>(gamma_bf16),
        eps, 0, qa, ldq, sa, nullptr, 0, mode == W8A8_SCALE_POW2,
        reinterpret_cast<cudaStream_t>(stream)));
}

w8a8_status w8a8_rmsnorm_linear(const void *x_bf16, int64_t ldx, const void *gamma_bf16, float eps,
                                const int8_t *qw, const float *sw, void *y, w8a8_dtype y_dtype,
                                int64_t M, int64_t N, int64_t K, void *workspace,
                                size_t workspace_bytes, w8a8_stream_t stream) {
    w8a8_status st = check_rmsnorm(x_bf16, ldx, gamma_bf16, eps, M, K);
    if (st != W8A8_OK) return st;
    st = check_linear(x_bf16, ldx, nullptr, qw, sw, y, y_dtype, M, 1, N, K, false, workspace,
                      workspace_bytes);
    if (st != W8A8_OK || M == 0) return st;
    const NormArg norm = {static_cast<const uint16_t *>(gamma_bf16), eps};
    return run_linear(x_bf16, ldx, nullptr, qw, sw, y, y_dtype, M, 1, N, K, workspace,
                      workspace_bytes, stream, 1, false, &norm);
}

w8a8_status w8a8_moe_route(const int32_t *topk_ids, int64_t T, int64_t k, int64_t E,
                           int32_t *offsets, int32_t *row_of, int32_t *token_of_row,
                           int32_t *pair_of_row, w8a8_stream_t stream) {
    if (T < 0 || k < 1 || E < 1 || E > w8a8::kMaxExperts || T > kMaxElems / k)
        return W8A8_ERR_INVALID_ARG;
    if (!offsets) return W8A8_ERR_INVALID_ARG;
    if (T > 0 && (!topk_ids || !row_of || !token_of_row || !pair_of_row))
        return W8A8_ERR_INVALID_ARG;
    if (!aligned(topk_ids, 4) || !aligned(offsets, 4) || !aligned(row_of, 4) ||
        !aligned(token_of_row, 4) || !aligned(pair_of_row, 4))
        return W8A8_ERR_INVALID_ARG;
    w8a8::DeviceInfo info;
    w8a8_status st = check_device(&info);
    if (st != W8A8_OK) return st;
    return from_cuda(w8a8::launch_moe_route(topk_ids, T, k, E, offsets, row_of, token_of_row,
                                            pair_of_row, reinterpret_cast<cudaStream_t>(stream)));
}

w8a8_status w8a8_quant_act_rows(const void *a_bf16, int64_t lda, const int32_t *src_rows,
                                int64_t rows, int64_t K, int8_t *qa, float *sa,
                                w8a8_stream_t stream) {
    if (rows < 0 || K <= 0 || lda < K || rows > kMaxElems / K) return W8A8_ERR_INVALID_ARG;
    if (rows == 0) return W8A8_OK;
    if (!a_bf16 || !src_rows || !qa || !sa || !aligned(a_bf16, 2) || !aligned(src_rows, 4) ||
        !aligned(sa, 4))
        return W8A8_ERR_INVALID_ARG;
    w8a8::DeviceInfo info;
    w8a8_status st = check_device(&info);
    if (st != W8A8_OK) return st;
    return from_cuda(w8a8::launch_quant_act_rows(static_cast<const uint16_t *>(a_bf16), rows, K,
                                                 lda, src_rows, qa, false, sa,
                                                 reinterpret_cast<cudaStream_t>(stream)));
}

w8a8_status w8a8_swiglu_quant(const float *U, int64_t rows, int64_t I, const int32_t *offsets,
                              int64_t E, int8_t *qh, float *sh, w8a8_stream_t stream) {
    if (rows < 0 || I <= 0 || I % 4 != 0 || I > w8a8::kSwigluMaxI || rows > kMaxElems / (2 * I))
        return W8A8_ERR_INVALID_ARG;
    if (offsets && (E < 1 || E > w8a8::kMaxExperts)) return W8A8_ERR_INVALID_ARG;
    if (rows == 0) return W8A8_OK;
    if (!U || !qh || !sh || !aligned(U, 16) || !aligned(qh, 4) || !aligned(sh, 4) ||
        !aligned(offsets, 4))
        return W8A8_ERR_INVALID_ARG;
    w8a8::DeviceInfo info;
    w8a8_status st = check_device(&info);
    if (st != W8A8_OK) return st;
    return from_cuda(w8a8::launch_swiglu_quant(U, rows, I, offsets, offsets ? E : 0, qh, 0, sh,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

w8a8_status w8a8_swiglu(const float *U, int64_t rows, int64_t I, float *h, w8a8_stream_t stream) {
    if (rows < 0 || I <= 0 || I % 4 != 0 || I > w8a8::kSwigluMaxI || rows > kMaxElems / (2 * I))
        return W8A8_ERR_INVALID_ARG;
    if (rows == 0) return W8A8_OK;
    if (!U || !h || !aligned(U, 16) || !aligned(h, 16)) return W8A8_ERR_INVALID_ARG;
    w8a8::DeviceInfo info;
    w8a8_status st = check_device(&info);
    if (st != W8A8_OK) return st;
    return from_cuda(w8a8::launch_swiglu_quant(U, rows, I, nullptr, 0, h, 2, nullptr,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

w8a8_status w8a8_moe_unpermute(const float *D, const int32_t *row_of, const float *topk_w,
                               int64_t T, int64_t k, int64_t H, void *y, w8a8_dtype y_dtype,
                               w8a8_stream_t stream) {
    if (y_dtype != W8A8_BF16 && y_dtype != W8A8_FP32) return W8A8_ERR_INVALID_ARG;
    if (T < 0 || k < 1 || k > w8a8::kMoeMaxTopK || H <= 0 || H % 4 != 0 || T > kMaxElems / H ||
        T > kMaxElems / k)
        return W8A8_ERR_INVALID_ARG;
    if (T == 0) return W8A8_OK;
    if (!D || !row_of || !topk_w || !y || !aligned(D, 16) || !aligned(row_of, 4) ||
        !aligned(topk_w, 4) || !aligned(y, 16))
        return W8A8_ERR_INVALID_ARG;
    w8a8::DeviceInfo info;
    w8a8_status st = check_device(&info);
    if (st != W8A8_OK) return st;
    return from_cuda(w8a8::launch_moe_unpermute(D, row_of, topk_w, T, k, H, y,
                                                y_dtype == W8A8_FP32,
                                                reinterpret_cast<cudaStream_t>(stream)));
}

size_t w8a8_moe_ffn_workspace_size(int64_t T, int64_t k, int64_t H, int64_t I, int64_t E) {
    if (check_ffn_shape(T, k, H, I, E) != W8A8_OK || T == 0) return 0;
    return ffn_layout(T, k, H, I, E).total;
}

w8a8_status w8a8_moe_ffn(const void *x_bf16, int64_t ldx, const int32_t *topk_ids,
                         const float *topk_w, int64_t T, int64_t k, int64_t H, int64_t I,
                         int64_t E, const int8_t *qw_up, const float *sw_up,
                         const int8_t *qw_down, const float *sw_down, void *y, w8a8_dtype y_dtype,
                         void *workspace, size_t workspace_bytes, w8a8_stream_t stream) {
    if (y_dtype != W8A8_BF16 && y_dtype != W8A8_FP32) return W8A8_ERR_INVALID_ARG;
    w8a8_status st = check_ffn_shape(T, k, H, I, E);
    if (st != W8A8_OK) return st;
    if (ldx < H || T > kMaxElems / ldx) return W8A8_ERR_INVALID_ARG;
    if (T == 0) return W8A8_OK;
    if (!x_bf16 || !topk_ids || !topk_w || !qw_up || !sw_up || !qw_down || !sw_down || !y)
        return W8A8_ERR_INVALID_ARG;
    if (!aligned(x_bf16, 2) || !aligned(topk_ids, 4) || !aligned(topk_w, 4) ||
        !aligned(qw_up, 16) || !aligned(qw_down, 16) || !aligned(sw_up, 4) ||
        !aligned(sw_down, 4) || !aligned(y, 16))
        return W8A8_ERR_INVALID_ARG;
    const FfnLayout L = ffn_layout(T, k, H, I, E);
    if (!workspace || workspace_bytes < L.total || !aligned(workspace, kWsAlign))
        return W8A8_ERR_WORKSPACE;
    w8a8::DeviceInfo info;
    st = check_device(&info);
    if (st != W8A8_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    int32_t *offsets = reinterpret_cast<int32_t *>(ws + L.offsets);
    int32_t *row_of = reinterpret_cast<int32_t *>(ws + L.row_of);
    int32_t *tok = reinterpret_cast<int32_t *>(ws + L.tok);
    int32_t *pair = reinterpret_cast<int32_t *>(ws + L.pair);
    float *sa_up = reinterpret_cast<float *>(ws + L.sa_up);
    float *U = reinterpret_cast<float *>(ws + L.u);
    float *sa_dn = reinterpret_cast<float *>(ws + L.sa_dn);
    float *D = reinterpret_cast<float *>(ws + L.d);
    const int64_t n = T * k;
    // 1. routing histogram -> offsets -> permutation (one CTA)
    cudaError_t e = w8a8::launch_moe_route(topk_ids, T, k, E, offsets, row_of, tok, pair, s);
    // 2. transfer + per-token quantization of the permuted token rows (fp16
    //    codes: the gate_up GEMM's operand)
    if (e == cudaSuccess)
        e = w8a8::launch_quant_act_rows(static_cast<const uint16_t *>(x_bf16), n, H, ldx, tok,
                                        ws + L.x_up, true, sa_up, s);
    // 3. gate_up grouped GEMM, FP32 output U [n, 2I]
    if (e == cudaSuccess) {
        w8a8::GemmProblem p;
        p.qa = nullptr;
        p.sa = sa_up;
        p.sw = sw_up;
        p.qw = qw_up;
        p.x16 = ws + L.x_up;
        p.offsets = offsets;
        p.y = U;
        p.debug_partials = nullptr;
        p.R = n;
        p.E = E;
        p.N = 2 * I;
        p.K = H;
        p.out_fp32 = true;
        e = w8a8::launch_gemm(p, info.num_sms, s);
    }
    // 4. SwiGLU + per-token requantization (fp16 codes: the down GEMM's operand)
    if (e == cudaSuccess)
        e = w8a8::launch_swiglu_quant(U, n, I, offsets, E, ws + L.x_dn, 1, sa_dn, s);
    // 5. down grouped GEMM, FP32 output D [n, H]
    if (e == cudaSuccess) {
        w8a8::GemmProblem p;
        p.qa = nullptr;
        p.sa = sa_dn;
        p.sw = sw_down;
        p.qw = qw_down;
        p.x16 = ws + L.x_dn;
        p.offsets = offsets;
        p.y = D;
        p.debug_partials = nullptr;
        p.R = n;
        p.E = E;
        p.N = H;
        p.K = I;
        p.out_fp32 = true;
        e = w8a8::launch_gemm(p, info.num_sms, s);
    }
    // 6. weighted un-permute into y [T, H]
    if (e == cudaSuccess)
        e = w8a8::launch_moe_unpermute(D, row_of, topk_w, T, k, H, y, y_dtype == W8A8_FP32, s);
    return from_cuda(e);
}

w8a8_status w8a8_selftest_wait_timeout(uint32_t limit_us, w8a8_stream_t stream) {
    if (limit_us == 0 || limit_us > 2000000u) return W8A8_ERR_INVALID_ARG;
    w8a8::DeviceInfo info;
    w8a8_status st = check_device(&info);
    if (st != W8A8_OK) return st;
    return from_cuda(w8a8::launch_selftest_wait(static_cast<unsigned long long>(limit_us) * 1000ull,
                                                reinterpret_cast<cudaStream_t>(stream)));
}

w8a8_status w8a8_probe_tc_rate(int32_t n, int32_t chains, int32_t distinct, int64_t steps,
                               int64_t *macs_out, w8a8_stream_t stream) {
    if (!macs_out || n < 16 || n > 256 || n % 16 != 0 || chains < 1 || chains > 4 ||
        chains * n > 256 || steps < 1 || steps > (int64_t(1) << 24))
        return W8A8_ERR_INVALID_ARG;
    w8a8::DeviceInfo info;
    w8a8_status st = check_device(&info);
    if (st != W8A8_OK) return st;
    *macs_out = int64_t(info.num_sms) * steps * 8 * chains * 128 * n * 16;
    return from_cuda(w8a8::launch_probe_tc(n, chains, distinct != 0 ? 1 : 0, steps, info.num_sms,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

w8a8_status w8a8_probe_dp4a_rate(int64_t iters, int64_t *macs_out, w8a8_stream_t stream) {
    if (!macs_out || iters < 1 || iters > (int64_t(1) << 26)) return W8A8_ERR_INVALID_ARG;
    w8a8::DeviceInfo info;
    w8a8_status st = check_device(&info);
    if (st != W8A8_OK) return st;
    *macs_out = int64_t(info.num_sms) * 4 * 512 * iters * 16 * 4;
    return from_cuda(w8a8::launch_probe_dp4a(iters, info.num_sms,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

w8a8_status w8a8_device_error(uint64_t *code_out, int clear) {
    if (!code_out) return W8A8_ERR_INVALID_ARG;
    unsigned long long v = 0;
    if (w8a8::read_device_error(&v, clear != 0) != cudaSuccess) return W8A8_ERR_CUDA;
    *code_out = v;
    return v ? W8A8_ERR_DEVICE_TIMEOUT : W8A8_OK;
}

}  // extern "C"
