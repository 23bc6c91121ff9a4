// C ABI of libw8a8 (declared in include/w8a8.h): argument validation,
// device capability check, workspace sizing and dispatch to the kernels.
// No call allocates device memory, synchronises the host or reads device data.
#include <cuda_runtime.h>

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
                     w8a8_stream_t stream) {
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

w8a8_status run_linear(const void *a, int64_t lda, const int32_t *offsets, const int8_t *qw,
                       const float *sw, void *y, w8a8_dtype y_dtype, int64_t R, int64_t E,
                       int64_t N, int64_t K, void *workspace, size_t workspace_bytes,
                       w8a8_stream_t stream) {
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
    if (w8a8::uses_gemv(R, grouped) && w8a8::gemv_can_fuse_quant(R, K, lda, a)) {
        // one kernel: the GEMV quantizes its token rows itself
        p.act = a16;
        p.lda = lda;
        p.qa = nullptr;
    } else if (w8a8::uses_gemv(R, grouped)) {
        e = w8a8::launch_quant_act(a16, R, K, lda, reinterpret_cast<int8_t *>(ws), K, sa, s);
        p.qa = reinterpret_cast<const int8_t *>(ws);
    } else {
        e = w8a8::launch_quant_act_f16(a16, R, K, lda, ws, sa, p.sk_cnt,
                                       p.sk_cnt != nullptr ? 2 * w8a8::kSkMaxCtas : 0, s);
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

w8a8_status w8a8_selftest_wait_timeout(uint32_t limit_us, w8a8_stream_t stream) {
    if (limit_us == 0 || limit_us > 2000000u) return W8A8_ERR_INVALID_ARG;
    w8a8::DeviceInfo info;
    w8a8_status st = check_device(&info);
    if (st != W8A8_OK) return st;
    return from_cuda(w8a8::launch_selftest_wait(static_cast<unsigned long long>(limit_us) * 1000ull,
                                                reinterpret_cast<cudaStream_t>(stream)));
}

w8a8_status w8a8_probe_tc_rate(int32_t n, int32_t chains, int64_t steps, int64_t *macs_out,
                               w8a8_stream_t stream) {
    if (!macs_out || n < 16 || n > 256 || n % 16 != 0 || chains < 1 || chains * n > 256 ||
        steps < 1 || steps > (int64_t(1) << 24))
        return W8A8_ERR_INVALID_ARG;
    w8a8::DeviceInfo info;
    w8a8_status st = check_device(&info);
    if (st != W8A8_OK) return st;
    *macs_out = int64_t(info.num_sms) * steps * 8 * chains * 128 * n * 16;
    return from_cuda(w8a8::launch_probe_tc(n, chains, steps, info.num_sms,
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
