// Internal declarations shared by the translation units of libw8a8 (host side).
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace w8a8 {

cudaError_t launch_quant_act(const uint16_t *a, int64_t M, int64_t K, int64_t lda, int8_t *qa,
                             int64_t ldq, float *sa, cudaStream_t stream);

cudaError_t launch_quant_weight(const float *w, int64_t N, int64_t K, int8_t *qw, float *sw,
                                cudaStream_t stream);

// int8 codes [rows, K] (row stride ldq) -> fp16 codes [rows, K] in `out`.
cudaError_t launch_widen_codes(const int8_t *q, int64_t rows, int64_t K, int64_t ldq, void *out,
                               int num_sms, cudaStream_t stream);

struct GemmProblem {
    const float *sa;          // [R]
    const float *sw;          // [E*N, G]
    const int8_t *qw;         // [E*N, K]
    const void *x16;          // [R, K] fp16 copy of the int8 activation codes (staging)
    const int32_t *offsets;   // [E+1] device, or nullptr for one dense segment [0, R)
    void *y;                  // [R, N]
    int32_t *debug_partials;  // nullable [R, N, G]
    int64_t R, E, N, K;
    bool out_fp32;
    int grouped_batch_rows = 64;  // token rows per MMA batch for grouped calls (32..128)
};

// Maximum number of experts a grouped call may have.
constexpr int kMaxExperts = 1024;

cudaError_t launch_gemm(const GemmProblem &p, int num_sms, cudaStream_t stream);

// Device error word of the GEMM kernel (read/clear; synchronising).
cudaError_t read_device_error(unsigned long long *value, bool clear);

// Per-device properties cached on first use.
struct DeviceInfo {
    int device = -1;
    int cc_major = 0, cc_minor = 0;
    int num_sms = 0;
};
cudaError_t current_device_info(DeviceInfo *out);

}  // namespace w8a8
