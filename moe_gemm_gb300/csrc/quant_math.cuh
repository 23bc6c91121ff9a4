// Per-token activation quantization arithmetic shared by the quantizer
// kernels and the GEMV that quantizes its own token rows: both must produce
// the same codes bit for bit (per-token scale s = amax/127, codes =
// round-half-even(x / s) clamped to [-127, 127]; "Deploying Hunyuan 770B in
// INT8 on domestic accelerators", §3.1).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace w8a8 {

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h) {
    return __uint_as_float(h << 16);
}

// round(x / s) with IEEE division and round-half-even, clamped to [-127, 127].
__device__ __forceinline__ int quantize_exact(float x, float s) {
    const int q = __float2int_rn(__fdiv_rn(x, s));
    return max(-127, min(127, q));
}

// Same result as quantize_exact(x, s) for a normal s > 0, computed with the
// reciprocal r = fl(1/s): y = fl(x*r) differs from the quotient x/s by at most
// 2^-23 * |x/s| <= 1.6e-5 (|x/s| <= 127.00001), and fl(x/s) differs from x/s
// by at most 0.8e-5. Unless y lies within 3e-5 of a half-integer, y and
// fl(x/s) round to the same integer; inside that window the exact division
// decides. So the codes are identical to round(fl(x/s)) in every case.
__device__ __forceinline__ int quantize_fast(float x, float s, float r) {
    const float y = x * r;
    const float yi = rintf(y);
    int q;
    if (fabsf(y - yi) >= 0.5f - 3.0e-5f)
        q = __float2int_rn(__fdiv_rn(x, s));
    else
        q = static_cast<int>(yi);
    return max(-127, min(127, q));
}

__device__ __forceinline__ uint32_t pack4(int a, int b, int c, int d) {
    return (static_cast<uint32_t>(a) & 0xFFu) | ((static_cast<uint32_t>(b) & 0xFFu) << 8) |
           ((static_cast<uint32_t>(c) & 0xFFu) << 16) | ((static_cast<uint32_t>(d) & 0xFFu) << 24);
}

// Quantize 8 BF16 values (one 16-byte vector) into 8 int8 codes.
__device__ __forceinline__ uint2 quantize8(const uint4 v, float s, float r, bool fast) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    int q[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float lo = bf16_bits_to_f32(w[i] & 0xFFFFu);
        const float hi = bf16_bits_to_f32(w[i] >> 16);
        if (s == 0.0f) {
            q[2 * i] = 0;
            q[2 * i + 1] = 0;
        } else if (fast) {
            q[2 * i] = quantize_fast(lo, s, r);
            q[2 * i + 1] = quantize_fast(hi, s, r);
        } else {
            q[2 * i] = quantize_exact(lo, s);
            q[2 * i + 1] = quantize_exact(hi, s);
        }
    }
    return make_uint2(pack4(q[0], q[1], q[2], q[3]), pack4(q[4], q[5], q[6], q[7]));
}

// Max of |bf16| over a 16-byte vector, as the BF16 magnitude bit pattern:
// for finite values, ordering of |x| equals the unsigned ordering of (bits & 0x7FFF).
__device__ __forceinline__ uint32_t amax_bits8(const uint4 v) {
    uint32_t m = 0;
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        m = max(m, w[i] & 0x7FFFu);
        m = max(m, (w[i] >> 16) & 0x7FFFu);
    }
    return m;
}

// Power-of-two (UE8M0) scale of a group whose largest magnitude is amax: the
// smallest 2^e >= amax / 127 (decided exactly: amax <= 127 * 2^e), e clamped
// to [-127, 127]; 2^-127 for amax == 0. For a normal amax in [2^E, 2^(E+1)),
// 127 * 2^(E-7) < amax <= 127 * 2^(E-5), so e is E - 6 or E - 5. Dividing
// by the scale is then exact, so the codes are round-half-even(x * 2^-e).
__device__ __forceinline__ float pow2_from_exponent(int e) {
    return e >= -126 ? __uint_as_float(static_cast<uint32_t>(e + 127) << 23)
                     : __uint_as_float(0x00400000u);   // 2^-127 (subnormal)
}

__device__ __forceinline__ float pow2_scale(float amax) {
    const uint32_t bits = __float_as_uint(amax);
    const int bexp = static_cast<int>((bits >> 23) & 0xFFu);
    if (bexp == 0) return pow2_from_exponent(-127);   // zero or subnormal amax
    int e = bexp - 127 - 6;
    if (e >= -127 && !(amax <= 127.0f * pow2_from_exponent(e))) ++e;
    e = max(-127, min(127, e));
    return pow2_from_exponent(e);
}
}  // namespace w8a8
