// Per-token activation quantization arithmetic shared by the quantizer
// kernels and the GEMV that quantizes its own token rows: both must produce
// the same codes bit for bit (per-token scale s = amax/127, codes =
// round-half-even(x / s) clamped to [-127, 127]; "Deploying Hunyuan 770B in
// INT8 on domestic accelerators", §3.1).
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
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

// The exact quotient's rounding, kept out of line: it runs for about one
// value in 16000, and inlining it at every use made the quantizer's loop large
// enough to stall on instruction fetch.
static __device__ __noinline__ float code_by_division(float x, float s) {
    return fminf(fmaxf(rintf(__fdiv_rn(x, s)), -127.0f), 127.0f);
}

// Adding 1.5 * 2^23 to a float of magnitude below 2^22 rounds it to an
// integer (round-half-even, the FP32 adder's mode) and leaves that integer,
// plus 2^22, in the low mantissa bits: the low byte is then the integer's
// two's-complement byte, and subtracting the constant back is exact.
constexpr float kRoundAdd = 12582912.0f;

// The code of x, as the float code + kRoundAdd: the same code quantize_fast /
// quantize_exact give. For finite x with |x| <= amax, s = fl(amax / 127) a
// normal number and r = fl(1 / s): |x * r| and |x / s| are at most
// 127 (1 + 2^-24)^3 < 127.5, so no clamp is needed on the fast path. A zero
// code is +0 (y + c - c is +0 for |y| < 1/2).
__device__ __forceinline__ float code_plus_round(float x, float s, float r, bool fast) {
    if (!fast) return __fadd_rn(s == 0.0f ? 0.0f : code_by_division(x, s), kRoundAdd);
    const float y = __fmul_rn(x, r);
    const float f = __fadd_rn(y, kRoundAdd);
    const float yi = __fsub_rn(f, kRoundAdd);
    return fabsf(__fsub_rn(y, yi)) >= 0.5f - 3.0e-5f ? __fadd_rn(code_by_division(x, s), kRoundAdd)
                                                      : f;
}

__device__ __forceinline__ uint32_t pack4(int a, int b, int c, int d) {
    return (static_cast<uint32_t>(a) & 0xFFu) | ((static_cast<uint32_t>(b) & 0xFFu) << 8) |
           ((static_cast<uint32_t>(c) & 0xFFu) << 16) | ((static_cast<uint32_t>(d) & 0xFFu) << 24);
}

// Two IEEE binary32 operations in one instruction (the f32x2 forms of
// sm_100-family GPUs): each half is rounded to nearest even exactly as the
// scalar __fmul_rn / __fadd_rn / __fsub_rn of that half would be.
__device__ __forceinline__ unsigned long long f2_bits(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_split(unsigned long long v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long f2_mul(unsigned long long a, unsigned long long b) {
    unsigned long long r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
    unsigned long long r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ unsigned long long f2_sub(unsigned long long a, unsigned long long b) {
    unsigned long long r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// The codes of 8 BF16 values (one 16-byte vector), each as code + kRoundAdd:
// code_plus_round for each value, with the near-half check of all 8 folded
// into one branch (taken for about one vector in 2000).
__device__ __forceinline__ void codes8(const uint4 v, float s, float r, bool fast, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float x[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = bf16_bits_to_f32(w[i] & 0xFFFFu);
        x[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
    }
    if (!fast) {
#pragma unroll
        for (int j = 0; j < 8; ++j) f[j] = code_plus_round(x[j], s, r, false);
        return;
    }
    bool near = false;
    const unsigned long long r2 = f2_bits(r, r), c2 = f2_bits(kRoundAdd, kRoundAdd);
#pragma unroll
    for (int i = 0; i < 4; ++i) {   // pairs: y = x*r, f = y + c, d = y - (f - c)
        const unsigned long long y2 = f2_mul(f2_bits(x[2 * i], x[2 * i + 1]), r2);
        const unsigned long long f2 = f2_add(y2, c2);
        float d0, d1;
        f2_split(f2_sub(y2, f2_sub(f2, c2)), d0, d1);
        f2_split(f2, f[2 * i], f[2 * i + 1]);
        near |= fabsf(d0) >= 0.5f - 3.0e-5f;
        near |= fabsf(d1) >= 0.5f - 3.0e-5f;
    }
    if (near) {
#pragma unroll
        for (int j = 0; j < 8; ++j) f[j] = code_plus_round(x[j], s, r, true);
    }
}

// The low bytes of four code + kRoundAdd floats, packed in order.
__device__ __forceinline__ uint32_t pack_code_bytes(float a, float b, float c, float d) {
    uint32_t lo, hi, w;
    asm("prmt.b32 %0, %1, %2, 0x0040;" : "=r"(lo) : "r"(__float_as_uint(a)), "r"(__float_as_uint(b)));
    asm("prmt.b32 %0, %1, %2, 0x0040;" : "=r"(hi) : "r"(__float_as_uint(c)), "r"(__float_as_uint(d)));
    asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(w) : "r"(lo), "r"(hi));
    return w;
}

// Quantize 8 BF16 values (one 16-byte vector) into 8 int8 codes.
__device__ __forceinline__ uint2 quantize8(const uint4 v, float s, float r, bool fast) {
    float f[8];
    codes8(v, s, r, fast, f);
    return make_uint2(pack_code_bytes(f[0], f[1], f[2], f[3]), pack_code_bytes(f[4], f[5], f[6], f[7]));
}

// The same 8 codes as fp16 (exact integers; the tensor-core GEMM's operand).
__device__ __forceinline__ uint4 quantize8_f16(const uint4 v, float s, float r, bool fast) {
    float f[8];
    codes8(v, s, r, fast, f);
    uint32_t h[4];
    const unsigned long long c2 = f2_bits(kRoundAdd, kRoundAdd);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float lo, hi;
        f2_split(f2_sub(f2_bits(f[2 * i], f[2 * i + 1]), c2), lo, hi);
        const __half2 p = __floats2half2_rn(lo, hi);
        h[i] = *reinterpret_cast<const uint32_t *>(&p);
    }
    return make_uint4(h[0], h[1], h[2], h[3]);
}

// Max of |bf16| over a 16-byte vector, as the BF16 magnitude bit pattern:
// for finite values, ordering of |x| equals the unsigned ordering of (bits & 0x7FFF).
__device__ __forceinline__ uint32_t amax_bits8(const uint4 v) {
    uint32_t m = __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                          __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
    return max(m & 0xFFFFu, m >> 16);
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
