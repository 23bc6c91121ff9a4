// Device-side helpers for the sm_103a kernels: mbarriers with bounded waits,
// TMA tensor loads, tcgen05 (TMEM alloc, MMA, ld/st, commit, fences) and the
// library-wide device error word.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace w8a8 {

// ---------------------------------------------------------------- error word
// A kernel whose bounded wait gave up writes a code into the library's device
// error word (first writer wins). Layout of the 64-bit code:
//   bits 56..63 kernel id, 48..55 role, 32..47 wait site, 0..31 CTA index.

enum KernelId : unsigned { KID_GEMM = 1, KID_SELFTEST = 2, KID_QUANT = 3 };
enum Role : unsigned {
    ROLE_PRODUCER = 1, ROLE_MMA = 2, ROLE_CONVERT = 3, ROLE_EPILOGUE = 4, ROLE_SELFTEST = 5
};

// A wait gives up after this many nanoseconds of %globaltimer time. Every wait
// in these kernels normally completes within microseconds.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void record_device_error(unsigned long long *err, unsigned kid,
                                                    unsigned role, unsigned site) {
    unsigned long long code = ((unsigned long long)kid << 56) |
                              ((unsigned long long)(role & 0xFF) << 48) |
                              ((unsigned long long)(site & 0xFFFF) << 32) |
                              (unsigned long long)blockIdx.x;
    atomicCAS(err, 0ull, code);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void fence_mbarrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Arrive without release semantics: for a consumer whose only reads of the
// guarded buffer are tensor-memory loads already completed by
// tcgen05.wait::ld. A release arrive would also wait for every outstanding
// global load or store of the thread (prefetches, output stores).
__device__ __forceinline__ void mbar_arrive_relaxed(uint32_t bar) {
    asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait with a suspend-time hint: a thread whose phase is not complete is
// suspended (it takes no issue slots from the warps doing work) until the
// phase completes or about `hint_ns` elapse.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity,
                                                    uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete. Returns false (and
// records a device error) if the wait gives up after limit_ns (kWaitLimitNs
// unless given), or if another role of this CTA has already given up
// (*abort != 0).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                          unsigned long long *err, unsigned role, unsigned site,
                                          unsigned long long limit_ns = kWaitLimitNs,
                                          unsigned kid = KID_GEMM) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, 1000000u)) return true;
        if (*abort) return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            *abort = 1;
            record_device_error(err, kid, role, site);
            return false;
        }
    }
}

// Same contract as mbar_wait, but polls with the non-blocking test_wait
// instead of suspending: for hand-offs on a pipeline's critical path, where
// the wake-up latency of a suspended thread (hundreds of cycles) would be
// paid on every step. Costs issue slots while it waits.
__device__ __forceinline__ bool mbar_wait_spin(uint32_t bar, uint32_t parity, volatile int *abort,
                                               unsigned long long *err, unsigned role,
                                               unsigned site) {
    if (mbar_test_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_test_wait(bar, parity)) return true;
        if ((i & 255u) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                *abort = 1;
                record_device_error(err, KID_GEMM, role, site);
                return false;
            }
        }
    }
}

// ------------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_prefetch_desc(const void *tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(tmap), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// Contiguous global -> shared copy of `bytes` (both addresses 16-byte aligned,
// bytes a multiple of 16), completing on the mbarrier's transaction count.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// -------------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T, kind::f16 (fp16 x fp16 -> fp32), cta_group::1.
__device__ __forceinline__ void mma_f16_tmemA(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on the mbarrier when all previously issued tcgen05 ops of this
// thread have completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 columns of 32-bit: thread t receives lane (base lane + t),
// columns [col, col + 32). The load and its completion wait are one asm
// statement, so no use of the registers can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld_32cols_sync(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// Two 32-column loads (e.g. the partials of two groups) and one wait, in one
// asm statement: the second load's latency overlaps the first's.
__device__ __forceinline__ void tmem_ld_2x32cols_sync(uint32_t taddr_a, uint32_t taddr_b,
                                                      uint32_t (&a)[32], uint32_t (&b)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(a[0]),"=r"(a[1]),"=r"(a[2]),"=r"(a[3]),"=r"(a[4]),"=r"(a[5]),"=r"(a[6]),"=r"(a[7]),"=r"(a[8]),"=r"(a[9]),"=r"(a[10]),"=r"(a[11]),"=r"(a[12]),"=r"(a[13]),"=r"(a[14]),"=r"(a[15]),"=r"(a[16]),"=r"(a[17]),"=r"(a[18]),"=r"(a[19]),"=r"(a[20]),"=r"(a[21]),"=r"(a[22]),"=r"(a[23]),"=r"(a[24]),"=r"(a[25]),"=r"(a[26]),"=r"(a[27]),"=r"(a[28]),"=r"(a[29]),"=r"(a[30]),"=r"(a[31]),"=r"(b[0]),"=r"(b[1]),"=r"(b[2]),"=r"(b[3]),"=r"(b[4]),"=r"(b[5]),"=r"(b[6]),"=r"(b[7]),"=r"(b[8]),"=r"(b[9]),"=r"(b[10]),"=r"(b[11]),"=r"(b[12]),"=r"(b[13]),"=r"(b[14]),"=r"(b[15]),"=r"(b[16]),"=r"(b[17]),"=r"(b[18]),"=r"(b[19]),"=r"(b[20]),"=r"(b[21]),"=r"(b[22]),"=r"(b[23]),"=r"(b[24]),"=r"(b[25]),"=r"(b[26]),"=r"(b[27]),"=r"(b[28]),"=r"(b[29]),"=r"(b[30]),"=r"(b[31])
        : "r"(taddr_a), "r"(taddr_b)
        : "memory");
}

// 32 lanes x 16 columns load, asynchronous: the registers are valid only
// after tmem_wait_ld_dep16() on the same array.
__device__ __forceinline__ void tmem_ld_16cols(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// tcgen05.wait::ld that also names the destination registers of the load it
// completes, so no use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_wait_ld_dep16(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
}

// 32 lanes x 16 columns store: thread t writes lane (base lane + t).
__device__ __forceinline__ void tmem_st_16cols(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

// Shared-memory matrix descriptor for a K-major operand stored with the
// 128-byte swizzle (8-row x 128-byte atoms, atoms 1024 bytes apart along
// the row dimension). Fields: start address >> 4 (bits 0-13), leading byte
// offset >> 4 (16-29, unused for this layout), stride byte offset >> 4
// (32-45), descriptor version 1 (bit 46), layout 2 = 128B swizzle (61-63).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
    d |= (uint64_t)(16 >> 4) << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor, kind::f16: fp16 A and B, fp32 D, both K-major,
// shape M x N (M = 128, N a multiple of 16 up to 256).
__host__ __device__ constexpr uint32_t idesc_f16_f32(uint32_t M, uint32_t N) {
    return (1u << 4)                // D format: f32
           | (0u << 7)              // A format: f16
           | (0u << 10)             // B format: f16
           | ((N >> 3) << 17)       // N / 8
           | ((M >> 4) << 24);      // M / 16
}

// Same for bf16 A and B operands (the weight-only path, BF16 activations).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N) {
    return (1u << 4)                // D format: f32
           | (1u << 7)              // A format: bf16
           | (1u << 10)             // B format: bf16
           | ((N >> 3) << 17)       // N / 8
           | ((M >> 4) << 24);      // M / 16
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy accesses (TMA, tcgen05.mma operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Loads issued exactly where they are written (volatile asm is not moved past
// other volatile asm such as barrier waits), so a prefetch stays a prefetch:
// the compiler may otherwise sink a load down to its first use.
__device__ __forceinline__ float ldg_nc_f32_now(const float *p) {
    float v;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ float4 ldg_nc_f32x4_now(const float *p) {
    float4 v;
    asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

// Programmatic dependent launch: wait until the kernels this one depends on
// have completed and their writes are visible (a no-op without the launch
// attribute), and let the next kernel in the stream start launching early.
__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Arrives on a named barrier without waiting (the other participants wait
// with named_barrier_sync; the arrival orders this thread's earlier memory
// accesses before their later ones, at CTA scope).
__device__ __forceinline__ void named_barrier_arrive(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also ORs a predicate over its participants: every thread
// gets true when any participant passed true. Warp-uniform use only.
__device__ __forceinline__ bool named_barrier_or(uint32_t id, uint32_t nthreads, bool c) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pc, pr;\n\t"
        "setp.ne.u32 pc, %1, 0;\n\t"
        "bar.red.or.pred pr, %2, %3, pc;\n\t"
        "selp.u32 %0, 1, 0, pr;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(c)), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// 4-byte asynchronous copy global -> shared; src_bytes 0 writes zero (the
// source is then not read, but must still be a valid address).
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

// Waits for this thread's cp.async copies.
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

template <uint32_t RegCount>
__device__ __forceinline__ void setmaxnreg_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(RegCount));
}

template <uint32_t RegCount>
__device__ __forceinline__ void setmaxnreg_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(RegCount));
}

// int8 x4 (one 32-bit word) -> two fp16x2 words holding the exact integers.
// Bias each byte to unsigned (x ^ 0x80 = x + 128), place it in the low
// mantissa bits of the fp16 number 1024 (0x6400 | u = 1024 + u), then
// subtract 1152 = 1024 + 128: every step is exact for |x| <= 128.
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t u = w ^ 0x80808080u;
    uint32_t a, b;
    asm("prmt.b32 %0, %1, %2, 0x7170;" : "=r"(a) : "r"(u), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x7372;" : "=r"(b) : "r"(u), "r"(0x64646464u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(0x64806480u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(0x64806480u));
}

// int8 x4 -> two bf16x2 words holding the exact integers (|x| <= 127): the
// magnitude goes into the low mantissa bits of the bf16 number 128
// (0x4300 | |x| = 128 + |x|, exact since bf16 has 7 mantissa bits), 128 is
// subtracted (exact), and each byte's sign bit is copied to its half's sign
// bit. (x = -128 never occurs: codes are clamped to [-127, 127].)
__device__ __forceinline__ void i8x4_to_bf16x4(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t mag = __vabsss4(w);
    const uint32_t sgn = w & 0x80808080u;
    uint32_t a, b, sl, sh;
    asm("prmt.b32 %0, %1, %2, 0x7170;" : "=r"(a) : "r"(mag), "r"(0x43434343u));
    asm("prmt.b32 %0, %1, %2, 0x7372;" : "=r"(b) : "r"(mag), "r"(0x43434343u));
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(0x43004300u));
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(0x43004300u));
    asm("prmt.b32 %0, %1, %2, 0x1404;" : "=r"(sl) : "r"(sgn), "r"(0u));
    asm("prmt.b32 %0, %1, %2, 0x3424;" : "=r"(sh) : "r"(sgn), "r"(0u));
    lo |= sl;
    hi |= sh;
}

}  // namespace w8a8
