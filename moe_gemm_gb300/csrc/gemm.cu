// Group-scaled W8A8 GEMM on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// What it computes ("Deploying Hunyuan 770B in INT8 on domestic
// accelerators", §3.1): for every output element, each 128-wide K group is
// multiplied INT8 x INT8 and summed exactly, the group sum is scaled by that
// group's FP32 weight scale into an FP32 accumulator, and the per-token FP32
// scale is applied once at the end. MoE expert layers (§1.3, §4.4) run the
// same tiles per expert over the rows routed to it.
//
// How, on GB300:
//  * sm_103a has no integer tcgen05 MMA, so the exact integer group sum is
//    formed by tcgen05.mma kind::f16 on fp16 copies of the int8 codes: every
//    int8 is an exact fp16 integer, every product (<= 127^2) is exact, and a
//    128-term group sum (|P| <= 2,064,512 < 2^24) is an exact FP32 integer.
//    Each group gets a FRESH accumulator in tensor memory, so the tensor core
//    never adds numbers that are not exactly representable.
//  * Swap-AB: the MMA's M side (128 TMEM lanes) is 128 weight rows n, its N
//    side is a tile of up to 128 token rows. So the weight scale sw[n, g] is
//    one register per epilogue thread.
//  * Weights stay int8 in HBM. TMA lands 128 x 256 int8 weight stages in
//    shared memory; a converter warpgroup widens them in registers and writes
//    the fp16 A operand straight into tensor memory (tcgen05.st), so the
//    widening costs no shared-memory bandwidth beyond one read.
//  * Token operand: an fp16 copy of the int8 codes (written just before this
//    kernel by the fused quantizer or by a staging kernel) is loaded by TMA
//    with the 128-byte swizzle, through a ring of token stages that runs
//    ahead of the MMAs. This kernel is launched as a programmatic dependent
//    of that kernel: the token producer waits for it (griddepcontrol.wait)
//    before loading codes, the epilogue before reading token scales; the
//    weight stream, the conversion and all set-up start at once.
//  * Two K groups move through the pipeline per step (one barrier hand-off,
//    one commit and one epilogue wait per 32 KB of weights); see the kernel.
//  * Epilogue warpgroups drain the partial buffers (tcgen05.ld), fma each
//    partial with sw[n,g] into register accumulators in K order, and at the
//    end of the tile multiply by sa[m] and store BF16 (round to nearest even)
//    or FP32.
//  * Persistent CTAs walk a tile list built on the device from the expert
//    offsets (no host read, graph-capture safe). Within an (expert, weight
//    tile) the token tiles are consecutive so CTAs running together share the
//    weight tile through L2.
//  * Every mbarrier wait is bounded (%globaltimer); a wait that gives up sets
//    the library error word and the CTA drains its copies, frees TMEM and
//    returns.
//  * Dense calls of at most 4 token rows run a CUDA-core kernel instead
//    (w8a8_gemv_kernel, below): exact int8 dot products (dp4a) cost less than
//    the weight stream there.
//  * Dense calls of 5..64 token rows split tile K ranges over all SMs
//    (stream-K) when the workspace has room for it.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "quant_math.cuh"
#include "internal.h"

namespace w8a8 {

__device__ unsigned long long g_device_error = 0;

namespace {

constexpr int kThreads = 512;
constexpr int kMaxAStages = 12;     // weight tiles in flight (shared memory)
constexpr int kMaxBStages = 8;      // token stages in flight
constexpr int kTileN = 128;         // weight rows per tile = MMA M = TMEM lanes
constexpr int kGroupK = 128;        // K elements per scale group
constexpr int kMaxBatchRows = 128;  // token rows per tile (MMA N <= 128)
constexpr int kBoxRows = 32;        // token rows per TMA box
constexpr int kAStageBytes = kTileN * kGroupK;   // 16 KB int8
constexpr int kTmemCols = 512;
constexpr int kTmemA0 = 256;        // TMEM fp16 weight operands from column 256
constexpr int kEpiRegs = 200;       // 256 threads x 200 + 256 x 56 = 512 x 128 at launch
constexpr int kOtherRegs = 56;
// Narrow tiles: one 32-column accumulator per epilogue thread, plus the
// split-tile publish/combine paths; the other roles carry the stream-K
// bookkeeping in 64.
constexpr int kSplitEpiRegs = 192;
constexpr int kSplitOtherRegs = 64;
constexpr int kSmemLimit = 232448;
// Dense problems with wide token tiles walk their tiles in bands of this many
// weight tiles (see decode_tile).
constexpr int kRasterBand = 8;

// Shared memory: a fixed area (barriers, flags, tile table), then the weight
// stages, then the token stages (offsets from a 1024-byte aligned base).
constexpr int kOffBar = 0;
constexpr int kOffMisc = 8 * 128;
constexpr int kOffTab = kOffMisc + 64;
constexpr int kTabBytes = 3 * (kMaxExperts + 1) * 4;
constexpr int kOffStages = ((kOffTab + kTabBytes + 1023) / 1024) * 1024;
static_assert((kThreads / 2) * (kEpiRegs + kOtherRegs) == 65536, "register split");
static_assert((kThreads / 2) * (kSplitEpiRegs + kSplitOtherRegs) == 65536, "register split");

struct KParams {
    const float *sa;
    const float *sw;
    const int32_t *offsets;
    void *y;
    int32_t *dbg;
    int R, E, N, K, G;
    int n_tiles;
    int out_fp32;
    int a_stages;       // weight pipeline depth (<= kMaxAStages)
    int b_stages;       // token pipeline depth (<= kMaxBStages)
    int b_rows;         // token rows per MMA batch and per token stage (32, 64, 96 or 128)
    int tile_tokens;    // token rows per tile (b_rows or 2 * b_rows)
    int tab_off;        // byte offset of the tile table in shared memory
    int group_tokens;   // wide tiles: token stages released per K group (dense calls)
    int gw;             // tile order: bands of gw weight tiles (0: expert-major, see decode_tile)
    // Weight scales: one row of G scales per 2^sw_shift weight rows (0: per
    // row; 7: [128, 128] blocks), sw_rows rows of scales per expert.
    int sw_shift;
    int sw_rows;
    // GEMV that quantizes its own token rows: BF16 activations [R, lda] and
    // the byte offset of the resident int8 code buffer in shared memory.
    const uint16_t *act;
    long long lda;
    int qbuf_off;
    unsigned long long *err;
    // Stream-K split of dense calls (null sk_cnt: whole tiles only).
    int *sk_cnt;        // [2 * grid] arrival counters of split tiles, zero at launch
    float *sk_part;     // [grid][2][sk_ld][128] FP32 piece partials
    int sk_ld;          // token columns per partial slot
};

// The token scale of row m: 1 when the call has none (weight-only path with
// BF16 activations).
__device__ __forceinline__ float load_sa(const KParams &p, int m) {
    return p.sa != nullptr ? __ldg(p.sa + m) : 1.0f;
}

// int8 x4 -> the MMA's A-operand type: fp16 (kBf16 false) or bf16, exact.
template <bool kBf16>
__device__ __forceinline__ void i8x4_to_op(uint32_t w, uint32_t &lo, uint32_t &hi) {
    if constexpr (kBf16)
        i8x4_to_bf16x4(w, lo, hi);
    else
        i8x4_to_f16x4(w, lo, hi);
}

struct TileInfo {
    int e, n0, m0, rows;
};

// Ring position of a pipeline with n slots: slot index and phase parity.
struct Ring {
    uint32_t idx = 0, phase = 0;
    __device__ __forceinline__ void advance(uint32_t n) {
        if (++idx == n) {
            idx = 0;
            phase ^= 1u;
        }
    }
};

// Tile t of the list: the expert e whose tiles [s_base[e], s_base[e+1])
// contain t, then its weight tile nt and token tile mt. gw == 0: the token
// tiles of one weight tile are consecutive (an expert's few token tiles share
// its weight tile through L2). gw > 0 (one dense segment): bands of gw weight
// tiles, and within a band the weight tiles of one token tile consecutive, so
// the CTAs running at the same time share a few token tiles and a few weight
// tiles instead of every token tile of the problem.
__device__ __forceinline__ TileInfo decode_tile(int t, const int *s_base, const int *s_lo,
                                                const int *s_cnt, int E, int tt, int n_tiles = 0,
                                                int gw = 0) {
    int lo = 0, hi = E;  // s_base[lo] <= t < s_base[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_base[mid] <= t) lo = mid; else hi = mid;
    }
    const int local = t - s_base[lo];
    const int cnt = s_cnt[lo];
    const int m_tiles = (cnt + tt - 1) / tt;
    int nt, mt;
    if (gw > 0) {
        const int band_tiles = gw * m_tiles;
        const int band = local / band_tiles;
        const int w = min(gw, n_tiles - band * gw);
        const int r = local - band * band_tiles;
        mt = r / w;
        nt = band * gw + (r - mt * w);
    } else {
        nt = local / m_tiles;
        mt = local - nt * m_tiles;
    }
    TileInfo ti;
    ti.e = lo;
    ti.n0 = nt * kTileN;
    ti.m0 = s_lo[lo] + mt * tt;
    ti.rows = min(tt, cnt - mt * tt);
    return ti;
}

// Tile table (one warp): expert e owns tiles [s_base[e], s_base[e+1]); its
// rows are [s_lo[e], s_lo[e] + s_cnt[e]) with the offsets clamped into [0, R]
// (a dense problem is one segment [0, R)). tt = token rows per tile.
__device__ __forceinline__ void build_tile_table(const KParams &p, int tt, int lane, int *s_base,
                                                 int *s_lo, int *s_cnt, volatile int *s_total) {
    int carry = 0;
    for (int e0 = 0; e0 < p.E; e0 += 32) {
        const int e = e0 + lane;
        int lo = 0, cnt = 0;
        if (e < p.E) {
            if (p.offsets != nullptr) {
                int a = p.offsets[e], b = p.offsets[e + 1];
                a = min(max(a, 0), p.R);
                b = min(max(b, 0), p.R);
                lo = a;
                cnt = max(b - a, 0);
            } else {
                lo = 0;
                cnt = p.R;
            }
        }
        const int tiles = (e < p.E) ? p.n_tiles * ((cnt + tt - 1) / tt) : 0;
        int incl = tiles;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += v;
        }
        if (e < p.E) {
            s_base[e] = carry + incl - tiles;
            s_lo[e] = lo;
            s_cnt[e] = cnt;
        }
        carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    if (lane == 0) {
        s_base[p.E] = carry;
        *s_total = carry;
    }
}

// Bounded wait used only on the exit path, independent of the abort flag.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) break;
    }
}

// Waits for the copies of the last min(issued, slots) issues of a ring.
__device__ __forceinline__ void drain_ring(uint32_t bar0, uint32_t issued, uint32_t slots) {
    for (uint32_t i = issued > slots ? issued - slots : 0; i < issued; ++i)
        drain_wait(bar0 + 8u * (i % slots), (i / slots) & 1u);
}

// Stream-K work split (dense narrow tiles, when the caller's workspace has
// room for it): the tiles that fill whole waves go round-robin to the CTAs;
// the L tiles left over are split in K. When the grid holds at least two
// CTAs per left-over tile, each of them is cut into k = min(S, grid / L)
// equal pieces, one per CTA (a CTA then holds one split piece, so it crosses
// one piece boundary and combines at most one tile); otherwise their steps
// are divided into equal contiguous ranges, one per CTA. A CTA works on its
// split piece(s) first and on its whole tiles after them. Each piece stores
// its FP32 partial sum (before the token scale) and counts itself in; the
// CTA that brings a tile's last piece adds the pieces in K order (so the
// result does not depend on arrival order), applies sa and stores y. No CTA
// waits for another.
//
// WorkPlan: this CTA's split steps [u0, u1) (steps of tiles [dp, total),
// S per tile, numbered from 0 at tile dp; g_sk CTAs take part), then
// round-robin whole tiles of [0, dp). k > 0: the aligned cut above.
// All of it in 32-bit arithmetic: U < grid * S fits an int, and
// floor(c U / g) is formed from U = q g + r as c q + floor(c r / g).
struct WorkPlan {
    int dp, S, g_sk, U, u0, u1, k;
};

__device__ __forceinline__ WorkPlan make_plan(int total, int G, bool stream_k) {
    WorkPlan w;
    w.S = (G + 1) >> 1;
    const int grid = static_cast<int>(gridDim.x);
    const int c = static_cast<int>(blockIdx.x);
    w.u0 = w.u1 = 0;
    w.k = 0;
    if (!stream_k) {
        w.dp = total;
        w.g_sk = 0;
        w.U = 0;
        return w;
    }
    w.dp = (total / grid) * grid;   // whole waves; fewer than grid tiles are split
    const int L = total - w.dp;
    w.U = L * w.S;
    const int k = L > 0 ? min(w.S, grid / L) : 0;
    if (k >= 2) {
        w.k = k;
        w.g_sk = k * L;
        if (c < w.g_sk) {
            const int tl = c / k, j = c - tl * k;
            w.u0 = tl * w.S + (j * w.S) / k;
            w.u1 = tl * w.S + ((j + 1) * w.S) / k;
        }
        return w;
    }
    w.g_sk = w.U < grid ? w.U : grid;
    if (c < w.g_sk) {
        const int q = w.U / w.g_sk, r = w.U - q * w.g_sk;
        w.u0 = c * q + (c * r) / w.g_sk;
        w.u1 = (c + 1) * q + ((c + 1) * r) / w.g_sk;
    }
    return w;
}

// Contiguous ranges: the CTA whose range contains step x (0 <= x < U): the
// largest c with floor(c U / g) <= x, i.e. c U < (x + 1) g. A float estimate
// is corrected with exact 64-bit products.
__device__ __forceinline__ int sk_owner(int x, const WorkPlan &w) {
    const long long rhs = static_cast<long long>(x + 1) * w.g_sk;
    int c = static_cast<int>(__fdividef(static_cast<float>(rhs), static_cast<float>(w.U)));
    c = min(max(c, 0), w.g_sk - 1);
    while (c > 0 && static_cast<long long>(c) * w.U >= rhs) --c;
    while (c + 1 < w.g_sk && static_cast<long long>(c + 1) * w.U < rhs) ++c;
    return c;
}

// The CTAs holding the pieces of split tile t, in K order.
__device__ __forceinline__ void tile_owners(int t, const WorkPlan &w, int &c_first,
                                            int &c_final) {
    if (w.k > 0) {
        c_first = (t - w.dp) * w.k;
        c_final = c_first + w.k - 1;
    } else {
        const int x0 = (t - w.dp) * w.S;
        c_first = sk_owner(x0, w);
        c_final = sk_owner(x0 + w.S - 1, w);
    }
}

// Calls f(tile, s0, s1) for every piece of this CTA in order; f returns false
// to stop. A stream-K range is shorter than a tile (fewer than grid tiles are
// left over), so it holds at most two pieces: they are formed up front and
// the walk is one counted loop with one call site. (A walk that advanced a
// step cursor through the range made every pipeline step ~15% slower in all
// roles, measured.)
template <class F>
__device__ __forceinline__ void for_each_piece(const WorkPlan &w, F &&f) {
    int t0 = 0, a0 = 0, b0 = 0, b1 = 0, nsk = 0;
    if (w.u0 < w.u1) {
        const int ts = w.u0 / w.S;
        t0 = w.dp + ts;
        a0 = w.u0 - ts * w.S;
        b0 = min(w.S, a0 + (w.u1 - w.u0));
        nsk = 1;
        const int u = w.u0 + (b0 - a0);   // the range goes on into tile t0 + 1
        if (u < w.u1) {
            b1 = min(w.S, w.u1 - u);
            nsk = 2;
        }
    }
    for (int i = 0;; ++i) {
        int t, s0, s1;
        if (i < nsk) {
            t = t0 + i;
            s0 = i == 0 ? a0 : 0;
            s1 = i == 0 ? b0 : b1;
        } else {
            t = static_cast<int>(blockIdx.x) + (i - nsk) * static_cast<int>(gridDim.x);
            if (t >= w.dp) return;
            s0 = 0;
            s1 = w.S;
        }
        if (!f(t, s0, s1)) return;
    }
}

// =============================================================================
// The tensor-core GEMM: every tile is one MMA batch of up to 128 token rows
// (decode shapes, MoE experts, 128-row tiles of large problems). Two K groups
// move through the pipeline per step, so every hand-off (barrier wait,
// arrive, commit) is paid once per 32 KB of weights instead of once per 16 KB:
//  * a weight stage is 128 rows x 256 K int8 (two TMA boxes, 256 contiguous
//    bytes per weight row);
//  * a step slot (2 of them) holds the fp16 A operands of both groups in TMEM
//    (128 columns) and their two partial buffers (2 x b_rows columns; one
//    pair shared by all steps in the wide form, see below); one commit per
//    step ("done") frees them and tells the epilogue the step's partials are
//    ready; token tiles sit in their own ring of shared-memory stages;
//  * each epilogue warpgroup owns 32-column chunks of the token tile and
//    drains both groups of a step with two loads and a single wait.
// Warp roles (512 threads): 0 weight TMA producer; 1 MMA issuer and TMEM
// allocation; 2 token TMA producer (the only thread that waits for the
// kernel that wrote the codes); 3 admission (token tiles landed, partial
// buffers free -> "ready"); 4-7 converter (int8 -> fp16 A operand in TMEM);
// 8-15 epilogue (for token tiles of <= 32 rows, 12-15 finish the split tiles
// instead). kDebug additionally writes every exact group partial.
// =============================================================================
constexpr int kNarrowSlots = 2;
constexpr int kWideOffTab = kOffMisc + 64;       // wide tiles: tile table in the fixed area
constexpr int kWideOffStages = 2048;
constexpr int kWideMaxExperts = (kWideOffStages - kWideOffTab) / 12 - 1;
constexpr int kNarrowAStageBytes = 2 * kAStageBytes;   // 32 KB

struct NBar {
    static constexpr int a_full = 0;                     // [kMaxAStages] TMA -> converter
    static constexpr int a_empty = a_full + kMaxAStages; // [kMaxAStages] converter -> TMA
    static constexpr int ready = a_empty + kMaxAStages;  // [2] converter (4) + admission (1) -> MMA
    static constexpr int done = ready + kNarrowSlots;    // [2] MMA commit -> epilogue, converter
    static constexpr int b_full = done + kNarrowSlots;   // [kMaxBStages] token TMA -> admission
    static constexpr int b_empty = b_full + kMaxBStages; // [kMaxBStages] epilogue -> token TMA
    static constexpr int p_empty = b_empty + kMaxBStages;// [2] epilogue -> admission
    static constexpr int p_full = p_empty + kNarrowSlots;  // [2] wide: MMA commit per group -> epilogue
    static constexpr int drain = p_full + kNarrowSlots;
    static constexpr int count = drain + 1;
};
static_assert(NBar::count <= 128, "barrier area");
// Token scales of the current whole tile, 64 per epilogue warpgroup, in the
// barrier area past the barriers.
constexpr int kOffTokScales = 512;
static_assert(NBar::count * 8 <= kOffTokScales && kOffTokScales + 2 * 64 * 4 <= kOffMisc,
              "token-scale area");

// kWide: 96- or 128-row token tiles. The two steps' partial buffers (2 x 2 x
// 128 columns) would not fit next to the operand slots in TMEM, so one pair
// of partial buffers serves every step, one buffer per group with its own
// commit ("p_full") and release ("p_empty"): the epilogue drains group 0
// while the MMAs of group 1 issue, and group 0 of the next step waits only
// for that drain. Each epilogue warpgroup owns two 32-column chunks; the tile
// table lives in the fixed area so that the weight stages fit beside the two
// token stages.
// kA16: weight-only form: BF16 activations are the token operand (no token
// scale), weights are widened to bf16.
template <bool kDebug, bool kWide, bool kA16 = false>
__global__ void __launch_bounds__(kThreads, 1)
w8a8_gemm_narrow_kernel(const __grid_constant__ CUtensorMap tmap_w,
                        const __grid_constant__ CUtensorMap tmap_x, const KParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw_addr);

    constexpr uint32_t NP = kWide ? 1u : kNarrowSlots;   // partial-buffer slots
    constexpr int NCH = kWide ? 2 : 1;                    // 32-column chunks per epilogue warpgroup
    constexpr uint32_t kStagesOff = kWide ? kWideOffStages : kOffStages;
    const uint32_t SA = static_cast<uint32_t>(p.a_stages);
    // Token stages: a ring of NB (narrow tiles; a stage is freed by the
    // epilogue once the step's MMAs are complete, so the token producer runs
    // NB - 1 steps ahead of the MMAs and the L2 latency of the token tiles is
    // off the critical path), or the two step slots (wide tiles, NB == 2,
    // freed by the step's commit).
    const uint32_t NB = static_cast<uint32_t>(p.b_stages);
    // Wide dense tiles: each stage's two K-group halves have their own
    // barriers, so group j's tokens are requested as soon as group j's MMAs of
    // the step that last used the stage are done (4096x8192x8192 GEMM: 640 ->
    // 627 us, measured); MoE expert tiles (a few steps each) were slower that
    // way (gate_up 266 -> 273 us) and keep whole-step stages.
    const bool gt = kWide && p.group_tokens != 0;
    const int b_rows = p.b_rows;                          // 32 or 64; 128 when kWide
    const uint32_t b_atom_bytes = static_cast<uint32_t>(b_rows) * 128u;
    const uint32_t b_stage_bytes = 4u * b_atom_bytes;     // 2 groups x 2 atoms
    const uint32_t sA = base + kStagesOff;
    const uint32_t sB = sA + SA * kNarrowAStageBytes;
    const uint32_t sBar = base + kOffBar;
    volatile uint32_t *s_tmem_base = reinterpret_cast<volatile uint32_t *>(smem + kOffMisc);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);
    volatile int *s_total = reinterpret_cast<volatile int *>(smem + kOffMisc + 8);
    volatile int *s_last = reinterpret_cast<volatile int *>(smem + kOffMisc + 12);
    const int tab_stride = kWide ? p.E + 1 : kMaxExperts + 1;
    int *s_base = reinterpret_cast<int *>(smem + (kWide ? kWideOffTab : kOffTab));
    int *s_lo = s_base + tab_stride;
    int *s_cnt = s_lo + tab_stride;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tt = p.tile_tokens;                         // == b_rows
    auto bar = [&](int i) -> uint32_t { return sBar + 8u * static_cast<uint32_t>(i); };
    // No griddepcontrol.launch_dependents here: the kernels of the next call
    // (programmatic dependents) then launch only when this grid completes.
    // Releasing them at the start, so that the next GEMM's CTAs stream
    // weights on SMs this grid frees, made a decode step slower (measured:
    // 162 -> 170 us).

    if (threadIdx.x == 0) {
        for (int i = 0; i < kMaxAStages; ++i) {
            mbar_init(bar(NBar::a_full + i), 1);
            mbar_init(bar(NBar::a_empty + i), 4);
        }
        for (int i = 0; i < kNarrowSlots; ++i) {
            mbar_init(bar(NBar::ready + i), 5);
            mbar_init(bar(NBar::done + i), 1);
            // the epilogue warps that drain partials: both warpgroups, or only
            // the first for token tiles of <= 32 rows (the second one then
            // combines split tiles; see the epilogue)
            mbar_init(bar(NBar::p_empty + i), (!kWide && p.b_rows <= 32) ? 4 : 8);
            mbar_init(bar(NBar::p_full + i), 1);
        }
        for (int i = 0; i < kMaxBStages; ++i) {
            mbar_init(bar(NBar::b_full + i), 1);
            mbar_init(bar(NBar::b_empty + i), 1);
        }
        mbar_init(bar(NBar::drain), 1);
        *s_abort = 0;
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmap_w);
        tma_prefetch_desc(&tmap_x);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(smem + kOffMisc), kTmemCols);
        tmem_relinquish();
    }
    if (warp == 2) build_tile_table(p, tt, lane, s_base, s_lo, s_cnt, s_total);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem_base = *s_tmem_base;
    const int total = *s_total;
    const int G = p.G;
    const int wg = warp >> 2;
    // Wide tiles are never split (their two accumulators leave no registers
    // for the bookkeeping).
    const WorkPlan plan = make_plan(total, G, !kWide && p.sk_cnt != nullptr);
    constexpr int kEpiR = kWide ? kEpiRegs : kSplitEpiRegs;
    constexpr int kOthR = kWide ? kOtherRegs : kSplitOtherRegs;
    // TMEM: partial buffer of (partial slot s, group j) at column
    // (2 s + j) * b_rows; fp16 A operand of (step slot s, group j) at column
    // 256 + 128 s + 64 j.
    auto pbuf_col = [&](uint32_t s, int j) -> uint32_t {
        return (2u * s + static_cast<uint32_t>(j)) * static_cast<uint32_t>(b_rows);
    };

    if (warp < 4) {
        setmaxnreg_dec<kOthR>();
        if (warp == 0 && lane == 0) {
            // ------------------------------------------- weight TMA producer
            Ring a;
            uint32_t issued = 0;
            bool ok = true;
            for_each_piece(plan, [&](int t, int s0, int s1) -> bool {
                const TileInfo ti = decode_tile(t, s_base, s_lo, s_cnt, p.E, tt, p.n_tiles, p.gw);
                const int wrow = ti.e * p.N + ti.n0;
                for (int sg = s0; sg < s1; ++sg) {
                    const int g0 = 2 * sg;
                    const int ng = min(2, G - g0);
                    if (!mbar_wait(bar(NBar::a_empty + a.idx), a.phase ^ 1u, s_abort, p.err,
                                   ROLE_PRODUCER, 1)) {
                        ok = false;
                        return false;
                    }
                    mbar_arrive_expect_tx(bar(NBar::a_full + a.idx), ng * kAStageBytes);
                    for (int j = 0; j < ng; ++j)
                        tma_load_2d(sA + a.idx * kNarrowAStageBytes + j * kAStageBytes, &tmap_w,
                                    (g0 + j) * kGroupK, wrow, bar(NBar::a_full + a.idx));
                    a.advance(SA);
                    ++issued;
                }
                return true;
            });
            if (!ok) drain_ring(bar(NBar::a_full), issued, SA);
        } else if (warp == 1 && lane == 0) {
            // ------------------------------------------------- MMA issuer
            Ring st, pr, bs;
            uint32_t gph[2] = {0u, 0u};   // wide: phase of each group's partial buffer
            bool ok = true;
            for_each_piece(plan, [&](int t, int s0, int s1) -> bool {
                const TileInfo ti = decode_tile(t, s_base, s_lo, s_cnt, p.E, tt, p.n_tiles, p.gw);
                const int n_eff = (ti.rows + 15) & ~15;
                const uint32_t idesc = kA16 ? idesc_bf16_f32(kTileN, static_cast<uint32_t>(n_eff))
                                            : idesc_f16_f32(kTileN, static_cast<uint32_t>(n_eff));
                for (int sg = s0; sg < s1; ++sg) {
                    const int g0 = 2 * sg;
                    const int ng = min(2, G - g0);
                    if (!mbar_wait(bar(NBar::ready + st.idx), st.phase, s_abort, p.err, ROLE_MMA,
                                   1)) {
                        ok = false;
                        return false;
                    }
                    tc_fence_after();
                    for (int j = 0; j < ng; ++j) {
                        if constexpr (kWide) {
                            // group j's partial buffer drained by the epilogue;
                            // group 1's tokens landed (admission covered group 0's)
                            if (!mbar_wait(bar(NBar::p_empty + j), gph[j] ^ 1u, s_abort, p.err,
                                           ROLE_MMA, 4) ||
                                (gt && j == 1 &&
                                 !mbar_wait(bar(NBar::b_full + 2 * bs.idx + 1), bs.phase, s_abort,
                                            p.err, ROLE_MMA, 5))) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                        }
                        const uint32_t d_tmem = tmem_base + pbuf_col(pr.idx, j);
                        const uint32_t a_tmem = tmem_base + kTmemA0 + st.idx * 128u + j * 64u;
                        const uint64_t bdesc0 = smem_desc_sw128(sB + bs.idx * b_stage_bytes +
                                                                j * 2u * b_atom_bytes);
                        const uint64_t atom_step = b_atom_bytes >> 4;
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint64_t bdesc =
                                bdesc0 + (kk >> 2) * atom_step + static_cast<uint64_t>((kk & 3) * 2);
                            mma_f16_tmemA(d_tmem, a_tmem + kk * 8, bdesc, idesc, kk > 0 ? 1u : 0u);
                        }
                        if constexpr (kWide) {
                            mma_commit(bar(NBar::p_full + j));
                            gph[j] ^= 1u;
                        }
                    }
                    if (!ok) return false;
                    mma_commit(bar(NBar::done + st.idx));
                    st.advance(kNarrowSlots);
                    pr.advance(NP);
                    bs.advance(NB);
                }
                return true;
            });
            mma_commit(bar(NBar::drain));
            drain_wait(bar(NBar::drain), 0);
        } else if (warp == 2 && lane == 0) {
            // -------------------------------------------- token TMA producer
            griddep_wait();   // the fp16 token codes come from the kernel launched before
            Ring bs;
            uint32_t issued = 0;
            bool ok = true;
            for_each_piece(plan, [&](int t, int s0, int s1) -> bool {
                const TileInfo ti = decode_tile(t, s_base, s_lo, s_cnt, p.E, tt, p.n_tiles, p.gw);
                const int n_eff = (ti.rows + 15) & ~15;
                const int nbox = (n_eff + kBoxRows - 1) / kBoxRows;
                for (int sg = s0; sg < s1; ++sg) {
                    const int g0 = 2 * sg;
                    const int ng = min(2, G - g0);
                    const uint32_t stage = sB + bs.idx * b_stage_bytes;
                    if (kWide && gt) {
                        // One barrier pair per group half of the stage: group j's
                        // tokens are requested as soon as group j's MMAs of the
                        // step that last used the stage are done (a missing
                        // second group completes its barrier empty).
                        for (int j = 0; j < 2; ++j) {
                            const uint32_t gb = 2u * bs.idx + static_cast<uint32_t>(j);
                            if (!mbar_wait(bar(NBar::b_empty + gb), bs.phase ^ 1u, s_abort,
                                           p.err, ROLE_PRODUCER, 2)) {
                                ok = false;
                                return false;
                            }
                            if (j < ng) {
                                mbar_arrive_expect_tx(
                                    bar(NBar::b_full + gb),
                                    static_cast<uint32_t>(2 * nbox * kBoxRows * 128));
                                for (int a = 0; a < 2; ++a)
                                    for (int i = 0; i < nbox; ++i)
                                        tma_load_2d(stage + (2 * j + a) * b_atom_bytes +
                                                        i * kBoxRows * 128,
                                                    &tmap_x, (g0 + j) * kGroupK + a * 64,
                                                    ti.m0 + i * kBoxRows, bar(NBar::b_full + gb));
                            } else {
                                mbar_arrive(bar(NBar::b_full + gb));
                            }
                            ++issued;
                        }
                        bs.advance(NB);
                        continue;
                    }
                    // narrow: the ring stage is freed by the epilogue; wide (whole
                    // steps): the stage is the step slot, freed by its commit
                    if (!mbar_wait(bar((kWide ? NBar::done : NBar::b_empty) + bs.idx),
                                   bs.phase ^ 1u, s_abort, p.err, ROLE_PRODUCER, 2)) {
                        ok = false;
                        return false;
                    }
                    mbar_arrive_expect_tx(bar(NBar::b_full + bs.idx),
                                          static_cast<uint32_t>(ng * 2 * nbox * kBoxRows * 128));
                    for (int j = 0; j < ng; ++j)
                        for (int a = 0; a < 2; ++a)
                            for (int i = 0; i < nbox; ++i)
                                tma_load_2d(stage + (2 * j + a) * b_atom_bytes + i * kBoxRows * 128,
                                            &tmap_x, (g0 + j) * kGroupK + a * 64,
                                            ti.m0 + i * kBoxRows, bar(NBar::b_full + bs.idx));
                    bs.advance(NB);
                    ++issued;
                }
                return true;
            });
            // wide: group barriers in issue order 0,1,2,3,0,...
            if (!ok) drain_ring(bar(NBar::b_full), issued, (kWide && gt) ? 2 * NB : NB);
        } else if (warp == 3 && lane == 0) {
            // --------------------------------------------------- admission
            Ring st, pr, bs;
            for_each_piece(plan, [&](int, int s0, int s1) -> bool {
                for (int sg = s0; sg < s1; ++sg) {
                    if (!mbar_wait(bar(NBar::b_full + ((kWide && gt) ? 2 * bs.idx : bs.idx)),
                                   bs.phase, s_abort, p.err, ROLE_MMA, 2) ||
                        (!kWide && !mbar_wait(bar(NBar::p_empty + pr.idx), pr.phase ^ 1u, s_abort,
                                              p.err, ROLE_MMA, 3)))
                        return false;
                    mbar_arrive(bar(NBar::ready + st.idx));
                    st.advance(kNarrowSlots);
                    pr.advance(NP);
                    bs.advance(NB);
                }
                return true;
            });
        }
    } else if (wg == 1) {
        // --------------------------------------- weight converter (A -> TMEM)
        setmaxnreg_dec<kOthR>();
        const int row = threadIdx.x - 128;
        const int q = warp & 3;
        Ring a, st;
        for_each_piece(plan, [&](int, int s0, int s1) -> bool {
            for (int sg = s0; sg < s1; ++sg) {
                const int g0 = 2 * sg;
                const int ng = min(2, G - g0);
                if (!mbar_wait(bar(NBar::a_full + a.idx), a.phase, s_abort, p.err, ROLE_CONVERT,
                               1) ||
                    !mbar_wait(bar(NBar::done + st.idx), st.phase ^ 1u, s_abort, p.err,
                               ROLE_CONVERT, 2))
                    return false;
                tc_fence_after();
                for (int j = 0; j < ng; ++j) {
                    const uint8_t *rowp =
                        smem + kStagesOff + a.idx * kNarrowAStageBytes + j * kAStageBytes + row * 128;
                    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                           kTmemA0 + st.idx * 128u + j * 64u;
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        uint32_t r16[16];
#pragma unroll
                        for (int cc = 0; cc < 2; ++cc) {
                            const int c = 2 * jj + cc;
                            const uint4 v =
                                *reinterpret_cast<const uint4 *>(rowp + ((c ^ (row & 7)) << 4));
                            i8x4_to_op<kA16>(v.x, r16[cc * 8 + 0], r16[cc * 8 + 1]);
                            i8x4_to_op<kA16>(v.y, r16[cc * 8 + 2], r16[cc * 8 + 3]);
                            i8x4_to_op<kA16>(v.z, r16[cc * 8 + 4], r16[cc * 8 + 5]);
                            i8x4_to_op<kA16>(v.w, r16[cc * 8 + 6], r16[cc * 8 + 7]);
                        }
                        tmem_st_16cols(taddr + jj * 16, r16);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(NBar::a_empty + a.idx));
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(NBar::ready + st.idx));
                a.advance(SA);
                st.advance(kNarrowSlots);
            }
            return true;
        });
    } else {
        // -------------------------------------------------------- epilogue
        setmaxnreg_inc<kEpiR>();
        // The token scales come from the kernel launched before (which lets
        // this grid start early): no read of them before that grid is done.
        griddep_wait();
        const int ewg = wg - 2;   // owns token columns [32 c, 32 c + 32) for chunks c = ewg + 2 h
        const int q = warp & 3;
        const int lrow = q * 32 + lane;
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        float *s_sa = reinterpret_cast<float *>(smem + kOffTokScales) + 32 * NCH * ewg;
        // 2 consecutive outputs of a row per store: N even and y aligned for it
        const bool vec_y = (p.N & 1) == 0 &&
                           (reinterpret_cast<uintptr_t>(p.y) & (p.out_fp32 ? 7u : 3u)) == 0;
        const bool vec_sw = (G % 4 == 0) && ((reinterpret_cast<uintptr_t>(p.sw) & 15u) == 0);
        auto store_out = [&](int m, int n_local, float v) {
            const float out = v;
            const size_t idx = static_cast<size_t>(m) * p.N + n_local;
            if (p.out_fp32)
                static_cast<float *>(p.y)[idx] = out;
            else
                static_cast<__nv_bfloat16 *>(p.y)[idx] = __float2bfloat16_rn(out);
        };
        // Token tiles of <= 32 rows leave the second epilogue warpgroup without
        // columns: it takes no part in the steps (the partial-buffer release
        // counts 4 warps) and instead finishes the split tiles. At the end of
        // each split piece the first warpgroup stores its partial and goes on
        // with the next piece at once; this one counts the piece in and, for
        // the tile's last piece, adds all pieces in K order and stores y, off
        // the MMA pipeline's critical path.
        const bool helper = !kWide && p.b_rows <= 32;
        if (helper && ewg == 1) {
            for_each_piece(plan, [&](int t, int s0, int s1) -> bool {
                if (s0 == 0 && s1 == plan.S) return true;
                named_barrier_sync(2, 256);   // the piece's partial is stored
                const TileInfo ti = decode_tile(t, s_base, s_lo, s_cnt, p.E, tt, p.n_tiles, p.gw);
                int c_first, c_final;
                tile_owners(t, plan, c_first, c_final);
                if (threadIdx.x == 384) {
                    int last = 0;
                    if (*s_abort == 0) {
                        // ordered after the kernel that zeroed the counters
                        griddep_wait();
                        __threadfence();
                        last = atomicAdd(p.sk_cnt + (t - plan.dp), 1) == c_final - c_first;
                        if (last) __threadfence();
                    }
                    *s_last = last;
                }
                named_barrier_sync(3, 128);
                const int n_local = ti.n0 + lrow;
                if (*s_last == 0 || n_local >= p.N) return true;
                auto slot = [&](int c) -> const float * {   // slot 1: the tile's first piece
                    return p.sk_part +
                           static_cast<size_t>(2 * c + (c == c_first ? 1 : 0)) * p.sk_ld * kTileN +
                           lrow;
                };
                // (off the critical path: one piece per round trip)
                float sum[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) sum[j] = 0.0f;
                for (int c = c_first; c <= c_final; ++c) {   // K order
                    const float *src = slot(c);
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __ldcg(src + min(j, ti.rows - 1) * kTileN);
#pragma unroll
                    for (int j = 0; j < 32; ++j) sum[j] += v[j];
                }
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    if (j < ti.rows) {
                        const size_t idx = static_cast<size_t>(ti.m0 + j) * p.N + n_local;
                        const float out = sum[j] * load_sa(p, ti.m0 + j);
                        if (p.out_fp32)
                            static_cast<float *>(p.y)[idx] = out;
                        else
                            static_cast<__nv_bfloat16 *>(p.y)[idx] = __float2bfloat16_rn(out);
                    }
                }
                return true;
            });
        } else {
        float acc[NCH][32];
#pragma unroll
        for (int h = 0; h < NCH; ++h)
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[h][j] = 0.0f;
        Ring st, pr, bs;
        uint32_t gph[2] = {0u, 0u};   // wide: phase of each group's partial buffer
        // After a failed wait the threads keep walking the same pieces with
        // no waits and no data work, so that every epilogue warp takes the
        // same named barriers at split pieces.
        bool failed = false;
        for_each_piece(plan, [&](int t, int s0, int s1) -> bool {
            const TileInfo ti = decode_tile(t, s_base, s_lo, s_cnt, p.E, tt, p.n_tiles, p.gw);
            const int n_eff = (ti.rows + 15) & ~15;
            const bool owned = 32 * ewg < n_eff;   // warp-uniform (first chunk)
            const int n_local = ti.n0 + lrow;
            const bool n_ok = n_local < p.N;
            const float *swp =
                p.sw + (static_cast<size_t>(ti.e) * p.sw_rows + ((n_ok ? n_local : 0) >> p.sw_shift)) * G;
            // Token scales of a whole tile's columns (this warpgroup's chunks),
            // copied into shared memory now, one per thread, and read at the
            // store: the copies land while the tile's steps run. (Loaded into
            // registers instead, they were waited for at the store, ~1.5 us
            // per tile under the weight stream.) The barrier first lets the
            // warpgroup finish reading the previous tile's.
            const bool whole = s0 == 0 && s1 == plan.S;
            if (whole) {
                named_barrier_sync(4 + ewg, 128);
                if (lrow < 32 * NCH) {
                    const int col = 32 * (ewg + 2 * (lrow >> 5)) + (lrow & 31);
                    if (p.sa != nullptr)
                        cp_async_4(smem_u32(s_sa + lrow), p.sa + ti.m0 + min(col, ti.rows - 1),
                                   col < ti.rows ? 4u : 0u);
                    else
                        s_sa[lrow] = 1.0f;
                }
            }
            // Scales of this row a quad of groups (two steps) ahead; loads are
            // issued in place and only read after the next quad boundary.
            auto load_quad = [&](int g) -> float4 {
                float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                if (!n_ok || !owned || failed) return v;
                if (vec_sw) {
                    if (g < G) v = ldg_nc_f32x4_now(swp + g);
                } else {
                    if (g < G) v.x = ldg_nc_f32_now(swp + g);
                    if (g + 1 < G) v.y = ldg_nc_f32_now(swp + g + 1);
                    if (g + 2 < G) v.z = ldg_nc_f32_now(swp + g + 2);
                    if (g + 3 < G) v.w = ldg_nc_f32_now(swp + g + 3);
                }
                return v;
            };
            const int qb = (2 * s0) & ~3;
            float4 cur = load_quad(qb);
            float4 nxt = load_quad(qb + 4);
            for (int sg = s0; sg < s1; ++sg) {
                const int g0 = 2 * sg;
                const int ng = min(2, G - g0);
                if ((g0 & 3) == 0 && g0 > qb) {
                    cur = nxt;
                    nxt = load_quad(g0 + 4);
                }
                const float sc0 = (g0 & 3) == 0 ? cur.x : cur.z;
                const float sc1 = (g0 & 3) == 0 ? cur.y : cur.w;
                if (failed) continue;
                if constexpr (kWide) {
                    // One group at a time: wait for its MMAs, drain its buffer,
                    // release it (group 0 drains while group 1's MMAs issue).
                    for (int j = 0; j < ng; ++j) {
                        const bool ok = mbar_wait(bar(NBar::p_full + j), gph[j], s_abort, p.err,
                                                  ROLE_EPILOGUE, 2);
                        if (__any_sync(0xFFFFFFFFu, !ok)) {   // the warp fails as one
                            failed = true;
                            break;
                        }
                        gph[j] ^= 1u;
                        // group j's MMAs are complete: its token half-stage is free
                        if (gt && threadIdx.x == 256)
                            mbar_arrive(bar(NBar::b_empty + 2 * bs.idx + j));
                        tc_fence_after();
                        const float sj = j == 0 ? sc0 : sc1;
                        uint32_t v[2][32];
#pragma unroll
                        for (int h = 0; h < NCH; ++h) {
                            const int chunk = ewg + 2 * h;
                            if (32 * chunk >= n_eff) continue;   // warp-uniform
                            tmem_ld_32cols_sync(lane_base + pbuf_col(0, j) + 32u * chunk, v[h]);
#pragma unroll
                            for (int jj = 0; jj < 32; ++jj)
                                acc[h][jj] = fmaf(__uint_as_float(v[h][jj]), sj, acc[h][jj]);
                            if (kDebug && n_ok) {
#pragma unroll
                                for (int jj = 0; jj < 32; ++jj) {
                                    const int col = 32 * chunk + jj;
                                    if (col < ti.rows)
                                        p.dbg[(static_cast<size_t>(ti.m0 + col) * p.N + n_local) * G +
                                              g0 + j] = __float2int_rn(__uint_as_float(v[h][jj]));
                                }
                            }
                        }
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive_relaxed(bar(NBar::p_empty + j));
                    }
                    if (!failed) {
                        // a step with one group releases the unused half at once
                        if (gt && ng == 1 && threadIdx.x == 256)
                            mbar_arrive(bar(NBar::b_empty + 2 * bs.idx + 1));
                        bs.advance(NB);
                    }
                    continue;
                }
                const bool ok =
                    mbar_wait(bar(NBar::done + st.idx), st.phase, s_abort, p.err, ROLE_EPILOGUE, 1);
                if (__any_sync(0xFFFFFFFFu, !ok)) {   // the warp fails as one
                    failed = true;
                    continue;
                }
                // The step's MMAs are complete: its token stage is free.
                if (threadIdx.x == 256) mbar_arrive(bar(NBar::b_empty + bs.idx));
                bs.advance(NB);
                tc_fence_after();
#pragma unroll
                for (int h = 0; h < NCH; ++h) {
                    const int chunk = ewg + 2 * h;
                    if (32 * chunk >= n_eff) continue;   // warp-uniform
                    const uint32_t c0 = lane_base + pbuf_col(pr.idx, 0) + 32u * chunk;
                    const uint32_t c1 = lane_base + pbuf_col(pr.idx, 1) + 32u * chunk;
                    uint32_t v0[32], v1[32];
                    if (ng == 2) {
                        tmem_ld_2x32cols_sync(c0, c1, v0, v1);
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            acc[h][j] = fmaf(__uint_as_float(v1[j]), sc1,
                                             fmaf(__uint_as_float(v0[j]), sc0, acc[h][j]));
                    } else {
                        tmem_ld_32cols_sync(c0, v0);
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            acc[h][j] = fmaf(__uint_as_float(v0[j]), sc0, acc[h][j]);
                    }
                    if (kDebug && n_ok) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const int col = 32 * chunk + j;
                            if (col < ti.rows) {
                                const size_t o =
                                    (static_cast<size_t>(ti.m0 + col) * p.N + n_local) * G + g0;
                                p.dbg[o] = __float2int_rn(__uint_as_float(v0[j]));
                                if (ng == 2) p.dbg[o + 1] = __float2int_rn(__uint_as_float(v1[j]));
                            }
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_relaxed(bar(NBar::p_empty + pr.idx));
                st.advance(kNarrowSlots);
                pr.advance(NP);
            }
            if (whole) {
                // the warpgroup's copies have landed once all its threads pass
                cp_async_wait_all();
                named_barrier_sync(4 + ewg, 128);
                if (vec_y) {
                    // Lane pairs (two consecutive weight rows n) swap one value
                    // per pair of token columns, so that each lane stores two
                    // consecutive n of one column in one 4-byte (BF16) or
                    // 8-byte (FP32) store: half the store instructions (MoE
                    // gate_up 258 -> 249 us, down 161 -> 148 us; a four-lane
                    // transpose with a quarter of the stores measured no faster).
                    const bool odd = lane & 1;
                    const size_t nb = static_cast<size_t>(n_local & ~1);
                    auto pairs = [&](auto store2) {
#pragma unroll
                        for (int h = 0; h < NCH; ++h) {
#pragma unroll
                            for (int j = 0; j < 32; j += 2) {
                                const float v0 = acc[h][j] * s_sa[32 * h + j];
                                const float v1 = acc[h][j + 1] * s_sa[32 * h + j + 1];
                                const float recv =
                                    __shfl_xor_sync(0xFFFFFFFFu, odd ? v0 : v1, 1);
                                const int col = 32 * (ewg + 2 * h) + j + (odd ? 1 : 0);
                                if (n_ok && !failed && col < ti.rows)
                                    store2(static_cast<size_t>(ti.m0 + col) * p.N + nb,
                                           odd ? recv : v0, odd ? v1 : recv);
                            }
                        }
                    };
                    if (p.out_fp32)
                        pairs([&](size_t idx, float lo, float hi) {
                            *reinterpret_cast<float2 *>(static_cast<float *>(p.y) + idx) =
                                make_float2(lo, hi);
                        });
                    else
                        pairs([&](size_t idx, float lo, float hi) {
                            *reinterpret_cast<__nv_bfloat162 *>(static_cast<__nv_bfloat16 *>(p.y) +
                                                                idx) = __floats2bfloat162_rn(lo, hi);
                        });
                } else if (n_ok && !failed) {
#pragma unroll
                    for (int h = 0; h < NCH; ++h) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const int col = 32 * (ewg + 2 * h) + j;
                            if (col < ti.rows)
                                store_out(ti.m0 + col, n_local, acc[h][j] * s_sa[32 * h + j]);
                        }
                    }
                }
            } else if constexpr (!kWide) {
                // Split piece: store its partial ([token column][weight row],
                // FP32, before sa), then count it in. The CTA that brings
                // the tile's last piece adds all pieces in K order (its own
                // from registers) and stores y. The other roles run on
                // meanwhile; the MMAs of the next steps fill the two
                // partial-buffer slots.
                const int me = static_cast<int>(blockIdx.x);
                int c_first, c_final;
                tile_owners(t, plan, c_first, c_final);
                auto slot = [&](int c) -> const float * {   // slot 1: the tile's first piece
                    return p.sk_part +
                           static_cast<size_t>(2 * c + (c == c_first ? 1 : 0)) * p.sk_ld * kTileN;
                };
                const int col0 = 32 * ewg;
                const bool mine = n_ok && !failed && col0 < ti.rows;
                if (mine) {
                    float *dst = const_cast<float *>(slot(me)) + lrow;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (col0 + j < ti.rows) __stcg(dst + (col0 + j) * kTileN, acc[0][j]);
                }
                if (helper) {
                    // the other warpgroup publishes and combines (above)
                    named_barrier_arrive(2, 256);
#pragma unroll
                    for (int j = 0; j < 32; ++j) acc[0][j] = 0.0f;
                    return true;
                }
                // Release: the barrier orders every epilogue thread's partial
                // stores before one thread's fence and counter update (fences
                // are cumulative); the last arrival's fence then orders its
                // reads of the other pieces after their release.
                named_barrier_sync(1, 256);
                if (threadIdx.x == 256) {
                    int last = 0;
                    if (*s_abort == 0) {
                        // Orders the counter update after the kernel before
                        // this one in the stream, which zeroed the counters
                        // (returns at once: the token producer has waited).
                        griddep_wait();
                        __threadfence();
                        last = atomicAdd(p.sk_cnt + (t - plan.dp), 1) == c_final - c_first;
                        if (last) __threadfence();
                    }
                    *s_last = last;
                }
                named_barrier_sync(1, 256);
                if (*s_last != 0 && mine) {
                    // Token scales loaded ahead of the pieces (the debug
                    // form loads them at the store: fewer live registers).
                    float sa_r[32], sum[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        sa_r[j] = kDebug ? 0.0f : load_sa(p, ti.m0 + min(col0 + j, ti.rows - 1));
                        sum[j] = 0.0f;
                    }
                    for (int c = c_first; c <= c_final; ++c) {   // K order
                        if (c == me) {
#pragma unroll
                            for (int j = 0; j < 32; ++j) sum[j] += acc[0][j];
                        } else {
                            const float *src = slot(c) + lrow;
                            float v[32];
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                v[j] = __ldcg(src + min(col0 + j, ti.rows - 1) * kTileN);
#pragma unroll
                            for (int j = 0; j < 32; ++j) sum[j] += v[j];
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if (col0 + j < ti.rows) {
                            const size_t idx =
                                static_cast<size_t>(ti.m0 + col0 + j) * p.N + n_local;
                            const float out =
                                sum[j] * (kDebug ? load_sa(p, ti.m0 + col0 + j) : sa_r[j]);
                            if (p.out_fp32)
                                static_cast<float *>(p.y)[idx] = out;
                            else
                                static_cast<__nv_bfloat16 *>(p.y)[idx] = __float2bfloat16_rn(out);
                        }
                    }
                }
            }
#pragma unroll
            for (int h = 0; h < NCH; ++h)
#pragma unroll
                for (int j = 0; j < 32; ++j) acc[h][j] = 0.0f;
            return true;
        });
        }   // draining warpgroups
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// =============================================================================
// Large dense problems (at least 256 token rows): tiles of 128 weight rows x
// 192 token rows, one K group per pipeline step, and one tcgen05.mma of
// N = 192 per 16 K. On this part an MMA instruction costs about the same
// whatever its token columns (~130-155 cycles at M = 128, K = 16 for N up to
// 256, measured with w8a8_probe_tc_rate), so wide instructions pay.
// Tensor memory: two buffers of a group's exact partial sums in columns
// [0, 192) and [192, 384), so the MMAs of group g + 1 run while the epilogue
// drains group g (with one 256-column buffer every group's MMAs waited for
// the previous group's drain), and the fp16 A operand (weights) of two groups
// in columns [384, 512), 64 each, so the converter runs a group ahead.
// Shared memory (exactly the 227 KB limit): four 48 KB token stages (192 rows
// x 128 K fp16, two 128-byte swizzle atom columns) and two 16 KB weight
// stages.
// Warp roles: 0 weight TMA producer; 1 MMA issuer and TMEM allocation; 2
// token TMA producer (waits for the kernel that wrote the codes); 4-7
// converter (int8 -> fp16 A operand in TMEM); 8-15 epilogue: warpgroup h
// drains token columns [96 h, 96 h + 96) of every lane (weight row), fma
// with sw[n, g] into 96 register accumulators per thread, and at the end of
// the tile multiplies by sa[m] and stores.
// =============================================================================
constexpr int kW2Tokens = 192;
constexpr int kW2TokStages = 4;
constexpr int kW2WStages = 2;
constexpr int kW2ASlots = 2;
constexpr int kW2Bufs = 2;                                  // partial-sum buffers in TMEM
constexpr int kW2Half = kW2Tokens / 2;                      // token columns per epilogue warpgroup
constexpr int kW2OffStages = 2048;
constexpr int kW2AtomBytes = kW2Tokens * 128;              // one 128-byte atom column, 24 KB
constexpr int kW2TokStageBytes = 2 * kW2AtomBytes;          // one K group of tokens, 48 KB
constexpr int kW2SmemBytes =
    kW2OffStages + kW2TokStages * kW2TokStageBytes + kW2WStages * kAStageBytes + 1024;
static_assert(kW2SmemBytes <= kSmemLimit, "wide-tile shared memory");
static_assert(kW2Half % 32 == 0, "32-column chunks per epilogue warpgroup");
constexpr uint32_t kW2TmemA0 = kW2Bufs * kW2Tokens;
static_assert(kW2TmemA0 + 64 * kW2ASlots <= kTmemCols, "wide-tile tensor memory");
// Token scales of the current tile, 96 per epilogue warpgroup, in the fixed
// area: after the barriers, and after the tile table of a dense call.
constexpr int kW2OffSa0 = 256;
constexpr int kW2OffSa1 = 1536;

struct W2Bar {
    static constexpr int a_full = 0;                       // [kW2WStages] weight TMA -> converter
    static constexpr int a_empty = a_full + kW2WStages;    // [kW2WStages] converter (4) -> weight TMA
    static constexpr int b_full = a_empty + kW2WStages;    // [kW2TokStages] token TMA -> MMA
    static constexpr int b_empty = b_full + kW2TokStages;  // [kW2TokStages] MMA commit -> token TMA
    static constexpr int a_ready = b_empty + kW2TokStages; // [kW2ASlots] converter (4) -> MMA
    static constexpr int a_free = a_ready + kW2ASlots;     // [kW2ASlots] MMA commit -> converter
    static constexpr int d_full = a_free + kW2ASlots;      // [kW2Bufs] MMA commit -> epilogue
    static constexpr int d_empty = d_full + kW2Bufs;       // [kW2Bufs] epilogue (8 warps) -> MMA
    static constexpr int drain = d_empty + kW2Bufs;
    static constexpr int count = drain + 1;
};
static_assert(W2Bar::count <= 128, "barrier area");
static_assert(W2Bar::count * 8 <= kW2OffSa0 && kW2OffSa0 + 512 <= kOffMisc, "token-scale area 0");
static_assert(kWideOffTab + 3 * 2 * 4 <= kW2OffSa1 && kW2OffSa1 + 512 <= kW2OffStages,
              "token-scale area 1 (dense calls: one expert)");

template <bool kDebug, bool kA16 = false>
__global__ void __launch_bounds__(kThreads, 1)
w8a8_gemm_wide_kernel(const __grid_constant__ CUtensorMap tmap_w,
                      const __grid_constant__ CUtensorMap tmap_x, const KParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw_addr);
    const uint32_t sTok = base + kW2OffStages;
    const uint32_t sW = sTok + kW2TokStages * kW2TokStageBytes;
    const uint32_t sBar = base + kOffBar;
    volatile uint32_t *s_tmem_base = reinterpret_cast<volatile uint32_t *>(smem + kOffMisc);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);
    volatile int *s_total = reinterpret_cast<volatile int *>(smem + kOffMisc + 8);
    int *s_base = reinterpret_cast<int *>(smem + kWideOffTab);
    int *s_lo = s_base + (p.E + 1);
    int *s_cnt = s_lo + (p.E + 1);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    auto bar = [&](int i) -> uint32_t { return sBar + 8u * static_cast<uint32_t>(i); };

    if (threadIdx.x == 0) {
        for (int i = 0; i < kW2WStages; ++i) {
            mbar_init(bar(W2Bar::a_full + i), 1);
            mbar_init(bar(W2Bar::a_empty + i), 4);
        }
        for (int i = 0; i < kW2TokStages; ++i) {
            mbar_init(bar(W2Bar::b_full + i), 1);
            mbar_init(bar(W2Bar::b_empty + i), 1);
        }
        for (int i = 0; i < kW2ASlots; ++i) {
            mbar_init(bar(W2Bar::a_ready + i), 4);
            mbar_init(bar(W2Bar::a_free + i), 1);
        }
        for (int i = 0; i < kW2Bufs; ++i) {
            mbar_init(bar(W2Bar::d_full + i), 1);
            mbar_init(bar(W2Bar::d_empty + i), 8);
        }
        mbar_init(bar(W2Bar::drain), 1);
        *s_abort = 0;
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmap_w);
        tma_prefetch_desc(&tmap_x);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(smem + kOffMisc), kTmemCols);
        tmem_relinquish();
    }
    if (warp == 2) build_tile_table(p, kW2Tokens, lane, s_base, s_lo, s_cnt, s_total);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem_base = *s_tmem_base;
    const int total = *s_total;
    const int G = p.G;
    const int grid = static_cast<int>(gridDim.x);
    const int wg = warp >> 2;
    auto tile_of = [&](int t) -> TileInfo {
        return decode_tile(t, s_base, s_lo, s_cnt, p.E, kW2Tokens, p.n_tiles, p.gw);
    };

    if (warp < 4) {
        setmaxnreg_dec<kOtherRegs>();
        if (warp == 0 && lane == 0) {
            // ------------------------------------------- weight TMA producer
            Ring a;
            uint32_t issued = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += grid) {
                const TileInfo ti = tile_of(t);
                const int wrow = ti.e * p.N + ti.n0;
                for (int g = 0; g < G; ++g) {
                    if (!mbar_wait(bar(W2Bar::a_empty + a.idx), a.phase ^ 1u, s_abort, p.err,
                                   ROLE_PRODUCER, 11)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar(W2Bar::a_full + a.idx), kAStageBytes);
                    tma_load_2d(sW + a.idx * kAStageBytes, &tmap_w, g * kGroupK, wrow,
                                bar(W2Bar::a_full + a.idx));
                    a.advance(kW2WStages);
                    ++issued;
                }
            }
            if (!ok) drain_ring(bar(W2Bar::a_full), issued, kW2WStages);
        } else if (warp == 1 && lane == 0) {
            // ------------------------------------------------- MMA issuer
            Ring b, sl, d;   // token stage, A slot, partial buffer
            bool ok = true;
            const uint32_t idesc =
                kA16 ? idesc_bf16_f32(kTileN, kW2Tokens) : idesc_f16_f32(kTileN, kW2Tokens);
            for (int t = blockIdx.x; t < total && ok; t += grid) {
                for (int g = 0; g < G; ++g) {
                    if (!mbar_wait(bar(W2Bar::a_ready + sl.idx), sl.phase, s_abort, p.err,
                                   ROLE_MMA, 11) ||
                        !mbar_wait(bar(W2Bar::b_full + b.idx), b.phase, s_abort, p.err, ROLE_MMA,
                                   12) ||
                        !mbar_wait(bar(W2Bar::d_empty + d.idx), d.phase ^ 1u, s_abort, p.err,
                                   ROLE_MMA, 13)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t stage = sTok + b.idx * kW2TokStageBytes;
                    const uint32_t a_tmem = tmem_base + kW2TmemA0 + sl.idx * 64u;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t bdesc = smem_desc_sw128(stage + (kk >> 2) * kW2AtomBytes) +
                                               static_cast<uint64_t>((kk & 3) * 2);
                        mma_f16_tmemA(tmem_base + d.idx * kW2Tokens, a_tmem + kk * 8, bdesc, idesc,
                                      kk > 0 ? 1u : 0u);
                    }
                    mma_commit(bar(W2Bar::d_full + d.idx));
                    mma_commit(bar(W2Bar::a_free + sl.idx));
                    mma_commit(bar(W2Bar::b_empty + b.idx));
                    sl.advance(kW2ASlots);
                    b.advance(kW2TokStages);
                    d.advance(kW2Bufs);
                }
            }
            mma_commit(bar(W2Bar::drain));
            drain_wait(bar(W2Bar::drain), 0);
        } else if (warp == 2 && lane == 0) {
            // -------------------------------------------- token TMA producer
            griddep_wait();   // the fp16 token codes come from the kernel launched before
            Ring b;
            uint32_t issued = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += grid) {
                const TileInfo ti = tile_of(t);
                for (int g = 0; g < G; ++g) {
                    if (!mbar_wait(bar(W2Bar::b_empty + b.idx), b.phase ^ 1u, s_abort, p.err,
                                   ROLE_PRODUCER, 12)) {
                        ok = false;
                        break;
                    }
                    const uint32_t stage = sTok + b.idx * kW2TokStageBytes;
                    mbar_arrive_expect_tx(bar(W2Bar::b_full + b.idx), kW2TokStageBytes);
                    for (int a = 0; a < 2; ++a)
                        tma_load_2d(stage + a * kW2AtomBytes, &tmap_x, g * kGroupK + a * 64, ti.m0,
                                    bar(W2Bar::b_full + b.idx));
                    b.advance(kW2TokStages);
                    ++issued;
                }
            }
            if (!ok) drain_ring(bar(W2Bar::b_full), issued, kW2TokStages);
        }
    } else if (wg == 1) {
        // --------------------------------------- weight converter (A -> TMEM)
        setmaxnreg_dec<kOtherRegs>();
        const int row = threadIdx.x - 128;
        const int q = warp & 3;
        Ring a, sl;
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += grid) {
            for (int g = 0; g < G; ++g) {
                if (!mbar_wait(bar(W2Bar::a_full + a.idx), a.phase, s_abort, p.err, ROLE_CONVERT,
                               11) ||
                    !mbar_wait(bar(W2Bar::a_free + sl.idx), sl.phase ^ 1u, s_abort, p.err,
                               ROLE_CONVERT, 12)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint8_t *rowp = smem + kW2OffStages + kW2TokStages * kW2TokStageBytes +
                                      a.idx * kAStageBytes + row * 128;
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                       kW2TmemA0 + sl.idx * 64u;
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    uint32_t r16[16];
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        const int c = 2 * jj + cc;
                        const uint4 v = *reinterpret_cast<const uint4 *>(rowp + ((c ^ (row & 7)) << 4));
                        i8x4_to_op<kA16>(v.x, r16[cc * 8 + 0], r16[cc * 8 + 1]);
                        i8x4_to_op<kA16>(v.y, r16[cc * 8 + 2], r16[cc * 8 + 3]);
                        i8x4_to_op<kA16>(v.z, r16[cc * 8 + 4], r16[cc * 8 + 5]);
                        i8x4_to_op<kA16>(v.w, r16[cc * 8 + 6], r16[cc * 8 + 7]);
                    }
                    tmem_st_16cols(taddr + jj * 16, r16);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(W2Bar::a_empty + a.idx));
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(W2Bar::a_ready + sl.idx));
                a.advance(kW2WStages);
                sl.advance(kW2ASlots);
            }
        }
    } else {
        // -------------------------------------------------------- epilogue
        setmaxnreg_inc<kEpiRegs>();
        griddep_wait();   // the token scales come from the kernel launched before
        const int h = wg - 2;   // token columns [kW2Half h, kW2Half (h + 1))
        const int q = warp & 3;
        const int lrow = q * 32 + lane;
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        float *s_sa = reinterpret_cast<float *>(smem + (h == 0 ? kW2OffSa0 : kW2OffSa1));
        float acc[kW2Half];
#pragma unroll
        for (int j = 0; j < kW2Half; ++j) acc[j] = 0.0f;
        Ring d;   // partial buffer
        bool failed = false;
        for (int t = blockIdx.x; t < total && !failed; t += grid) {
            const TileInfo ti = tile_of(t);
            const int n_local = ti.n0 + lrow;
            const bool n_ok = n_local < p.N;
            const float *swp =
                p.sw + (static_cast<size_t>(ti.e) * p.sw_rows + ((n_ok ? n_local : 0) >> p.sw_shift)) * G;
            // this row's weight scales two groups ahead (loads issued in place)
            float sc0 = n_ok ? ldg_nc_f32_now(swp) : 0.0f;
            float sc1 = (n_ok && G > 1) ? ldg_nc_f32_now(swp + 1) : 0.0f;
            const int col0 = kW2Half * h;
            // The tile's token scales, copied into shared memory now (one per
            // thread, asynchronously) and read at the store: the copies land
            // while the tile's groups run. The barrier first lets every
            // thread of the warpgroup finish reading the previous tile's.
            named_barrier_sync(1 + h, 128);
            if (lrow < kW2Half) {
                const int col = col0 + lrow;
                if (p.sa != nullptr)
                    cp_async_4(smem_u32(s_sa + lrow), p.sa + ti.m0 + min(col, ti.rows - 1),
                               col < ti.rows ? 4u : 0u);
                else
                    s_sa[lrow] = 1.0f;
            }
            for (int g = 0; g < G; ++g) {
                const float sc = sc0;
                sc0 = sc1;
                sc1 = (n_ok && g + 2 < G) ? ldg_nc_f32_now(swp + g + 2) : 0.0f;
                const bool ok = mbar_wait(bar(W2Bar::d_full + d.idx), d.phase, s_abort, p.err,
                                          ROLE_EPILOGUE, 11);
                if (__any_sync(0xFFFFFFFFu, !ok)) {   // the warp fails as one
                    failed = true;
                    break;
                }
                tc_fence_after();
                const uint32_t dcol = d.idx * kW2Tokens;
#pragma unroll
                for (int c = 0; c < kW2Half / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld_32cols_sync(lane_base + dcol + col0 + 32u * c, v);
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        acc[32 * c + j] = fmaf(__uint_as_float(v[j]), sc, acc[32 * c + j]);
                    if (kDebug && n_ok) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const int col = col0 + 32 * c + j;
                            if (col < ti.rows)
                                p.dbg[(static_cast<size_t>(ti.m0 + col) * p.N + n_local) * G + g] =
                                    __float2int_rn(__uint_as_float(v[j]));
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_relaxed(bar(W2Bar::d_empty + d.idx));
                d.advance(kW2Bufs);
            }
            // The warpgroup's copies have landed once all its threads pass the
            // barrier, which also makes a failure of any of its warps theirs.
            cp_async_wait_all();
            if (named_barrier_or(1 + h, 128, failed)) break;
            if (n_ok) {
                // Token rows [m0 + col0, m0 + col0 + kW2Half) of output column
                // n_local through one running pointer.
                const int rows_here = ti.rows - col0;
                const size_t first = static_cast<size_t>(ti.m0 + col0) * p.N + n_local;
                if (p.out_fp32) {
                    float *yp = static_cast<float *>(p.y) + first;
#pragma unroll
                    for (int j = 0; j < kW2Half; ++j) {
                        if (j < rows_here) *yp = acc[j] * s_sa[j];
                        yp += p.N;
                    }
                } else {
                    __nv_bfloat16 *yp = static_cast<__nv_bfloat16 *>(p.y) + first;
#pragma unroll
                    for (int j = 0; j < kW2Half; ++j) {
                        if (j < rows_here) *yp = __float2bfloat16_rn(acc[j] * s_sa[j]);
                        yp += p.N;
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < kW2Half; ++j) acc[j] = 0.0f;
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// =============================================================================
// Decode-sized dense problems (at most 4 token rows): a batched GEMV on the
// CUDA cores. With at most 4 multiply-adds per weight byte, the exact int8
// group sums fit the integer dot-product units (dp4a: four int8 products
// summed into an int32, exact) in less time than the weights take to stream
// from HBM, so the tensor cores' fixed cost per instruction is not paid, and
// the kernel runs at the weight-stream rate (whole tiles, no K split). The
// weight stream (TMA, 128-byte swizzle, two K groups per step), tile table
// and FP32 accumulation order are those of the narrow kernel; the int8 token
// codes are read directly (no fp16 staging copy), in the same stages as the
// weights. (5..8 token rows run faster on the split tensor-core kernel.)
// Warp 0 (lane 0) streams the stages; the other warps compute. In a step,
// a thread forms the exact partials P[m] of its rows, token rows and group;
// the two threads holding the step's two groups of the same rows swap them
// and both apply the group scales in K order, acc = fma(P_g0, sw_g0, acc),
// acc = fma(P_g1, sw_g1, acc).
// =============================================================================
constexpr int gemv_threads(int cw) { return 32 * (1 + cw); }   // producer warp + cw
constexpr int kGemvOffStages = 2048;     // barriers, flags; the tile table follows the stages
constexpr int gemv_stage_bytes(int mr) {
    return 2 * kAStageBytes + ((2 * mr * 128 + 1023) / 1024) * 1024;
}

struct GBar {
    static constexpr int full = 0;                      // [kMaxAStages] TMA -> compute warps
    static constexpr int empty = full + kMaxAStages;    // [kMaxAStages] compute warps (8) -> TMA
    static constexpr int count = empty + kMaxAStages;
};
static_assert(GBar::count <= 128, "barrier area");
static_assert(gemv_stage_bytes(kGemvMaxTokens) % 1024 == 0, "stage alignment");

// GEMV work of this CTA, f(tile, half): the tiles that fill whole waves go
// round-robin (half 0); when at most half a wave is left over, each left-over
// tile is cut into two 64-row halves (half 1: weight rows [0, 64), 2: [64,
// 128)), one per CTA, taken first, so that every SM streams the same number of
// weight bytes (a partial last wave of whole tiles streams on fewer SMs). One
// counted loop with one call site, as for_each_piece.
template <class F>
__device__ __forceinline__ void gemv_for_each(int total, F &&f) {
    const int grid = static_cast<int>(gridDim.x);
    const int c = static_cast<int>(blockIdx.x);
    int dp = (total / grid) * grid;
    const int L = total - dp;
    int nh = 0;
    if (L > 0 && 2 * L <= grid)
        nh = c < 2 * L ? 1 : 0;
    else
        dp = total;
    for (int i = 0;; ++i) {
        int t, h;
        if (i < nh) {
            t = dp + c / 2;
            h = 1 + (c & 1);
        } else {
            t = c + (i - nh) * grid;
            if (t >= dp) return;
            h = 0;
        }
        if (!f(t, h)) return;
    }
}

// Stage producer of the GEMV kernels (one thread): weights and the token
// codes of each step into one stage, per the work split above (half tiles
// load 64 weight rows through tmap_w64).
template <int MR, bool kFuseQ>
__device__ __forceinline__ void gemv_produce(const KParams &p, int total, const CUtensorMap &tmap_w,
                                             const CUtensorMap &tmap_w64,
                                             const CUtensorMap &tmap_q,
                                             uint32_t sA, uint32_t kStage, uint32_t SA,
                                             uint32_t full0, uint32_t empty0, volatile int *s_abort,
                                             const int *s_base, const int *s_lo, const int *s_cnt,
                                             int tt) {
    const int G = p.G;
    // ---------------------------------------------- stage producer
    // The kernel may start while the quantizer that writes the token
    // codes still runs (programmatic dependent launch): the first
    // stage's weight loads go out at once, its token loads (and all
    // later stages) after griddepcontrol.wait. (Deferring more stages
    // delays the first token loads more than it gains: measured.)
    Ring a;
    uint32_t issued = 0;
    bool ok = true;
    bool dep_done = false;
    auto issue_tokens = [&](uint32_t stage, int x, int y, int ng, uint32_t fb) {
        for (int j = 0; j < ng; ++j)
            tma_load_2d(stage + 2 * kAStageBytes + j * MR * 128, &tmap_q, x + j * kGroupK,
                        y, fb);
    };
    gemv_for_each(total, [&](int t, int h) -> bool {
        const TileInfo ti = decode_tile(t, s_base, s_lo, s_cnt, p.E, tt, p.n_tiles, p.gw);
        const int wrow = ti.e * p.N + ti.n0 + (h > 0 ? 64 * (h - 1) : 0);
        const uint32_t wbytes = h > 0 ? kAStageBytes / 2 : kAStageBytes;
        const CUtensorMap *tw = h > 0 ? &tmap_w64 : &tmap_w;
        for (int g0 = 0; g0 < G; g0 += 2) {
            const int ng = min(2, G - g0);
            if (!mbar_wait(empty0 + 8u * a.idx, a.phase ^ 1u, s_abort, p.err,
                           ROLE_PRODUCER, 1)) {
                ok = false;
                return false;
            }
            const uint32_t stage = sA + a.idx * kStage;
            const uint32_t fb = full0 + 8u * a.idx;
            mbar_arrive_expect_tx(fb, static_cast<uint32_t>(ng * (wbytes + (kFuseQ ? 0 : MR * 128))));
            for (int j = 0; j < ng; ++j)
                tma_load_2d(stage + j * kAStageBytes, tw, (g0 + j) * kGroupK, wrow, fb);
            if constexpr (kFuseQ) {   // the compute warps quantize the token rows themselves
                a.advance(SA);
                ++issued;
                continue;
            }
            if (!dep_done) {
                griddep_wait();
                dep_done = true;
            }
            issue_tokens(stage, g0 * kGroupK, ti.m0, ng, fb);
            a.advance(SA);
            ++issued;
        }
        return true;
    });
    if (!kFuseQ && !dep_done) griddep_wait();   // no step at all (or an abort before the first)
    if (!ok) drain_ring(full0, issued, SA);
}

// Register blocking: a compute thread covers RR weight rows x RM token rows
// of one group, so a step's loads from shared memory are amortised over
// RR * RM dot products per word. CW compute warps cover the tile's 128 rows
// x 2 groups in CW * RR / 8 token blocks, so MR = CW * RR / 8 * RM token rows.
// kFuseQ: the kernel quantizes its token rows itself (per-token scale and
// codes exactly as the quantizer kernel computes them) from the BF16
// activations into a resident shared-memory code buffer, so a fused
// quantizer + GEMM call of <= 4 token rows is one kernel; the stages then
// carry weights only.
template <bool kDebug, int RR, int RM, int CW, bool kFuseQ = false>
__global__ void __launch_bounds__(gemv_threads(CW), 1)
w8a8_gemv_kernel(const __grid_constant__ CUtensorMap tmap_w,
                 const __grid_constant__ CUtensorMap tmap_w64,
                 const __grid_constant__ CUtensorMap tmap_q, const KParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw_addr);
    constexpr int TB = CW * RR / 8;
    constexpr int MR = TB * RM;
    static_assert(TB >= 1 && CW * RR % 8 == 0, "compute warps cover whole token blocks");
    constexpr uint32_t kStage =
        kFuseQ ? 2u * kAStageBytes : static_cast<uint32_t>(gemv_stage_bytes(MR));
    static_assert(!kFuseQ || (TB == 1 && !kDebug), "fused quantization: one token block");
    const uint32_t SA = static_cast<uint32_t>(p.a_stages);
    const uint32_t sA = base + kGemvOffStages;
    const uint32_t sBar = base + kOffBar;
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);
    volatile int *s_total = reinterpret_cast<volatile int *>(smem + kOffMisc + 8);
    int *s_base = reinterpret_cast<int *>(smem + p.tab_off);
    int *s_lo = s_base + (p.E + 1);
    int *s_cnt = s_lo + (p.E + 1);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tt = p.tile_tokens;
    auto bar = [&](int i) -> uint32_t { return sBar + 8u * static_cast<uint32_t>(i); };

    if (threadIdx.x == 0) {
        for (int i = 0; i < kMaxAStages; ++i) {
            mbar_init(bar(GBar::full + i), 1);
            mbar_init(bar(GBar::empty + i), CW);
        }
        *s_abort = 0;
        fence_mbarrier_init();
    }
    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&tmap_w);
            tma_prefetch_desc(&tmap_w64);
            tma_prefetch_desc(&tmap_q);
        }
        build_tile_table(p, tt, lane, s_base, s_lo, s_cnt, s_total);
    }
    __syncthreads();
    const int total = *s_total;
    const int G = p.G;

    if (warp == 0) {
        if (lane == 0) {
            gemv_produce<MR, kFuseQ>(p, total, tmap_w, tmap_w64, tmap_q, sA, kStage, SA,
                                     bar(GBar::full), bar(GBar::empty), s_abort, s_base, s_lo,
                                     s_cnt, tt);
        }
    } else {
        // ------------------------------------------------- compute warps
        // Thread (row block rb, token block tb, group j): rows rb + i*128/RR,
        // token rows tb*RM + u. The 8 lanes of a shared-memory phase read 8
        // consecutive rows (conflict-free under the 128-byte swizzle); all
        // lanes of a half-warp read the same token words (broadcast).
        const int ct = threadIdx.x - 32;
        const int cw = ct >> 5;
        constexpr int kWarpsPerTb = 8 / RR;
        const int tb = cw / kWarpsPerTb;
        const int rb = (cw % kWarpsPerTb) * 16 + (lane & 15);
        const int j = lane >> 4;                      // group of the step
        const bool vec_sw = (G % 4 == 0) && ((reinterpret_cast<uintptr_t>(p.sw) & 15u) == 0);
        float s_tok[MR];   // kFuseQ: the token rows' scales
        const uint8_t *qbuf = smem + p.qbuf_off;
        if constexpr (kFuseQ) {
            // The activations may come from the kernel launched before this
            // one (programmatic dependent launch): wait for it, then form each
            // row's scale (block max of |x|) and its codes, group by group in
            // the layout the stages use ([group][token row][128 codes]).
            griddep_wait();
            uint32_t *red = reinterpret_cast<uint32_t *>(smem + 512);   // [MR][CW], spare barrier area
            const int nvec = p.K >> 3;
            constexpr int kCT = 32 * CW;
#pragma unroll
            for (int u = 0; u < MR; ++u) {
                uint32_t m = 0;
                if (u < p.R) {
                    const uint4 *src = reinterpret_cast<const uint4 *>(p.act + u * p.lda);
                    for (int v = ct; v < nvec; v += kCT) m = max(m, amax_bits8(__ldg(src + v)));
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
                if (lane == 0) red[u * CW + cw] = m;
            }
            named_barrier_sync(1, kCT);
            float r_tok[MR];
            bool fast[MR];
#pragma unroll
            for (int u = 0; u < MR; ++u) {
                uint32_t m = 0;
                for (int w = 0; w < CW; ++w) m = max(m, red[u * CW + w]);
                s_tok[u] = __fdiv_rn(bf16_bits_to_f32(m), 127.0f);
                fast[u] = s_tok[u] >= 1.17549435e-38f;   // normal scale: 1/s is finite
                r_tok[u] = fast[u] ? __frcp_rn(s_tok[u]) : 0.0f;
            }
#pragma unroll
            for (int u = 0; u < MR; ++u) {
                if (u >= p.R) continue;
                const uint4 *src = reinterpret_cast<const uint4 *>(p.act + u * p.lda);
                for (int v = ct; v < nvec; v += kCT) {
                    const int k = v << 3;
                    *reinterpret_cast<uint2 *>(const_cast<uint8_t *>(qbuf) +
                                               ((k >> 7) * MR + u) * 128 + (k & 127)) =
                        quantize8(__ldg(src + v), s_tok[u], r_tok[u], fast[u]);
                }
            }
            named_barrier_sync(1, kCT);   // codes complete before the first step reads them
        }
        // After a failed wait the warp stops waiting and doing data work.
        bool failed = false;
        Ring a;
        float acc[RR][RM];
        gemv_for_each(total, [&](int t, int h) -> bool {
            const TileInfo ti = decode_tile(t, s_base, s_lo, s_cnt, p.E, tt, p.n_tiles, p.gw);
            // a half tile's 64 rows sit in stage rows [0, 64)
            const int n0 = ti.n0 + (h > 0 ? 64 * (h - 1) : 0);
            const int s0 = 0, s1 = (G + 1) >> 1;
            int n_row[RR];
            bool n_ok[RR];
            const float *swp[RR];
#pragma unroll
            for (int i = 0; i < RR; ++i) {
                const int lr = rb + i * (128 / RR);
                n_row[i] = n0 + lr;
                n_ok[i] = n_row[i] < p.N && (h == 0 || lr < 64);
                swp[i] = p.sw + (static_cast<size_t>(ti.e) * p.sw_rows +
                                 ((n_ok[i] ? n_row[i] : 0) >> p.sw_shift)) * G;
#pragma unroll
                for (int u = 0; u < RM; ++u) acc[i][u] = 0.0f;
            }
            auto load_quad = [&](int i, int g) -> float4 {
                float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                if (!n_ok[i] || failed) return v;
                if (vec_sw) {
                    if (g < G) v = ldg_nc_f32x4_now(swp[i] + g);
                } else {
                    if (g < G) v.x = ldg_nc_f32_now(swp[i] + g);
                    if (g + 1 < G) v.y = ldg_nc_f32_now(swp[i] + g + 1);
                    if (g + 2 < G) v.z = ldg_nc_f32_now(swp[i] + g + 2);
                    if (g + 3 < G) v.w = ldg_nc_f32_now(swp[i] + g + 3);
                }
                return v;
            };
            const int qb = (2 * s0) & ~3;
            float4 cur[RR], nxt[RR];
#pragma unroll
            for (int i = 0; i < RR; ++i) {
                cur[i] = load_quad(i, qb);
                nxt[i] = load_quad(i, qb + 4);
            }
            for (int sg = s0; sg < s1; ++sg) {
                const int g0 = 2 * sg;
                const int ng = min(2, G - g0);
                if ((g0 & 3) == 0 && g0 > qb) {
#pragma unroll
                    for (int i = 0; i < RR; ++i) {
                        cur[i] = nxt[i];
                        nxt[i] = load_quad(i, g0 + 4);
                    }
                }
                if (!failed) {
                    const bool waited = *s_abort == 0 &&
                                        mbar_wait_spin(bar(GBar::full + a.idx), a.phase, s_abort,
                                                       p.err, ROLE_CONVERT, 1);
                    failed = __any_sync(0xFFFFFFFFu, !waited);
                }
                if (failed) continue;
                int P[RR][RM];
#pragma unroll
                for (int i = 0; i < RR; ++i)
#pragma unroll
                    for (int u = 0; u < RM; ++u) P[i][u] = 0;
                if (j < ng) {
                    const uint8_t *stage = smem + kGemvOffStages + a.idx * kStage;
                    const uint8_t *wg = stage + j * kAStageBytes;
                    const uint8_t *tok =
                        kFuseQ ? qbuf + ((g0 + j) * MR + tb * RM) * 128
                               : stage + 2 * kAStageBytes + (j * MR + tb * RM) * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        uint4 wv[RR], tv[RM];
#pragma unroll
                        for (int i = 0; i < RR; ++i) {
                            const int r = rb + i * (128 / RR);
                            wv[i] = *reinterpret_cast<const uint4 *>(wg + r * 128 + ((c ^ (r & 7)) << 4));
                        }
#pragma unroll
                        for (int u = 0; u < RM; ++u)
                            tv[u] = *reinterpret_cast<const uint4 *>(tok + u * 128 + c * 16);
#pragma unroll
                        for (int i = 0; i < RR; ++i)
#pragma unroll
                            for (int u = 0; u < RM; ++u) {
                                P[i][u] = __dp4a(static_cast<int>(wv[i].x), static_cast<int>(tv[u].x), P[i][u]);
                                P[i][u] = __dp4a(static_cast<int>(wv[i].y), static_cast<int>(tv[u].y), P[i][u]);
                                P[i][u] = __dp4a(static_cast<int>(wv[i].z), static_cast<int>(tv[u].z), P[i][u]);
                                P[i][u] = __dp4a(static_cast<int>(wv[i].w), static_cast<int>(tv[u].w), P[i][u]);
                            }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(GBar::empty + a.idx));
                a.advance(SA);
#pragma unroll
                for (int i = 0; i < RR; ++i) {
                    const float sc0 = (g0 & 3) == 0 ? cur[i].x : cur[i].z;
                    const float sc1 = (g0 & 3) == 0 ? cur[i].y : cur[i].w;
#pragma unroll
                    for (int u = 0; u < RM; ++u) {
                        const int other = __shfl_xor_sync(0xFFFFFFFFu, P[i][u], 16);
                        const int p0 = j ? other : P[i][u];
                        const int p1 = j ? P[i][u] : other;
                        acc[i][u] = fmaf(static_cast<float>(p0), sc0, acc[i][u]);
                        if (ng == 2) acc[i][u] = fmaf(static_cast<float>(p1), sc1, acc[i][u]);
                    }
                }
                if (kDebug && j < ng) {
#pragma unroll
                    for (int i = 0; i < RR; ++i)
#pragma unroll
                        for (int u = 0; u < RM; ++u) {
                            const int m = tb * RM + u;
                            if (n_ok[i] && m < ti.rows)
                                p.dbg[(static_cast<size_t>(ti.m0 + m) * p.N + n_row[i]) * G + g0 + j] =
                                    P[i][u];
                        }
                }
            }
            auto store_out = [&](int i, int u, float v) {
                const int m = tb * RM + u;
                const float out = v * (kFuseQ ? s_tok[u] : load_sa(p, ti.m0 + m));
                const size_t idx = static_cast<size_t>(ti.m0 + m) * p.N + n_row[i];
                if (p.out_fp32)
                    static_cast<float *>(p.y)[idx] = out;
                else
                    static_cast<__nv_bfloat16 *>(p.y)[idx] = __float2bfloat16_rn(out);
            };
            if (j == 0 && !failed) {
#pragma unroll
                for (int i = 0; i < RR; ++i)
#pragma unroll
                    for (int u = 0; u < RM; ++u)
                        if (n_ok[i] && tb * RM + u < ti.rows) store_out(i, u, acc[i][u]);
            }
            return true;
        });
    }
}

// Diagnostic of the bounded-wait error path: one thread arms an mbarrier for
// 16 bytes that no copy will ever deliver (a mis-sized expect-tx) and waits on
// it through the same bounded wait the GEMM roles use, with a short limit.
// The wait gives up, writes its code into the error word and the kernel
// returns; nothing traps or hangs, and no copy is left in flight.
__global__ void selftest_wait_kernel(unsigned long long *err, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ volatile int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbarrier_init();
        mbar_arrive_expect_tx(smem_u32(&bar), 16);
        mbar_wait(smem_u32(&bar), 0, &abort_flag, err, ROLE_SELFTEST, 1, limit_ns, KID_SELFTEST);
    }
}

// ------------------------------------------------------------------- host
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

bool encode_2d(CUtensorMap *map, CUtensorMapDataType dtype, size_t elem_bytes, const void *ptr,
               uint64_t inner, uint64_t outer, uint32_t box_inner, uint32_t box_outer) {
    auto fn = get_encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * elem_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, dtype, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The token operand: fp16 codes [R, K] (dense rows) or, for the weight-only
// path, the caller's BF16 activations [R, ldx] (rows ldx elements apart).
bool encode_tokens(CUtensorMap *map, const GemmProblem &pr, uint32_t box_rows) {
    auto fn = get_encode_fn();
    if (fn == nullptr) return false;
    const uint64_t pitch = static_cast<uint64_t>(pr.ldx > 0 ? pr.ldx : pr.K);
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(pr.K), static_cast<cuuint64_t>(pr.R)};
    cuuint64_t strides[1] = {pitch * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, pr.a16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                          2, const_cast<void *>(pr.x16), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Same without swizzle (row-major box in shared memory).
bool encode_2d_plain(CUtensorMap *map, CUtensorMapDataType dtype, size_t elem_bytes,
                     const void *ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
                     uint32_t box_outer) {
    auto fn = get_encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * elem_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, dtype, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Pipeline shape of one call: batch width, tile rows, partial buffers and
// stage counts, filling shared memory with weight stages after the token stages.
struct PipeShape {
    int b_rows, tile_tokens, b_stages, a_stages, smem_bytes;
    bool narrow;    // tiles of <= 64 token rows: w8a8_gemm_narrow_kernel
    bool wide;      // tiles of 96 or 128 token rows: its kWide form
};

PipeShape choose_pipe(const GemmProblem &pr) {
    PipeShape s;
    if (pr.offsets == nullptr) {
        // Dense: one tile of the rounded-up token count up to 128 rows,
        // 128-row tiles beyond.
        s.b_rows = pr.R <= kMaxBatchRows
                       ? static_cast<int>((pr.R + kBoxRows - 1) / kBoxRows * kBoxRows)
                       : kMaxBatchRows;
    } else {
        // Expert tiles of 128 rows when the tile table fits the wide form's
        // fixed area (fewer tiles, and fewer weight passes, for experts with
        // 65..128 routed rows), else 64.
        s.b_rows = pr.E <= kWideMaxExperts ? kMaxBatchRows : 64;
    }
    s.tile_tokens = s.b_rows;
    s.narrow = s.b_rows <= 64;
    s.wide = !s.narrow;
    // Token stages (b_rows x 512 B each): the two step slots for wide tiles; a
    // deeper ring for narrow ones, so that token tiles are requested several
    // steps ahead (their L2 latency, ~1 us under the weight stream, was on the
    // critical path with two), at the cost of one weight stage.
    s.b_stages = s.wide ? kNarrowSlots : (s.b_rows <= 32 ? 4 : 3);
    const int b_slot_bytes = 4 * s.b_rows * 128;
    // Weight stages after the fixed area: 14 KB (tile table for up to 1024
    // experts) for narrow tiles, 2 KB for wide ones.
    const int off = s.wide ? kWideOffStages : kOffStages;
    const int avail = kSmemLimit - 1024 - off - s.b_stages * b_slot_bytes;
    s.a_stages = avail / kNarrowAStageBytes;
    if (s.a_stages > kMaxAStages) s.a_stages = kMaxAStages;
    s.smem_bytes = off + s.a_stages * kNarrowAStageBytes + s.b_stages * b_slot_bytes + 1024;
    return s;
}

template <auto kernel>
cudaError_t launch_kernel(const GemmProblem &pr, const PipeShape &ps, int num_sms,
                          cudaStream_t stream) {
    if (ps.a_stages < 2 || ps.b_stages > kMaxBStages || ps.b_rows % kBoxRows != 0 ||
        ps.b_rows > kMaxBatchRows ||
        ps.smem_bytes > kSmemLimit)
        return cudaErrorInvalidConfiguration;
    CUtensorMap tw, tx;
    if (!encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, pr.qw, (uint64_t)pr.K,
                   (uint64_t)(pr.E * pr.N), kGroupK, kTileN) ||
        !encode_tokens(&tx, pr, kBoxRows))
        return cudaErrorInvalidValue;

    static int attr_done[64] = {0};   // per device, per kernel instance
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        // setmaxnreg.inc can only take registers the CTA was launched with:
        // refuse to launch unless the launch allocation covers the split.
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
        if (e != cudaSuccess) return e;
        if (fa.numRegs * kThreads < (kThreads / 2) * (kEpiRegs + kOtherRegs))
            return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
        if (e != cudaSuccess) return e;
        attr_done[dev] = 1;
    }

    KParams kp;
    kp.sa = pr.sa;
    kp.sw = pr.sw;
    kp.sw_shift = pr.sw_block_rows == 128 ? 7 : 0;
    kp.sw_rows = static_cast<int>((pr.N + (1 << kp.sw_shift) - 1) >> kp.sw_shift);
    kp.offsets = pr.offsets;
    kp.y = pr.y;
    kp.dbg = pr.debug_partials;
    kp.R = static_cast<int>(pr.R);
    kp.E = static_cast<int>(pr.E);
    kp.N = static_cast<int>(pr.N);
    kp.K = static_cast<int>(pr.K);
    kp.G = static_cast<int>(pr.K / kGroupK);
    kp.n_tiles = static_cast<int>((pr.N + kTileN - 1) / kTileN);
    kp.out_fp32 = pr.out_fp32 ? 1 : 0;
    kp.a_stages = ps.a_stages;
    kp.b_stages = ps.b_stages;
    kp.b_rows = ps.b_rows;
    kp.tile_tokens = ps.tile_tokens;
    kp.tab_off = kOffTab;
    kp.group_tokens = (ps.wide && pr.offsets == nullptr) ? 1 : 0;
    kp.gw = (ps.wide && pr.offsets == nullptr) ? kRasterBand : 0;
    unsigned long long *err = nullptr;
    cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void **>(&err), g_device_error);
    if (e != cudaSuccess) return e;
    kp.err = err;

    // Upper bound on the number of tiles (exact for one dense segment).
    const int64_t tt = ps.tile_tokens;
    const int64_t m_tiles_bound = pr.offsets == nullptr ? (pr.R + tt - 1) / tt
                                                        : (pr.R + tt - 1) / tt + pr.E;
    const int64_t tiles_bound = m_tiles_bound * kp.n_tiles;
    // Dense narrow tiles split their K ranges across CTAs (stream-K) when the
    // workspace holds the split area: one CTA per SM, or per step if fewer.
    const bool split = !ps.wide && pr.offsets == nullptr && pr.sk_cnt != nullptr &&
                       num_sms <= kSkMaxCtas && pr.sk_ld >= pr.R;
    const int64_t units = split ? tiles_bound * ((kp.G + 1) / 2) : tiles_bound;
    const int64_t grid = units < num_sms ? units : num_sms;
    if (grid <= 0) return cudaSuccess;
    kp.sk_cnt = split ? pr.sk_cnt : nullptr;
    kp.sk_part = split ? pr.sk_part : nullptr;
    kp.sk_ld = split ? pr.sk_ld : 0;

    // Programmatic dependent launch: the kernel may start while the staging
    // kernel before it in the stream is still running; its token producer and
    // its epilogue wait for that kernel (griddepcontrol.wait).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(ps.smem_bytes);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, tw, tx, kp);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Dense calls of at least kW2Tokens token rows: w8a8_gemm_wide_kernel.
template <auto kernel>
cudaError_t launch_wide(const GemmProblem &pr, int num_sms, cudaStream_t stream) {
    CUtensorMap tw, tx;
    if (!encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, pr.qw, (uint64_t)pr.K,
                   (uint64_t)(pr.E * pr.N), kGroupK, kTileN) ||
        !encode_tokens(&tx, pr, kW2Tokens))
        return cudaErrorInvalidValue;
    static int attr_done[64] = {0};   // per device, per kernel instance
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        // setmaxnreg.inc can only take registers the CTA was launched with.
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
        if (e != cudaSuccess) return e;
        if (fa.numRegs * kThreads < (kThreads / 2) * (kEpiRegs + kOtherRegs))
            return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kW2SmemBytes);
        if (e != cudaSuccess) return e;
        attr_done[dev] = 1;
    }
    KParams kp = {};
    kp.sa = pr.sa;
    kp.sw = pr.sw;
    kp.sw_shift = pr.sw_block_rows == 128 ? 7 : 0;
    kp.sw_rows = static_cast<int>((pr.N + (1 << kp.sw_shift) - 1) >> kp.sw_shift);
    kp.offsets = nullptr;
    kp.y = pr.y;
    kp.dbg = pr.debug_partials;
    kp.R = static_cast<int>(pr.R);
    kp.E = 1;
    kp.N = static_cast<int>(pr.N);
    kp.K = static_cast<int>(pr.K);
    kp.G = static_cast<int>(pr.K / kGroupK);
    kp.n_tiles = static_cast<int>((pr.N + kTileN - 1) / kTileN);
    kp.out_fp32 = pr.out_fp32 ? 1 : 0;
    kp.tile_tokens = kW2Tokens;
    kp.gw = kRasterBand;
    cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void **>(&kp.err), g_device_error);
    if (e != cudaSuccess) return e;
    const int64_t tiles = (pr.R + kW2Tokens - 1) / kW2Tokens * kp.n_tiles;
    const int64_t grid = tiles < num_sms ? tiles : num_sms;
    if (grid <= 0) return cudaSuccess;
    // Programmatic dependent launch: the token producer and the epilogue wait
    // for the kernel before it (which writes the fp16 codes and the scales).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(kW2SmemBytes);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, tw, tx, kp);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Batched GEMV on the CUDA cores for dense calls of at most 4 token rows.
// kExtra: bytes of shared memory the kernel keeps after its stages.
template <auto kernel, int MR, int CW, int kExtra, bool kFuseQ = false>
cudaError_t launch_gemv(const GemmProblem &pr, int num_sms, cudaStream_t stream) {
    // kFuseQ: weight-only stages plus a resident code buffer of all K groups
    constexpr int stage = kFuseQ ? 2 * kAStageBytes : gemv_stage_bytes(MR);
    const int qbuf_bytes = kFuseQ ? static_cast<int>(pr.K / kGroupK) * MR * 128 : 0;
    const int tab_bytes = static_cast<int>((3 * (pr.E + 1) * 4 + 15) / 16 * 16);
    int stages = (kSmemLimit - 1024 - kGemvOffStages - kExtra - qbuf_bytes - tab_bytes) / stage;
    if (stages > kMaxAStages) stages = kMaxAStages;
    if (stages < 2 || pr.R > MR) return cudaErrorInvalidConfiguration;
    const int qbuf_off = kGemvOffStages + stages * stage + kExtra;
    const int tab_off = qbuf_off + qbuf_bytes;
    const int smem_bytes = tab_off + tab_bytes + 1024;
    CUtensorMap tw, tw64, tq;
    if (!encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, pr.qw, (uint64_t)pr.K,
                   (uint64_t)(pr.E * pr.N), kGroupK, kTileN) ||
        !encode_2d(&tw64, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, pr.qw, (uint64_t)pr.K,
                   (uint64_t)(pr.E * pr.N), kGroupK, kTileN / 2))
        return cudaErrorInvalidValue;
    if (kFuseQ) {
        tq = tw;   // not read: the kernel quantizes the token rows itself
    } else if (!encode_2d_plain(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, pr.qa, (uint64_t)pr.K,
                                (uint64_t)pr.R, kGroupK, MR)) {
        return cudaErrorInvalidValue;
    }
    static int attr_done[64] = {0};   // per device, per kernel instance
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        const cudaError_t e =
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
        if (e != cudaSuccess) return e;
        attr_done[dev] = 1;
    }
    KParams kp = {};
    kp.sa = pr.sa;
    kp.sw = pr.sw;
    kp.sw_shift = pr.sw_block_rows == 128 ? 7 : 0;
    kp.sw_rows = static_cast<int>((pr.N + (1 << kp.sw_shift) - 1) >> kp.sw_shift);
    kp.offsets = nullptr;
    kp.y = pr.y;
    kp.dbg = pr.debug_partials;
    kp.R = static_cast<int>(pr.R);
    kp.E = static_cast<int>(pr.E);
    kp.N = static_cast<int>(pr.N);
    kp.K = static_cast<int>(pr.K);
    kp.G = static_cast<int>(pr.K / kGroupK);
    kp.n_tiles = static_cast<int>((pr.N + kTileN - 1) / kTileN);
    kp.out_fp32 = pr.out_fp32 ? 1 : 0;
    kp.a_stages = stages;
    kp.act = pr.act;
    kp.lda = pr.lda;
    kp.qbuf_off = qbuf_off;
    kp.b_rows = MR;
    kp.tile_tokens = MR;
    kp.tab_off = tab_off;
    unsigned long long *err = nullptr;
    cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void **>(&err), g_device_error);
    if (e != cudaSuccess) return e;
    kp.err = err;
    const int64_t grid = kp.n_tiles < num_sms ? kp.n_tiles : num_sms;
    // Programmatic dependent launch: the kernel may start while the kernel
    // before it in the stream (the quantizer) still runs; its stage producer
    // waits for that kernel before loading the token codes.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(gemv_threads(CW));
    cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, tw, tw64, tq, kp);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int RR, int RM, int CW>
cudaError_t launch_gemv_mr(const GemmProblem &pr, int num_sms, cudaStream_t stream) {
    constexpr int MR = CW * RR / 8 * RM;
    if (pr.act != nullptr)   // fused quantizer (no debug partials on that path)
        return launch_gemv<w8a8_gemv_kernel<false, RR, RM, CW, true>, MR, CW, 0, true>(
            pr, num_sms, stream);
    return pr.debug_partials != nullptr
               ? launch_gemv<w8a8_gemv_kernel<true, RR, RM, CW>, MR, CW, 0>(pr, num_sms, stream)
               : launch_gemv<w8a8_gemv_kernel<false, RR, RM, CW>, MR, CW, 0>(pr, num_sms, stream);
}

}  // namespace

cudaError_t launch_gemm(const GemmProblem &pr, int num_sms, cudaStream_t stream) {
    if (pr.a16) {
        // weight-only path: tensor-core kernels only, no debug partials, no K split
        if (pr.debug_partials != nullptr || pr.sk_cnt != nullptr)
            return cudaErrorInvalidValue;
        if (uses_wide256(pr.R, pr.offsets != nullptr))
            return launch_wide<w8a8_gemm_wide_kernel<false, true>>(pr, num_sms, stream);
        const PipeShape ps = choose_pipe(pr);
        if (ps.wide) {
            if (pr.E > kWideMaxExperts) return cudaErrorInvalidConfiguration;
            return launch_kernel<w8a8_gemm_narrow_kernel<false, true, true>>(pr, ps, num_sms,
                                                                              stream);
        }
        return launch_kernel<w8a8_gemm_narrow_kernel<false, false, true>>(pr, ps, num_sms, stream);
    }
    if (uses_gemv(pr.R, pr.offsets != nullptr)) {
        if (pr.R <= 1) return launch_gemv_mr<1, 1, 8>(pr, num_sms, stream);
        if (pr.R <= 2) return launch_gemv_mr<1, 2, 8>(pr, num_sms, stream);
        return launch_gemv_mr<1, 4, 8>(pr, num_sms, stream);
    }
    const bool dbg = pr.debug_partials != nullptr;
    if (uses_wide256(pr.R, pr.offsets != nullptr))
        return dbg ? launch_wide<w8a8_gemm_wide_kernel<true>>(pr, num_sms, stream)
                   : launch_wide<w8a8_gemm_wide_kernel<false>>(pr, num_sms, stream);
    const PipeShape ps = choose_pipe(pr);
    if (ps.wide) {
        if (pr.E > kWideMaxExperts) return cudaErrorInvalidConfiguration;
        return dbg ? launch_kernel<w8a8_gemm_narrow_kernel<true, true>>(pr, ps, num_sms, stream)
                   : launch_kernel<w8a8_gemm_narrow_kernel<false, true>>(pr, ps, num_sms, stream);
    }
    return dbg ? launch_kernel<w8a8_gemm_narrow_kernel<true, false>>(pr, ps, num_sms, stream)
               : launch_kernel<w8a8_gemm_narrow_kernel<false, false>>(pr, ps, num_sms, stream);
}

cudaError_t launch_selftest_wait(unsigned long long limit_ns, cudaStream_t stream) {
    unsigned long long *err = nullptr;
    cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void **>(&err), g_device_error);
    if (e != cudaSuccess) return e;
    selftest_wait_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
    return cudaGetLastError();
}

cudaError_t device_error_word(unsigned long long **out) {
    return cudaGetSymbolAddress(reinterpret_cast<void **>(out), g_device_error);
}

cudaError_t read_device_error(unsigned long long *value, bool clear) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(value, g_device_error, sizeof(unsigned long long));
    if (e != cudaSuccess) return e;
    if (clear && *value != 0) {
        const unsigned long long zero = 0;
        e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
    }
    return e;
}

}  // namespace w8a8
