// sgemm_kernel.cuh — the warp-specialised strict-FP32 SGEMM kernel for sm_103a.
//
// C = alpha * A * B + beta * C, row-major A (M x K, lda), B (K x N, ldb),
// C (M x N, ldc); every multiply-add is a single-rounding FP32 FMA on the
// CUDA cores (scalar FFMA or the packed two-lane FFMA2).
//
// Structure (persistent CTAs, one per SM for the 128 x 128 tile):
//   * producer warp(s) fill an S-deep ring of shared-memory stages, each a
//     tile of A (BM x BK, or BK x BM) and a BK x BN tile of B. An operand whose base and
//     row stride are 16-byte aligned is moved by TMA (cp.async.bulk.tensor,
//     one elected thread, zero fill past the matrix edges); otherwise by
//     4-byte cp.async with zero fill (src-size 0). Either way the stage's
//     "full" mbarrier completes when every byte has landed.
//   * consumer warps (each a 32 x 64 warp tile, 4 x 8 lanes, 8 x 8 outputs
//     per lane) wait on "full", run the register outer product, and arrive on
//     "empty" so the producer can refill the stage.
//   * the epilogue writes alpha * acc + beta * C straight from registers with
//     float4 stores where C allows it, masked scalar stores elsewhere; C is
//     not read when beta == 0.
//
// Work schedule (hybrid data-parallel + stream-K): the first dp_tiles tiles
// are whole work items handed out round-robin (tile = CTA + wave * grid).
// The k-iterations of the remaining tiles are split into sk_ctas equal
// contiguous ranges, one per CTA, so the last, partial wave costs a fraction
// of a tile instead of a whole one. A split tile is finished by the CTA that
// holds its first k-segment, which is that CTA's last work item: the CTAs
// holding the later segments processed them first (as their first items),
// wrote their raw sums to workspace slots and set a flag each, so by the
// time the finishing CTA gets there the flags are normally set already; it
// waits for them (bounded), adds the slots in k order and runs the
// epilogue. Such a wait is only ever on a CTA with a higher index, and the
// grid never has more CTAs than the GPU holds at once. The older form,
// every partial segment to a slot and a second kernel (sk_fixup_kernel) to
// finish the tiles, with no CTA waiting for another, stays selectable.
//
// The pages this follows ("The road to a fast GEMM": sections "v4:
// two-dimensional register tiling", "v5: vectorized loads", "Where to go
// next" on double buffering, multi-stage pipelines, warp tiling and split-K;
// the Tinyforge README on BK = 16 + padding and XOR swizzling; the T4
// article's "Tiling" section on zero-filled tails) use __syncthreads double
// buffering on sm_75..sm_89. Here the ring is deeper, the barriers are
// mbarriers and the loads are TMA where the strides allow it. A reaches the
// consumers in one of two shared-memory layouts: row-major under the
// 128-byte TMA swizzle (each lane reads float4 runs along k for its 8 rows),
// or k-major, [BK][BM], the layout of the pages' transposing store (each
// lane reads two float4 of 4 rows per k-step; the FMA pipe stays busier).
// The k-major layout comes from an A given transposed, from a transposed
// copy of A (made by a kernel before this one, or by this kernel's own
// transposer warps while its first tiles run, which then also make the
// row-major copy of a transposed B), or from transposer warps that rewrite
// each TMA-landed stage.
//
// Every wait, on an mbarrier or on another CTA's flag, is bounded
// (globaltimer): on timeout the thread sets a bit in the device status word,
// lets its own copies in flight land (again bounded) and returns. Nothing
// spins forever.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "ptx.cuh"

namespace sg {

// LOAD_TMA_XP (A only): TMA brings the row-major A tile into a raw staging
// buffer and three transposer warps rewrite it as [BK][BM] for the
// consumers (see transposer()).
enum LoadMode : int { LOAD_TMA = 0, LOAD_CPASYNC = 1, LOAD_TMA_XP = 2 };

// Status bits written by the kernels when a bounded wait gives up or a
// schedule invariant fails.
enum : int {
    STATUS_CONSUMER_TIMEOUT = 1,
    STATUS_PRODUCER_TIMEOUT = 2,
    STATUS_DRAIN_TIMEOUT = 4,
    STATUS_SCHEDULE = 8,
    STATUS_INDEX = 16,
};

// Device-side invariant checks of the debug build (-DSGEMM_DEBUG): a check
// that fails sets STATUS_INDEX in the status word and execution carries on
// (no trap), so the host sees it in the status check. In the ordinary build
// they compile to nothing.
#ifdef SGEMM_DEBUG
#define SG_DCHECK(p, cond)                                       \
    do {                                                         \
        if (!(cond)) atomicOr((p).status, ::sg::STATUS_INDEX);  \
    } while (0)
#else
#define SG_DCHECK(p, cond) \
    do {                   \
    } while (0)
#endif

struct GemmParams {
    int M, N, K;
    int tiles_m, tiles_n, k_tiles;
    int group_m;        // raster: tiles walk group_m tile-rows at a time
    int c_vec;          // C base 16-byte aligned and ldc % 4 == 0
    const float* A;
    const float* B;
    float* C;
    long long lda, ldb, ldc;
    float alpha, beta;
    unsigned long long timeout_ns;
    int* status;
    // Schedule: tiles [0, dp_tiles) are whole items; the k-iterations of
    // tiles [dp_tiles, tiles) (sk_iters of them) are split over sk_ctas CTAs.
    int dp_tiles;
    int sk_ctas;
    long long sk_iters;
    // How split tiles are finished. sk_fixup == 0: inside this kernel, by the
    // CTA that holds the tile's first k-segment (its last work item); every
    // other segment's CTA leaves its raw sums in slot blockIdx.x of ws and
    // then sets sk_flags[blockIdx.x] = sk_tag (release), and the finishing
    // CTA waits (bounded, acquire) for those flags, adds the slots in k order,
    // resets the flags to 0 and runs the epilogue. sk_fixup == 1: every
    // partial segment goes to a slot (2c for a range's first segment, 2c + 1
    // for its last) and sk_fixup_kernel finishes the tiles.
    float* ws;          // sk_ctas (or 2 sk_ctas) partial-tile slots of BM x BN floats
    unsigned long long* sk_flags;   // sk_ctas flags (sk_fixup == 0)
    unsigned long long sk_tag;      // this launch's flag value, never 0
    int sk_fixup;
    // Transposed A made inside the kernel (Cfg::FUSED): the transposer warps
    // of every CTA write A (row-major at at_src, row stride at_lds) as its
    // transpose into the workspace at A (K rows of lda floats), one unit of
    // BK k-rows x BM columns at a time, and set at_flags[tm * k_tiles + kt]
    // to at_tag (release) when unit (tm, kt) is complete; the TMA producer
    // waits (bounded, acquire) for a unit's flag before it loads the unit.
    const float* at_src;
    long long at_lds;
    unsigned long long* at_flags;
    unsigned long long at_tag;      // this launch's flag value, never 0
    // The same for a transposed B (stored N x K at bt_src, row stride
    // bt_lds): its row-major copy at B (K rows of ldb floats), units of BK
    // k-rows x BN columns, flags bt_flags[tn * k_tiles + kt] = at_tag. Either
    // copy may be absent (source null).
    const float* bt_src;
    long long bt_lds;
    unsigned long long* bt_flags;
};

// Kernel configuration. FORDER: FMA form of the outer product (0: scalar
// FFMA, 2: packed FFMA2 over column pairs, rows outer, 3: the same with the
// column pairs outer).
// EARLY: halfway through a stage, probe (without blocking) whether the next
// stage of the same work item has landed, so the blocking wait at the stage
// boundary is skipped when it has.
// LMAP: lane -> (row group tr, column group tc) of the 4 x 8 lane grid.
//   0: tr = lane / 8, tc = lane % 8. A quarter-warp (8 lanes) reads one A
//      chunk and the same 8 B chunks as every other quarter: a B float4 load
//      costs 4 shared-memory wavefronts, an A load 2.
//   1: tr = lane % 4, tc = lane / 4. A quarter-warp reads 2 B chunks and 4 A
//      chunks: both loads cost 2 wavefronts (measured on sm_103a), a third
//      fewer wavefronts per FMA.
// A_T: A is given transposed (stored K x M, element (i, k) at A[k * lda + i]).
//   The stage then holds A as [BK][BM] (k rows of BM contiguous m, no
//   swizzle), the layout "The road to a fast GEMM" (v5) builds by a
//   transposing store: a lane reads its rows as two float4 per k. TMA only.
// A_MODE == LOAD_TMA_XP: a row-major A reaches the consumers in the same
//   [BK][BM] layout, built in shared memory by transposer warps, with the
//   16-byte chunks of k-row k XOR-swizzled by (k / 4) mod 8 so that both the
//   transposing stores and the consumers' reads are free of bank conflicts.
// CS: CTAs per thread-block cluster. With CS > 1 the CTAs of a cluster share
//   one tile: CTA rank r takes k-tiles [r kt / CS, (r + 1) kt / CS); the
//   ranks then exchange their sums through each other's shared memory
//   (distributed shared memory) so that each adds, in rank order, the sums of
//   8 / CS of every lane's 8 rows (a reduce-scatter) and writes those rows of
//   C. The grid is tiles x CS, one tile per cluster, no
//   stream-K tail.
template <int BM_, int BN_, int BK_, int STAGES_, int A_MODE_, int B_MODE_, int FORDER_ = 2,
          int EARLY_ = 0, int LMAP_ = 0, int A_T_ = 0, int ALOAD_ = 4, int TN_ = 8,
          int KSPLIT_ = 1, int CS_ = 1, int FUSED_ = 0>
struct Cfg {
    static constexpr int BM = BM_, BN = BN_, BK = BK_, STAGES = STAGES_;
    static constexpr int A_MODE = A_MODE_, B_MODE = B_MODE_;
    static constexpr int FORDER = FORDER_, EARLY = EARLY_, LMAP = LMAP_, A_T = A_T_;
    // ALOAD (row-major A only): k-values per shared load of a lane's row,
    // 4 (float4 runs read once per 4 k-steps), 2 (float2 per 2 k-steps) or
    // 1 (one float per row and k-step: fewest live registers).
    static constexpr int ALOAD = ALOAD_;
    static_assert(ALOAD == 1 || ALOAD == 2 || ALOAD == 4, "ALOAD is 1, 2 or 4");
    static_assert(A_T == 0 || A_MODE == LOAD_TMA, "a transposed A is loaded by TMA only");
    static constexpr bool A_XP = A_MODE == LOAD_TMA_XP;
    static_assert(!A_XP || B_MODE == LOAD_TMA, "the in-smem transpose runs with a TMA-loaded B");
    // The consumers read A as [BK][BM] (a transposed A, or the transposers'
    // output), with the chunk swizzle in the second case.
    static constexpr bool A_KROWS = A_T || A_XP;
    // TN: columns a lane owns (8, or 16 for a 32 x 128 warp tile: twice the
    // multiply-adds per shared load, for warps with up to 255 registers).
    static constexpr int TN = TN_;
    static_assert(TN == 8 || TN == 16, "TN is 8 or 16");
    static_assert(BK == 32, "A rows are one 128-byte swizzle span");
    static_assert(BM % 32 == 0 && BN % (8 * TN) == 0, "warp tile is 32 x 8 TN");
    static constexpr int WARPS_M = BM / 32, WARPS_N = BN / (8 * TN);
    // KSPLIT: groups of consumer warps that each cover the whole tile for
    // their own share of every stage's k (k-groups g KQ/KSPLIT .. ), their
    // sums added in group order in shared memory at the end of each work
    // item: more warps per SM for tiles too few to fill the GPU.
    static constexpr int KSPLIT = KSPLIT_;
    static_assert(KSPLIT == 1 || KSPLIT == 2 || KSPLIT == 4, "KSPLIT is 1, 2 or 4");
    static constexpr int GROUP_WARPS = WARPS_M * WARPS_N;
    static constexpr int CONSUMER_WARPS = GROUP_WARPS * KSPLIT;
    static constexpr int CONSUMERS = CONSUMER_WARPS * 32;
    static constexpr bool ANY_CP = (A_MODE == LOAD_CPASYNC) || (B_MODE == LOAD_CPASYNC);
    // FUSED: the transposed-A path with the transposed copy of a row-major A
    // and/or the row-major copy of a transposed B made inside this kernel by
    // three transposer warps per CTA (see GemmParams::at_flags, bt_flags and
    // at_transposer()) instead of by kernels before it.
    static constexpr bool FUSED = FUSED_ != 0;
    static constexpr bool ANY_TMA = (A_MODE != LOAD_CPASYNC) || (B_MODE == LOAD_TMA);
    // cp.async producers: one warp per SM sub-partition so the copy
    // instructions do not all land on one scheduler. With the in-smem
    // transpose: one TMA warp and three transposer warps (12 warps in all
    // for 128 x 128, still three per scheduler, so 168 registers a thread).
    static constexpr int PRODUCER_WARPS = (ANY_CP || A_XP || FUSED) ? 4 : 1;
    static constexpr int TRANSPOSERS = (A_XP || FUSED) ? 96 : 0;
    static constexpr int THREADS = CONSUMERS + 32 * PRODUCER_WARPS;
    static constexpr int A_BYTES = BM * BK * 4;
    static constexpr int B_BYTES = BK * BN * 4;
    static constexpr uint32_t TX_BYTES =
        (A_MODE != LOAD_CPASYNC ? A_BYTES : 0) + (B_MODE == LOAD_TMA ? B_BYTES : 0);
    // With the in-smem transpose the TMA bytes land on the "raw" barrier and
    // "full" counts the transposer threads.
    static constexpr uint32_t FULL_COUNT =
        A_XP ? TRANSPOSERS : (ANY_TMA ? 1 : 0) + (ANY_CP ? 32 * PRODUCER_WARPS : 0);
    static constexpr int RAW_BYTES = A_XP ? A_BYTES : 0;   // raw A staging, per stage
    static constexpr int RED_BYTES = (KSPLIT - 1) * BM * BN * 4;   // k-group sums
    static constexpr int CS = CS_;
    static_assert(CS == 1 || CS == 2 || CS == 4, "CS is 1, 2 or 4");
    // Other ranks' sums of the rows this rank finishes (cluster k-split).
    static constexpr int CKS_BYTES = (CS - 1) * BM * BN * 4 / CS;
    // FUSED: the transposer warps' staging tile, BM rows of BK + 1 floats.
    static constexpr int XT_BYTES = FUSED ? BM * (BK + 1) * 4 : 0;
    static constexpr int SMEM_BYTES = 1024 /* alignment slack */ +
                                      STAGES * (A_BYTES + B_BYTES + RAW_BYTES) + RED_BYTES +
                                      CKS_BYTES + XT_BYTES + (3 * STAGES + 6) * 8;
    static constexpr bool FUSED_OK = !FUSED || (A_T && A_MODE == LOAD_TMA &&
                                                B_MODE == LOAD_TMA && KSPLIT == 1 && CS == 1);
    static constexpr bool FITS = SMEM_BYTES <= 227 * 1024 && FUSED_OK;
    // Tiles of at most 128 x 64 are sized to run two CTAs per SM.
    static constexpr int MIN_BLOCKS = (BM * BN * KSPLIT <= 128 * 64) ? 2 : 1;
};

// Tile index -> (tile row, tile column), grouped so that the CTAs running at
// the same time share A row-blocks and B column-blocks in L2.
__device__ __forceinline__ void tile_coords(int t, const GemmParams& p, int& tm, int& tn) {
    const int per_group = p.group_m * p.tiles_n;
    const int g = t / per_group;
    const int first = g * p.group_m;
    const int gm = min(p.tiles_m - first, p.group_m);
    const int r = t - g * per_group;
    tm = first + r % gm;
    tn = r / gm;
}

// ---- work schedule ----------------------------------------------------------

// One work item: k-tiles [kb, ke) of tile `tile`. slot == kWhole: the item
// covers the whole tile and ends in the epilogue; slot == kFinish: the item
// holds the tile's first k-segment and finishes the tile (adds the other
// segments' slots, then the epilogue); slot >= 0: its raw sums go to
// workspace slot `slot`.
constexpr int kWhole = -1;
constexpr int kFinish = -2;

struct Item {
    int tile, kb, ke, slot;
};

// Start of stream-K range c (of sk_ctas) over sk_iters iterations.
__device__ __forceinline__ long long sk_start(long long c, const GemmParams& p) {
    return (c * p.sk_iters) / p.sk_ctas;
}

template <int CS = 1>
struct Schedule {
    int t_dp;            // next data-parallel tile
    long long s, i, e;   // this CTA's stream-K range [s, e), next iteration i

    __device__ __forceinline__ explicit Schedule(const GemmParams& p) {
        if (CS > 1) {
            // One item: this cluster's tile, this rank's share of its k-tiles.
            t_dp = static_cast<int>(cluster_id_x());
            const long long r = cluster_ctarank();
            s = i = r * p.k_tiles / CS;
            e = (r + 1) * p.k_tiles / CS;
            return;
        }
        t_dp = static_cast<int>(blockIdx.x);
        if (static_cast<int>(blockIdx.x) < p.sk_ctas) {
            s = sk_start(blockIdx.x, p);
            e = sk_start(blockIdx.x + 1, p);
        } else {
            s = e = 0;
        }
        i = s;
    }

    __device__ __forceinline__ bool next(const GemmParams& p, Item& it) {
        if (CS > 1) {
            if (t_dp < 0) return false;
            it.tile = t_dp;
            it.kb = static_cast<int>(s);
            it.ke = static_cast<int>(e);
            it.slot = kWhole;
            t_dp = -1;
            check(p, it);
            return true;
        }
        if (t_dp < p.dp_tiles) {
            it.tile = t_dp;
            it.kb = 0;
            it.ke = p.k_tiles;
            it.slot = kWhole;
            t_dp += static_cast<int>(gridDim.x);
            check(p, it);
            return true;
        }
        if (i >= e) return false;
        const long long u = i / p.k_tiles;
        const int kb = static_cast<int>(i - u * p.k_tiles);
        const long long left = e - i;
        const int ke = left < static_cast<long long>(p.k_tiles - kb) ? kb + static_cast<int>(left)
                                                                      : p.k_tiles;
        it.tile = p.dp_tiles + static_cast<int>(u);
        it.kb = kb;
        it.ke = ke;
        // Only the first and the last segment of a range can be partial. A
        // partial segment that starts at k-tile 0 is the range's last item
        // and, finishing in the kernel, completes the tile; one that starts
        // later is the range's first item and goes to slot c. For the fixup
        // kernel: the first segment to slot 2c, any later one to 2c + 1.
        if (kb == 0 && ke == p.k_tiles)
            it.slot = kWhole;
        else if (p.sk_fixup)
            it.slot = 2 * static_cast<int>(blockIdx.x) + (i == s ? 0 : 1);
        else
            it.slot = kb == 0 ? kFinish : static_cast<int>(blockIdx.x);
        i += ke - kb;
        check(p, it);
        return true;
    }

    // Debug build: every item names an existing tile, a k-range inside it
    // (non-empty, but for a cluster rank's share of a tile with fewer
    // k-tiles than ranks) and a slot the workspace has.
    __device__ __forceinline__ static void check(const GemmParams& p, const Item& it) {
        SG_DCHECK(p, it.tile >= 0 && it.tile < p.tiles_m * p.tiles_n);
        SG_DCHECK(p, it.kb >= 0 && (CS > 1 ? it.kb <= it.ke : it.kb < it.ke) &&
                         it.ke <= p.k_tiles);
        SG_DCHECK(p, it.slot == kWhole || it.slot == kFinish ||
                         (it.slot >= 0 && it.slot < (p.sk_fixup ? 2 : 1) * p.sk_ctas));
        SG_DCHECK(p, it.slot != kFinish || (it.kb == 0 && !p.sk_fixup));
    }
};

// ---- waits ------------------------------------------------------------------

// Bounded mbarrier wait. Returns false (after setting `code` in the status
// word) if the phase did not complete within p.timeout_ns.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity,
                                             const GemmParams& p, int code) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > p.timeout_ns) {
            atomicOr(p.status, code);
            return false;
        }
    }
}

// The same with acquire at cluster scope (a barrier other CTAs of the
// cluster arrive on after writing this CTA's shared memory).
__device__ __forceinline__ bool wait_bounded_cluster(uint32_t bar, uint32_t parity,
                                                     const GemmParams& p, int code) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (mbar_try_wait_cluster(bar, parity)) return true;
        if (globaltimer_ns() - t0 > p.timeout_ns) {
            atomicOr(p.status, code);
            return false;
        }
    }
}

// Bounded wait until *flag == tag (acquire at GPU scope). Returns false
// (after setting `code` in the status word) if it did not happen within
// p.timeout_ns.
__device__ __forceinline__ bool wait_flag_bounded(const unsigned long long* flag,
                                                  unsigned long long tag, const GemmParams& p,
                                                  int code) {
    if (ld_acquire_gpu(flag) == tag) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (ld_acquire_gpu(flag) == tag) return true;
        if (globaltimer_ns() - t0 > p.timeout_ns) {
            atomicOr(p.status, code);
            return false;
        }
    }
}

// The stream-K CTA whose range holds k-iteration g: the largest c with
// sk_start(c) <= g.
__device__ __forceinline__ long long sk_cta_of(long long g, const GemmParams& p) {
    return ((g + 1) * p.sk_ctas + p.sk_iters - 1) / p.sk_iters - 1;
}

// ---- producer -----------------------------------------------------------------

// Byte offset of A element (row r, column k) inside one stage: 128-byte rows,
// 16-byte chunk index XOR (r mod 8) — the TMA 128B swizzle pattern.
__device__ __forceinline__ uint32_t a_swz(int r, int k) {
    return static_cast<uint32_t>(r * 128 + ((((k >> 2) ^ r) & 7) << 4) + ((k & 3) << 2));
}

template <class C>
__device__ __forceinline__ void producer(const CUtensorMap* tmA, const CUtensorMap* tmB,
                                         const GemmParams& p, uint32_t sA, uint32_t sB,
                                         uint32_t sRaw, uint32_t full0, uint32_t empty0,
                                         uint32_t raw0, uint32_t sk_pub, int pw, int lane) {
    const bool tma_thread = C::ANY_TMA && pw == 0 && lane == 0;
    if (!C::ANY_CP && !tma_thread) return;
    if (tma_thread) {
        if (C::A_MODE != LOAD_CPASYNC) tma_prefetch_desc(tmA);
        if (C::B_MODE == LOAD_TMA) tma_prefetch_desc(tmB);
    }
    // The barrier the TMA bytes complete on: "full" for the consumers, or,
    // with the in-smem transpose, "raw" for the transposer warps.
    const uint32_t tx0 = C::A_XP ? raw0 : full0;
    int s = 0;
    uint32_t ph = 0;
    int issued = 0;
    bool ok = true;
    // The slot this CTA's consumers fill (an item finished by another CTA;
    // at most one per launch) and whose flag this thread releases, at GPU
    // scope, once the consumers have all arrived on sk_pub after their
    // stores (cumulativity carries their stores with the release). It checks
    // without blocking before each stage it issues later, and blocks
    // (bounded) only once it has nothing left to issue. The release is kept
    // off the consumers: their stores' write acknowledgements can take
    // microseconds when L2 is busy, and the extra state in their loop cost
    // registers in the hot loop.
    const bool publisher = pw == 0 && lane == 0;
    int pend = -1;
    Schedule<C::CS> sched(p);
    Item it;
    while (ok && sched.next(p, it)) {
        if (publisher && !p.sk_fixup && it.slot >= 0) pend = it.slot;
        int tm, tn;
        tile_coords(it.tile, p, tm, tn);
        const int m0 = tm * C::BM, n0 = tn * C::BN;
        for (int kt = it.kb; kt < it.ke; ++kt) {
            if (!wait_bounded(empty0 + 8 * s, ph ^ 1u, p, STATUS_PRODUCER_TIMEOUT)) {
                ok = false;
                break;
            }
            if (pend >= 0 && mbar_test_wait(sk_pub, 0)) {
                st_release_gpu(p.sk_flags + pend, p.sk_tag);
                pend = -1;
            }
            const uint32_t full = full0 + 8 * s;
            const uint32_t tx = tx0 + 8 * s;
            const uint32_t dA = sA + s * C::A_BYTES, dB = sB + s * C::B_BYTES;
            const int k0 = kt * C::BK;
            if (C::FUSED && tma_thread) {
                // The units of the transposed copies this stage reads are
                // written by some CTA's transposer warps in this kernel: wait
                // for their flags, then order the async-proxy loads after them.
                SG_DCHECK(p, tm < p.tiles_m && tn < p.tiles_n && kt < p.k_tiles);
                if ((p.at_src != nullptr &&
                     !wait_flag_bounded(p.at_flags + static_cast<long long>(tm) * p.k_tiles + kt,
                                        p.at_tag, p, STATUS_PRODUCER_TIMEOUT)) ||
                    (p.bt_src != nullptr &&
                     !wait_flag_bounded(p.bt_flags + static_cast<long long>(tn) * p.k_tiles + kt,
                                        p.at_tag, p, STATUS_PRODUCER_TIMEOUT))) {
                    ok = false;
                    break;
                }
                fence_proxy_async_global();
            }
            if (tma_thread) {
                mbar_arrive_expect_tx(tx, C::TX_BYTES);
                if (C::A_XP) {
                    tma_load_2d(sRaw + s * C::A_BYTES, tmA, tx, k0, m0);
                } else if (C::A_MODE == LOAD_TMA) {
                    if (C::A_T) tma_load_2d(dA, tmA, tx, m0, k0);
                    else tma_load_2d(dA, tmA, tx, k0, m0);
                }
                if (C::B_MODE == LOAD_TMA) tma_load_2d(dB, tmB, tx, n0, k0);
            }
            SG_DCHECK(p, s >= 0 && s < C::STAGES);
            if (C::A_MODE == LOAD_CPASYNC) {
                // One row of BK = 32 floats per warp instruction, lane = k.
                const int k = k0 + lane;
                for (int r = pw; r < C::BM; r += C::PRODUCER_WARPS) {
                    const int m = m0 + r;
                    const bool v = (m < p.M) && (k < p.K);
                    const float* src = v ? p.A + (long long)m * p.lda + k : p.A;
                    SG_DCHECK(p, a_swz(r, lane) + 4 <= static_cast<uint32_t>(C::A_BYTES));
                    cp_async_4(dA + a_swz(r, lane), src, v);
                }
            }
            if (C::B_MODE == LOAD_CPASYNC) {
                for (int kr = pw; kr < C::BK; kr += C::PRODUCER_WARPS) {
                    const int k = k0 + kr;
#pragma unroll
                    for (int j = 0; j < C::BN / 32; ++j) {
                        const int nn = j * 32 + lane;
                        const int n = n0 + nn;
                        const bool v = (k < p.K) && (n < p.N);
                        const float* src = v ? p.B + (long long)k * p.ldb + n : p.B;
                        SG_DCHECK(p, (kr * C::BN + nn) * 4 + 4 <= C::B_BYTES);
                        cp_async_4(dB + (kr * C::BN + nn) * 4, src, v);
                    }
                }
            }
            if (C::ANY_CP) cp_async_mbar_arrive_noinc(full);
            ++issued;
            if (++s == C::STAGES) { s = 0; ph ^= 1u; }
        }
    }
    if (ok && pend >= 0 && wait_bounded(sk_pub, 0, p, STATUS_PRODUCER_TIMEOUT))
        st_release_gpu(p.sk_flags + pend, p.sk_tag);
    if (!ok) {
        // Let the copies this thread started land before the CTA can exit:
        // wait (bounded) for the last phase of each stage it filled.
        const int n = issued < C::STAGES ? issued : C::STAGES;
        int ss = s;
        uint32_t pp = ph;
        for (int i = 0; i < n; ++i) {
            if (--ss < 0) { ss = C::STAGES - 1; pp ^= 1u; }
            wait_bounded(tx0 + 8 * ss, pp, p, STATUS_DRAIN_TIMEOUT);
        }
    }
    if (C::ANY_CP) asm volatile("cp.async.wait_all;" ::: "memory");
}

// ---- transposer (A_MODE == LOAD_TMA_XP) -------------------------------------------

// Three warps (t = 0..95) rewrite each landed raw A stage (BM rows of 32 k,
// 128B-swizzled as TMA wrote it) as BK rows of BM m for the consumers. Work
// unit: a 4 x 4 block (rows 4 mb.., k-chunk kb) read as four float4 (one per
// row) and written as four float4 (one per k). The eight lanes of a
// quarter-warp take kb = 0..7 of one mb: their reads hit eight different
// chunks of one 128-byte row, and their writes, at chunk mb ^ kb of k-rows
// 4 kb + c, eight different bank groups. Then each thread arrives on the
// stage's "full" barrier, which counts the 96 of them.
template <class C>
__device__ __forceinline__ void transposer(const GemmParams& p, const uint8_t* raw, uint8_t* sA,
                                           uint32_t raw0, uint32_t full0, int t) {
    constexpr int BLOCKS = C::BM * 2;   // (BM / 4) row groups x 8 k-chunks
    int s = 0;
    uint32_t ph = 0;
    Schedule<C::CS> sched(p);
    Item it;
    while (sched.next(p, it)) {
        for (int kt = it.kb; kt < it.ke; ++kt) {
            if (!wait_bounded(raw0 + 8 * s, ph, p, STATUS_PRODUCER_TIMEOUT)) return;
            const uint8_t* src = raw + s * C::A_BYTES;
            uint8_t* dst = sA + s * C::A_BYTES;
#pragma unroll 1
            for (int b = t; b < BLOCKS; b += C::TRANSPOSERS) {
                const int kb = b & 7, mb = b >> 3;
                float4 v[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int r = 4 * mb + j;
                    v[j] = *reinterpret_cast<const float4*>(src + r * 128 + (((kb ^ r) & 7) << 4));
                }
                const int chunk = mb ^ kb;
                uint8_t* d = dst + (4 * kb) * (C::BM * 4) + (chunk << 4);
                SG_DCHECK(p, (4 * mb + 3) * 128 + 128 <= C::A_BYTES);
                SG_DCHECK(p, (4 * kb + 3) * (C::BM * 4) + (chunk << 4) + 16 <= C::A_BYTES);
                *reinterpret_cast<float4*>(d) = make_float4(v[0].x, v[1].x, v[2].x, v[3].x);
                *reinterpret_cast<float4*>(d + C::BM * 4) = make_float4(v[0].y, v[1].y, v[2].y, v[3].y);
                *reinterpret_cast<float4*>(d + 2 * C::BM * 4) = make_float4(v[0].z, v[1].z, v[2].z, v[3].z);
                *reinterpret_cast<float4*>(d + 3 * C::BM * 4) = make_float4(v[0].w, v[1].w, v[2].w, v[3].w);
            }
            mbar_arrive(full0 + 8 * s);
            if (++s == C::STAGES) { s = 0; ph ^= 1u; }
        }
    }
}

// ---- transposer warps of the fused transposed copies (Cfg::FUSED) ------------------

// Three warps (t = 0..95) of every CTA write the transposed copies the TMA
// producers load: of a row-major A (unit (tm, kt): A's rows tm BM .. + BM and
// columns kt BK .. + BK, stored at rows kt BK .. and columns tm BM .. of the
// copy) and of a transposed B (unit (tn, kt): rows tn BN .. of the stored
// N x K B, columns kt BK .., stored at rows kt BK .. and columns tn BN .. of
// B's row-major copy), whichever the call has. The units are taken in the
// order the tiles first need them (see at_transposer) and dealt out
// round-robin over the CTAs, so the first wave's first k-tiles are done
// first, by many CTAs at once. A unit goes through a staging tile in shared
// memory (BM rows of BK + 1 floats: the 128-byte row reads and the column
// reads both stay within a bank or two), 128-byte rows in, 512-byte rows of
// the copy out, both 16-byte vectors where the source allows. Elements past
// the matrix are neither read nor written (the tensor maps' bounds supply
// zeros). After a unit's stores every thread fences them for the async proxy
// and at GPU scope, the 96 threads meet at named barrier 1, and one releases
// the unit's flag. Nothing here waits on another CTA, so every unit gets done.
template <class C>
__device__ __forceinline__ void transpose_unit(const GemmParams& p, float* xt, int t,
                                               const float* src, long long lds, bool vec,
                                               float* dst, long long ldd, int rows, int r0, int k0) {
    constexpr int BR = C::BM, BK = C::BK, LD = C::BK + 1;
    // Source rows in: BR rows x BK / 4 float4.
#pragma unroll 2
    for (int q = t; q < BR * (BK / 4); q += C::TRANSPOSERS) {
        const int rr = q / (BK / 4), c4 = (q % (BK / 4)) * 4;
        const int r = r0 + rr, k = k0 + c4;
        float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (r < rows) {
            const float* sp = src + static_cast<long long>(r) * lds + k;
            if (vec && k + 3 < p.K) {
                v = *reinterpret_cast<const float4*>(sp);
            } else {
                if (k < p.K) v.x = sp[0];
                if (k + 1 < p.K) v.y = sp[1];
                if (k + 2 < p.K) v.z = sp[2];
                if (k + 3 < p.K) v.w = sp[3];
            }
        }
        SG_DCHECK(p, (rr * LD + c4 + 3) * 4 + 4 <= C::XT_BYTES);
        float* d = xt + rr * LD + c4;
        d[0] = v.x;
        d[1] = v.y;
        d[2] = v.z;
        d[3] = v.w;
    }
    named_bar_sync(1, C::TRANSPOSERS);
    // Rows of the copy out: BK rows x BR / 4 float4 (ldd is a multiple of 4
    // and r a multiple of 4 below rows, so the float4 stays in the row).
#pragma unroll 2
    for (int q = t; q < BK * (BR / 4); q += C::TRANSPOSERS) {
        const int kk = q / (BR / 4), r4 = (q % (BR / 4)) * 4;
        const int k = k0 + kk, r = r0 + r4;
        if (k < p.K && r < rows) {
            SG_DCHECK(p, r + 3 < ldd && ((r4 + 3) * LD + kk) * 4 + 4 <= C::XT_BYTES);
            *reinterpret_cast<float4*>(dst + static_cast<long long>(k) * ldd + r) =
                make_float4(xt[r4 * LD + kk], xt[(r4 + 1) * LD + kk], xt[(r4 + 2) * LD + kk],
                            xt[(r4 + 3) * LD + kk]);
        }
    }
    fence_proxy_async_global();
    __threadfence();
    named_bar_sync(1, C::TRANSPOSERS);
}

template <class C>
__device__ __forceinline__ void at_transposer(const GemmParams& p, float* xt, int t) {
    static_assert(!C::FUSED || (C::BK == 32 && C::BM == C::BN && C::BM % 4 == 0),
                  "units of 32 k x BM");
    const bool do_a = p.at_src != nullptr, do_b = p.bt_src != nullptr;
    const bool vec_a = do_a && (reinterpret_cast<uintptr_t>(p.at_src) % 16 == 0) &&
                       (p.at_lds % 4 == 0);
    const bool vec_b = do_b && (reinterpret_cast<uintptr_t>(p.bt_src) % 16 == 0) &&
                       (p.bt_lds % 4 == 0);
    // The raster visits raster group 0 (gmr tile rows) column by column, so
    // the data-parallel wave w first needs B's column blocks up to tn_end(w).
    const int gmr = min(p.tiles_m, p.group_m);
    const int grid = static_cast<int>(gridDim.x);
    auto tn_end = [&](int w) {
        const long long e = (static_cast<long long>(w + 1) * grid + gmr - 1) / gmr;
        return static_cast<int>(e < p.tiles_n ? e : p.tiles_n);
    };
    // Order: (1) k-tile by k-tile, group 0's A units and the first wave's B
    // units; (2) wave by wave, k-tile by k-tile, the B units a later wave
    // needs first; (3) raster group by raster group, k-tile by k-tile, tile
    // row by tile row, the A units of groups 1.. (B's column blocks are all
    // needed again by each group, A's rows only by their own).
    const long long per_group = static_cast<long long>(p.group_m) * p.k_tiles;
    const int gm0 = do_a ? gmr : 0;
    const int nb0 = do_b ? tn_end(0) : 0;
    const int per_kt = gm0 + nb0;
    const long long first = static_cast<long long>(per_kt) * p.k_tiles;
    const long long b_rest = do_b ? static_cast<long long>(p.tiles_n - nb0) * p.k_tiles : 0;
    const long long a_units = do_a ? static_cast<long long>(p.tiles_m) * p.k_tiles : 0;
    const long long units =
        first + b_rest + (a_units - static_cast<long long>(gm0) * p.k_tiles);
    for (long long u = blockIdx.x; u < units; u += gridDim.x) {
        int kt = 0, tm = -1, tn = -1;
        if (u < first) {
            kt = static_cast<int>(u / per_kt);
            const int r = static_cast<int>(u - static_cast<long long>(kt) * per_kt);
            if (r < gm0) tm = r;
            else tn = r - gm0;
        } else if (u < first + b_rest) {
            long long v = u - first;
            int start = nb0;
            for (int w = 1;; ++w) {
                const int end = tn_end(w);
                const long long cnt = static_cast<long long>(end - start) * p.k_tiles;
                if (v < cnt) {
                    kt = static_cast<int>(v / (end - start));
                    tn = start + static_cast<int>(v - static_cast<long long>(kt) * (end - start));
                    break;
                }
                v -= cnt;
                start = end;
            }
        } else {
            const long long ua = u - first - b_rest + static_cast<long long>(gm0) * p.k_tiles;
            const int g = static_cast<int>(ua / per_group);
            const long long r = ua - g * per_group;
            const int gm = min(p.tiles_m - g * p.group_m, p.group_m);
            kt = static_cast<int>(r / gm);
            tm = g * p.group_m + static_cast<int>(r - static_cast<long long>(kt) * gm);
        }
        SG_DCHECK(p, kt >= 0 && kt < p.k_tiles && (tm >= 0) != (tn >= 0) &&
                         tm < p.tiles_m && tn < p.tiles_n && (tm < 0 || do_a) &&
                         (tn < 0 || do_b));
        unsigned long long* flag;
        if (tm >= 0) {
            transpose_unit<C>(p, xt, t, p.at_src, p.at_lds, vec_a, const_cast<float*>(p.A), p.lda,
                              p.M, tm * C::BM, kt * C::BK);
            flag = p.at_flags + static_cast<long long>(tm) * p.k_tiles + kt;
        } else {
            transpose_unit<C>(p, xt, t, p.bt_src, p.bt_lds, vec_b, const_cast<float*>(p.B), p.ldb,
                              p.N, tn * C::BN, kt * C::BK);
            flag = p.bt_flags + static_cast<long long>(tn) * p.k_tiles + kt;
        }
        if (t == 0) st_release_gpu(flag, p.at_tag);
    }
}

// ---- consumer -----------------------------------------------------------------

// Offset of a lane's row i (0..7) from its row_base (see consumer()).
template <class C>
__device__ __forceinline__ constexpr int lane_row(int i) {
    return C::A_KROWS ? (i & 3) + 16 * (i >> 2) : 4 * i;
}

// A fragment of k-group kq (4 consecutive k) for the lane's 8 rows
// {tr, tr+4, ..., tr+28}: row r's 16-byte chunk kq sits at chunk kq ^ (r % 8),
// and r % 8 is tr for even i, tr + 4 (= tr ^ 4) for odd i.
__device__ __forceinline__ void load_a_group(float4 (&a)[8], const uint8_t* a_rows, int kq, int tr) {
    const int c0 = ((kq ^ tr) & 7) << 4;
    const int c1 = c0 ^ 64;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        a[i] = *reinterpret_cast<const float4*>(a_rows + i * 4 * 128 + ((i & 1) ? c1 : c0));
}

__device__ __forceinline__ float lane_of(const float4& v, int kk) {
    return kk == 0 ? v.x : kk == 1 ? v.y : kk == 2 ? v.z : v.w;
}

// One k-step of the 8 x TN register outer product (b: the lane's TN B
// values of this k as TN / 4 float4).
//   FORDER 0: scalar FFMA.
//   FORDER 2: packed FFMA2 (fma.rn.f32x2: two IEEE single-precision FMAs,
//             each rounded once, in one instruction): pairs of adjacent
//             columns share one instruction with the row's A value in both
//             lanes, rows outer. Every output still sees the same FMA
//             sequence, so the result is bit-identical to the scalar form.
//   FORDER 3: the same with the column pairs outer: consecutive
//             instructions share the B pair and change the A value.
template <int FORDER, int TN>
__device__ __forceinline__ void outer_product(float (&acc)[8][TN], const float (&av8)[8],
                                              const float4 (&b)[TN / 4]) {
    float2 bp[TN / 2];
#pragma unroll
    for (int h = 0; h < TN / 4; ++h) {
        bp[2 * h] = make_float2(b[h].x, b[h].y);
        bp[2 * h + 1] = make_float2(b[h].z, b[h].w);
    }
    if (FORDER == 3) {
#pragma unroll
        for (int jp = 0; jp < TN / 2; ++jp) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float av = av8[i];
                float2 c = make_float2(acc[i][2 * jp], acc[i][2 * jp + 1]);
                c = __ffma2_rn(make_float2(av, av), bp[jp], c);
                acc[i][2 * jp] = c.x;
                acc[i][2 * jp + 1] = c.y;
            }
        }
    } else if (FORDER == 2) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float av = av8[i];
            const float2 aa = make_float2(av, av);
#pragma unroll
            for (int jp = 0; jp < TN / 2; ++jp) {
                float2 c = make_float2(acc[i][2 * jp], acc[i][2 * jp + 1]);
                c = __ffma2_rn(aa, bp[jp], c);
                acc[i][2 * jp] = c.x;
                acc[i][2 * jp + 1] = c.y;
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float av = av8[i];
#pragma unroll
            for (int jp = 0; jp < TN / 2; ++jp) {
                acc[i][2 * jp] = fmaf(av, bp[jp].x, acc[i][2 * jp]);
                acc[i][2 * jp + 1] = fmaf(av, bp[jp].y, acc[i][2 * jp + 1]);
            }
        }
    }
}

template <class C>
__device__ __forceinline__ void consumer(const GemmParams& p, const uint8_t* sA_ptr,
                                         const uint8_t* sB_ptr, uint32_t full0, uint32_t empty0,
                                         float4* red, uint32_t red_full, uint32_t red_empty,
                                         float4* cks, uint32_t cks_full, volatile int* sk_fail,
                                         uint32_t sk_pub, uint32_t sk_go, int warp, int lane) {
    // k-group of this warp (KSPLIT > 1) and its place in the group's tile.
    const int grp = C::KSPLIT > 1 ? warp / C::GROUP_WARPS : 0;
    const int wq = C::KSPLIT > 1 ? warp % C::GROUP_WARPS : warp;
    const int wm = wq % C::WARPS_M, wn = wq / C::WARPS_M;
    uint32_t red_ph = 0;
    const int tr = C::LMAP == 1 ? (lane & 3) : (lane >> 3);
    const int tc = C::LMAP == 1 ? (lane >> 2) : (lane & 7);
    // Lane rows: row_base + 4 i (row-major A: one swizzled 128-byte row per
    // row, so rows 4 apart spread over the chunks), or, for a transposed A,
    // row_base + (i & 3) + 16 (i >> 2) with row_base a multiple of 4 (two
    // float4 runs along m per k).
    const int row_base = C::A_KROWS ? wm * 32 + 4 * tr : wm * 32 + tr;
    // Lane columns: col_base + 32 h + {0..3}, h = 0 .. TN / 4 - 1.
    const int col_base = wn * (8 * C::TN) + 4 * tc;
    constexpr int KQ = C::BK / 4;

    int s = 0;
    uint32_t ph = 0;
    Schedule<C::CS> sched(p);
    Item it;
    while (sched.next(p, it)) {
        float acc[8][C::TN];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < C::TN; ++j) acc[i][j] = 0.0f;

        if (it.slot < 0 && p.beta != 0.0f && grp == 0) {
            // The epilogue reads this tile of C: start moving it into L2 now.
            // Lane l takes row l of the warp tile, the 128-byte lines of its
            // 8 TN columns (those that start inside the matrix).
            int tm, tn;
            tile_coords(it.tile, p, tm, tn);
            const int r = tm * C::BM + wm * 32 + lane;
            const int c = tn * C::BN + wn * (8 * C::TN);
            if (r < p.M) {
                const float* crow = p.C + (long long)r * p.ldc + c;
#pragma unroll
                for (int h = 0; h < C::TN / 4; ++h)
                    if (c + 32 * h < p.N) prefetch_l2(crow + 32 * h);
            }
        }

        bool ready = false;   // EARLY: stage s already seen complete
        for (int kt = it.kb; kt < it.ke; ++kt) {
            if (!ready && !wait_bounded(full0 + 8 * s, ph, p, STATUS_CONSUMER_TIMEOUT)) return;
            ready = false;
            // [BK][BM] stages: a transposed A is addressed directly; the
            // transposers' output has chunk q of k-row k at q ^ ((k / 4) % 8),
            // so the lane's two chunks are found per k-group below.
            const uint8_t* a_st = C::A_XP ? sA_ptr + s * C::A_BYTES
                                  : C::A_T ? sA_ptr + s * C::A_BYTES + row_base * 4
                                           : sA_ptr + s * C::A_BYTES + row_base * 128;
            const uint8_t* b_st = sB_ptr + s * C::B_BYTES + col_base * 4;
            const int s_nx = (s + 1 == C::STAGES) ? 0 : s + 1;
            const uint32_t ph_nx = (s + 1 == C::STAGES) ? (ph ^ 1u) : ph;
            constexpr int KQG = KQ / C::KSPLIT;   // k-groups of 4 k per k-group of warps
#pragma unroll
            for (int kql = 0; kql < KQG; ++kql) {
                const int kq = grp * KQG + kql;
                if (C::EARLY && kql == KQG / 2 && kt + 1 < it.ke)
                    ready = mbar_test_wait(full0 + 8 * s_nx, ph_nx);
                float4 a[8];
                if (!C::A_KROWS && C::ALOAD == 4) load_a_group(a, a_st, kq, tr);
                // Transposer layout: byte offsets of the lane's chunks (rows
                // row_base.. and row_base + 16..) in k-rows 4 kq .. 4 kq + 3.
                const int xq0 = ((((row_base >> 2) ^ kq) & 7) | ((row_base >> 2) & ~7)) << 4;
                const int xq1 = (((((row_base >> 2) + 4) ^ kq) & 7) | (((row_base >> 2) + 4) & ~7)) << 4;
                // Byte offsets of the lane's chunk kq in even and odd rows.
                const int c0 = ((kq ^ tr) & 7) << 4, c1 = c0 ^ 64;
                SG_DCHECK(p, ((kq * 4 + 3) * C::BN + col_base + 32 * (C::TN / 4 - 1)) * 4 + 16 <=
                                 C::B_BYTES);
                SG_DCHECK(p, C::A_KROWS ? ((kq * 4 + 3) * C::BM + row_base + 16) * 4 + 16 <= C::A_BYTES
                                        : (row_base + 28) * 128 + 128 <= C::A_BYTES);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint8_t* brow = b_st + (kq * 4 + kk) * C::BN * 4;
                    float4 bq[C::TN / 4];
#pragma unroll
                    for (int h = 0; h < C::TN / 4; ++h)
                        bq[h] = *reinterpret_cast<const float4*>(brow + 32 * 4 * h);
                    float av[8];
                    if (C::A_KROWS) {
                        const uint8_t* arow = a_st + (kq * 4 + kk) * C::BM * 4;
                        const float4 a0 = *reinterpret_cast<const float4*>(arow + (C::A_XP ? xq0 : 0));
                        const float4 a1 = *reinterpret_cast<const float4*>(arow + (C::A_XP ? xq1 : 16 * 4));
                        av[0] = a0.x; av[1] = a0.y; av[2] = a0.z; av[3] = a0.w;
                        av[4] = a1.x; av[5] = a1.y; av[6] = a1.z; av[7] = a1.w;
                    } else {
                        if (C::ALOAD == 4) {
#pragma unroll
                            for (int i = 0; i < 8; ++i) av[i] = lane_of(a[i], kk);
                        } else if (C::ALOAD == 2) {
                            if ((kk & 1) == 0) {
#pragma unroll
                                for (int i = 0; i < 8; ++i) {
                                    const float2 v = *reinterpret_cast<const float2*>(
                                        a_st + i * 4 * 128 + ((i & 1) ? c1 : c0) + kk * 4);
                                    a[i].x = v.x;
                                    a[i].y = v.y;
                                }
                            }
#pragma unroll
                            for (int i = 0; i < 8; ++i) av[i] = (kk & 1) ? a[i].y : a[i].x;
                        } else {
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                av[i] = *reinterpret_cast<const float*>(
                                    a_st + i * 4 * 128 + ((i & 1) ? c1 : c0) + kk * 4);
                        }
                    }
                    outer_product<C::FORDER, C::TN>(acc, av, bq);
                }
            }
            mbar_arrive(empty0 + 8 * s);
            s = s_nx;
            ph = ph_nx;
        }

        if (C::KSPLIT > 1) {
            // Add the k-groups' sums in group order: groups 1.. leave theirs
            // in shared memory (float4 j of lane l of warp wq at
            // ((g - 1) GROUP_WARPS + wq) 2 TN + j, lane-interleaved), group 0
            // adds them to its own and goes on to the epilogue.
            constexpr int NF4 = 8 * C::TN / 4;   // float4 of accumulators a lane
            if (grp > 0) {
                if (!wait_bounded(red_empty, red_ph ^ 1u, p, STATUS_CONSUMER_TIMEOUT)) return;
                float4* dst = red + (((grp - 1) * C::GROUP_WARPS + wq) * NF4) * 32 + lane;
                SG_DCHECK(p, ((((grp - 1) * C::GROUP_WARPS + wq) * NF4 + NF4 - 1) * 32 + lane + 1) * 16 <=
                                 C::RED_BYTES);
#pragma unroll
                for (int i = 0; i < 8; ++i)
#pragma unroll
                    for (int h = 0; h < C::TN / 4; ++h)
                        dst[(i * (C::TN / 4) + h) * 32] =
                            make_float4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2],
                                        acc[i][4 * h + 3]);
                mbar_arrive(red_full);
                red_ph ^= 1u;
                continue;
            }
            if (!wait_bounded(red_full, red_ph, p, STATUS_CONSUMER_TIMEOUT)) return;
#pragma unroll 1
            for (int g = 1; g < C::KSPLIT; ++g) {
                const float4* srcg = red + (((g - 1) * C::GROUP_WARPS + wq) * NF4) * 32 + lane;
#pragma unroll
                for (int i = 0; i < 8; ++i)
#pragma unroll
                    for (int h = 0; h < C::TN / 4; ++h) {
                        const float4 v = srcg[(i * (C::TN / 4) + h) * 32];
                        acc[i][4 * h] += v.x;
                        acc[i][4 * h + 1] += v.y;
                        acc[i][4 * h + 2] += v.z;
                        acc[i][4 * h + 3] += v.w;
                    }
            }
            mbar_arrive(red_empty);
            red_ph ^= 1u;
        }

        if (C::CS > 1) {
            // Cluster k-split, reduce-scatter: rank r finishes the
            // accumulator rows i in [r R, (r + 1) R), R = 8 / CS, of every
            // lane of group 0, and writes only those rows of C. Each rank
            // stores the rows another rank finishes into that rank's shared
            // memory (its slot there: ranks below the receiver in rank order,
            // then those above; float4 j of lane l of warp wq of slot s at
            // (s GROUP_WARPS + wq) R TN / 4 + j, lane-interleaved), arrives on
            // its barrier, then waits for its own and adds the ranks' sums in
            // rank order: the order rank 0 alone would add them in, so the
            // bits do not depend on which rank finishes a row. One item per
            // CTA, so the phase is 0.
            constexpr int R = 8 / C::CS;
            constexpr int NF4 = R * C::TN / 4;
            const uint32_t rank = cluster_ctarank();
            SG_DCHECK(p, rank < static_cast<uint32_t>(C::CS));
#pragma unroll
            for (int d = 0; d < C::CS; ++d) {
                if (static_cast<uint32_t>(d) == rank) continue;
                const int slot = static_cast<int>(rank) < d ? static_cast<int>(rank)
                                                            : static_cast<int>(rank) - 1;
                SG_DCHECK(p, (((slot * C::GROUP_WARPS + wq) * NF4 + NF4 - 1) * 32 + lane + 1) * 16 <=
                                 C::CKS_BYTES);
                const uint32_t dst = mapa_shared(
                    smem_u32(cks + ((slot * C::GROUP_WARPS + wq) * NF4) * 32 + lane),
                    static_cast<uint32_t>(d));
#pragma unroll
                for (int ii = 0; ii < R; ++ii)
#pragma unroll
                    for (int h = 0; h < C::TN / 4; ++h)
                        st_cluster_v4(dst + (ii * (C::TN / 4) + h) * 32 * 16,
                                      make_float4(acc[d * R + ii][4 * h], acc[d * R + ii][4 * h + 1],
                                                  acc[d * R + ii][4 * h + 2],
                                                  acc[d * R + ii][4 * h + 3]));
                mbar_arrive_remote(mapa_shared(cks_full, static_cast<uint32_t>(d)));
            }
            if (!wait_bounded_cluster(cks_full, 0, p, STATUS_CONSUMER_TIMEOUT)) return;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (static_cast<uint32_t>(i / R) != rank) continue;
                const int ii = i % R;
#pragma unroll
                for (int h = 0; h < C::TN / 4; ++h) {
                    const float4 own = make_float4(acc[i][4 * h], acc[i][4 * h + 1],
                                                   acc[i][4 * h + 2], acc[i][4 * h + 3]);
                    float4 t = own;
#pragma unroll
                    for (int r = 0; r < C::CS; ++r) {
                        float4 v = own;
                        if (static_cast<uint32_t>(r) != rank) {
                            const int slot = r < static_cast<int>(rank) ? r : r - 1;
                            v = cks[((slot * C::GROUP_WARPS + wq) * NF4 + ii * (C::TN / 4) + h) * 32 +
                                    lane];
                        }
                        if (r == 0) {
                            t = v;
                        } else {
                            t.x += v.x;
                            t.y += v.y;
                            t.z += v.z;
                            t.w += v.w;
                        }
                    }
                    acc[i][4 * h] = t.x;
                    acc[i][4 * h + 1] = t.y;
                    acc[i][4 * h + 2] = t.z;
                    acc[i][4 * h + 3] = t.w;
                }
            }
        }

        // From here on only group 0's consumer threads hold the tile's sums
        // (the other k-groups have moved on to their next item).
        if (it.slot >= 0) {
            // Partial tile: raw sums to the workspace slot, row-major BM x BN,
            // bypassing L1 (the finishing CTA or sk_fixup_kernel reads them
            // from L2).
            float* slot = p.ws + static_cast<long long>(it.slot) * (C::BM * C::BN);
            SG_DCHECK(p, p.ws != nullptr && it.slot < (p.sk_fixup ? 2 : 1) * p.sk_ctas);
            SG_DCHECK(p, row_base + lane_row<C>(7) < C::BM && col_base + 32 * (C::TN / 4 - 1) + 4 <= C::BN);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float* row = slot + (row_base + lane_row<C>(i)) * C::BN + col_base;
#pragma unroll
                for (int h = 0; h < C::TN / 4; ++h)
                    __stcg(reinterpret_cast<float4*>(row + 32 * h),
                           make_float4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2],
                                       acc[i][4 * h + 3]));
            }
            // Publish the slot: every thread arrives on sk_pub (release at CTA
            // scope) after its stores; the producer thread releases the flag
            // at GPU scope once sk_pub has completed (see producer()).
            if (!p.sk_fixup) mbar_arrive(sk_pub);
            continue;
        }
        if (it.slot == kFinish) {
            // This CTA holds the tile's first k-segment [0, ke): add the
            // segments [ke, k_tiles) that the next CTAs left in their slots,
            // in increasing k order (the order sk_fixup_kernel uses, so the
            // bits are the same). Warp 0 of the group waits for their flags,
            // a lane per flag (a tile split over many CTAs costs one round
            // trip, not one per segment), resets them to 0 for a later
            // replay of the same launch and arrives on sk_go, which the
            // other warps wait on (bounded): that hands the lanes' acquires
            // to them. A CTA finishes at most one tile per launch (phase 0).
            const long long u = it.tile - p.dp_tiles;
            const long long c0 = sk_cta_of(u * p.k_tiles + it.ke, p);
            const long long c1 = sk_cta_of(u * p.k_tiles + p.k_tiles - 1, p);
            SG_DCHECK(p, c0 > static_cast<long long>(blockIdx.x) && c0 <= c1 && c1 < p.sk_ctas);
            SG_DCHECK(p, p.sk_flags != nullptr && p.sk_tag != 0ull);
            if (wq == 0) {
                int fail = 0;
                for (long long c = c0 + lane; c <= c1 && !fail; c += 32)
                    if (!wait_flag_bounded(p.sk_flags + c, p.sk_tag, p, STATUS_CONSUMER_TIMEOUT))
                        fail = 1;
                fail = __any_sync(0xffffffffu, fail);
                if (!fail)
                    for (long long c = c0 + lane; c <= c1; c += 32) p.sk_flags[c] = 0ull;
                __syncwarp();
                if (lane == 0) {
                    *sk_fail = fail;
                    mbar_arrive(sk_go);
                }
                __syncwarp();
            } else if (!wait_bounded(sk_go, 0, p, STATUS_CONSUMER_TIMEOUT)) {
                return;
            }
            if (*sk_fail) return;
#pragma unroll 1
            for (long long c = c0; c <= c1; ++c) {
                const float* slot = p.ws + c * (C::BM * C::BN);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float* row = slot + (row_base + lane_row<C>(i)) * C::BN + col_base;
#pragma unroll
                    for (int h = 0; h < C::TN / 4; ++h) {
                        const float4 v = __ldcg(reinterpret_cast<const float4*>(row + 32 * h));
                        acc[i][4 * h] += v.x;
                        acc[i][4 * h + 1] += v.y;
                        acc[i][4 * h + 2] += v.z;
                        acc[i][4 * h + 3] += v.w;
                    }
                }
            }
        }

        // Epilogue: C = alpha * acc + beta * C, straight from registers; in
        // a cluster k-split only the rows this rank finished.
        const int own_lo = C::CS > 1 ? static_cast<int>(cluster_ctarank()) * (8 / C::CS) : 0;
        const int own_hi = own_lo + 8 / C::CS;
        int tm, tn;
        tile_coords(it.tile, p, tm, tn);
        const int m0 = tm * C::BM + row_base;
        const int n0 = tn * C::BN + col_base;
        const bool use_c = p.beta != 0.0f;
        // Two halves of four rows: each half first reads all the old-C
        // float4s it owns, then writes, so eight loads are in flight together
        // instead of one round trip per store (the compiler cannot move a
        // load of C above a store to C). Half the rows at a time keeps the
        // extra registers within the budget of the main loop.
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            float4 cold[4][C::TN / 4];
            if (use_c) {
#pragma unroll
                for (int ii = 0; ii < 4; ++ii) {
                    const int m = m0 + lane_row<C>(4 * q + ii);
                    const bool own = 4 * q + ii >= own_lo && 4 * q + ii < own_hi;
#pragma unroll
                    for (int h = 0; h < C::TN / 4; ++h) {
                        const int n = n0 + 32 * h;
                        cold[ii][h] = (own && m < p.M && p.c_vec && n + 3 < p.N)
                                          ? *reinterpret_cast<const float4*>(p.C + (long long)m * p.ldc + n)
                                          : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    }
                }
            }
#pragma unroll
            for (int ii = 0; ii < 4; ++ii) {
                const int i = 4 * q + ii;
                const int m = m0 + lane_row<C>(i);
                if (m >= p.M || i < own_lo || i >= own_hi) continue;
                float* crow = p.C + (long long)m * p.ldc;
                SG_DCHECK(p, m >= 0 && n0 >= 0 && n0 % 4 == 0);
#pragma unroll
                for (int h = 0; h < C::TN / 4; ++h) {
                    const int n = n0 + 32 * h;
                    float v[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) v[e] = p.alpha * acc[i][4 * h + e];
                    if (p.c_vec && n + 3 < p.N) {
                        if (use_c) {
                            const float4 c = cold[ii][h];
                            v[0] = fmaf(p.beta, c.x, v[0]);
                            v[1] = fmaf(p.beta, c.y, v[1]);
                            v[2] = fmaf(p.beta, c.z, v[2]);
                            v[3] = fmaf(p.beta, c.w, v[3]);
                        }
                        *reinterpret_cast<float4*>(crow + n) = make_float4(v[0], v[1], v[2], v[3]);
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            if (n + e < p.N) {
                                float out = v[e];
                                if (use_c) out = fmaf(p.beta, crow[n + e], out);
                                crow[n + e] = out;
                            }
                        }
                    }
                }
            }
        }
    }
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, C::MIN_BLOCKS)
sgemm_ws_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const GemmParams p) {
    static_assert(C::FITS, "ring does not fit in 227 KB of shared memory");
    extern __shared__ __align__(16) uint8_t smem_raw[];
    // 1024-byte alignment: the 128B-swizzle pattern repeats every 8 rows.
    // (Pointer arithmetic on the __shared__ array keeps the shared address
    // space visible to the compiler, so the tile reads stay LDS.)
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* sA = smem;
    uint8_t* sB = smem + C::STAGES * C::A_BYTES;
    uint8_t* sRaw = sB + C::STAGES * C::B_BYTES;      // C::RAW_BYTES per stage
    float4* red = reinterpret_cast<float4*>(sRaw + C::STAGES * C::RAW_BYTES);  // RED_BYTES
    float4* cks = reinterpret_cast<float4*>(sRaw + C::STAGES * C::RAW_BYTES + C::RED_BYTES);
    float* xt = reinterpret_cast<float*>(sRaw + C::STAGES * C::RAW_BYTES + C::RED_BYTES +
                                         C::CKS_BYTES);   // C::XT_BYTES
    uint64_t* bars = reinterpret_cast<uint64_t*>(sRaw + C::STAGES * C::RAW_BYTES + C::RED_BYTES +
                                                 C::CKS_BYTES + C::XT_BYTES);
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = smem_u32(bars + C::STAGES);
    const uint32_t raw0 = smem_u32(bars + 2 * C::STAGES);
    const uint32_t red_full = smem_u32(bars + 3 * C::STAGES);
    const uint32_t red_empty = red_full + 8;
    const uint32_t cks_full = red_full + 16;
    volatile int* sk_fail = reinterpret_cast<volatile int*>(bars + 3 * C::STAGES + 3);
    const uint32_t sk_pub = red_full + 32;
    const uint32_t sk_go = red_full + 40;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full0 + 8 * s, C::FULL_COUNT);
            mbar_init(empty0 + 8 * s, C::CONSUMERS);
            if (C::A_XP) mbar_init(raw0 + 8 * s, 1);
        }
        if (C::KSPLIT > 1) {
            mbar_init(red_full, (C::KSPLIT - 1) * C::GROUP_WARPS * 32);
            mbar_init(red_empty, C::GROUP_WARPS * 32);
        }
        if (C::CS > 1) mbar_init(cks_full, (C::CS - 1) * C::GROUP_WARPS * 32);
        // In-kernel stream-K finishing: group 0's consumers publish a slot
        // through sk_pub; the flag-waiting thread releases the others
        // through sk_go.
        mbar_init(sk_pub, C::GROUP_WARPS * 32);
        mbar_init(sk_go, 1);
        fence_barrier_init();
    }
    __syncthreads();
    // The other CTAs of the cluster arrive on cks_full only after it has
    // been initialised: every thread of the cluster passes this first.
    if (C::CS > 1) cluster_sync();
    // Up to here only shared memory and kernel parameters were touched; the
    // kernel before this one on the stream (a packing copy of an operand)
    // may still be running until this returns.
    griddep_wait();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp >= C::CONSUMER_WARPS) {
        const int pw = warp - C::CONSUMER_WARPS;
        if (C::A_XP && pw > 0)
            transposer<C>(p, sRaw, sA, raw0, full0, (pw - 1) * 32 + lane);
        else if (C::FUSED && pw > 0)
            at_transposer<C>(p, xt, (pw - 1) * 32 + lane);
        else
            producer<C>(&tmA, &tmB, p, smem_u32(sA), smem_u32(sB), smem_u32(sRaw), full0, empty0,
                        raw0, sk_pub, pw, lane);
    } else {
        consumer<C>(p, sA, sB, full0, empty0, red, red_full, red_empty, cks, cks_full, sk_fail,
                    sk_pub, sk_go, warp, lane);
    }
    // No CTA of a cluster leaves while another may still write its shared
    // memory: every role returns here (all of their waits are bounded).
    if (C::CS > 1) cluster_sync();
}

}  // namespace sg
