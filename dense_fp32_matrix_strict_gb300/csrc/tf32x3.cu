// tf32x3.cu — sgemm_3xtf32: FP32 SGEMM on the 5th-generation tensor cores
// (tcgen05, TMEM accumulators) by the three-term TF32 split.
//
// Every FP32 input x is split into x_hi = tf32(x) and x_lo = tf32(x - x_hi)
// (round to nearest, ties away). Then
//     a * b ~ a_hi*b_hi + a_hi*b_lo + a_lo*b_hi,
// where each TF32 x TF32 product is exact in FP32 and only a_lo*b_lo
// (|.| <= 2^-22 |a b|) and the split remainders (|x - x_hi - x_lo| <=
// 2^-22 |x|) are dropped: about 3 * 2^-22 |a b| per product, i.e. within the
// library's FP32 bound 4 K 2^-24 (|alpha| sum|a b| + |beta c|) for K >= 3.
// The tensor cores accumulate in FP32 in TMEM. This path is optional and
// reported separately from the FFMA kernels; the pages measure TF32 only as
// a faster, less accurate mode (Tinyforge README: cuBLAS TF32 7,728 GFLOPS,
// failing the FP32 tolerance) and do not describe a split.
//
// Steps per call (all on the caller's stream):
//   1. split_rows_kernel: A (M x K, lda) -> A_hi, A_lo (M x Kp, Kp = K rounded
//      up to 4), K-major as A already is.
//   2. split_transpose_kernel: B (K x N, ldb) -> B_hi^T, B_lo^T (N x Kp): the
//      MMA takes both operands K-major.
//   3. tf32x3_kernel: persistent, one CTA per SM, 128 x BN output tiles
//      (BN = 128 with a 3-stage ring by default, 256 with 2 stages). By
//      default the CTAs run in clusters of two on neighbouring tiles of one
//      tile row: each TMA-loads one of the row's A_hi / A_lo tiles multicast
//      into both CTAs, and each MMA thread releases a stage in both CTAs, so
//      A comes from L2 once per pair.
//      warp 0: TMA producer (one thread) filling the ring, each stage the
//              128 x 32 A_hi/A_lo and BN x 32 B_hi/B_lo tiles (64 or 96 KB,
//              128-byte swizzle);
//      warp 1: allocates 2 BN TMEM columns (two 128 x BN FP32 accumulators)
//              and one thread issues tcgen05.mma.kind::tf32 (M 128, N BN,
//              K 8): for each 8-wide k-slice, hi*hi, hi*lo and lo*hi into the
//              tile's accumulator; tcgen05.commit releases the stage and, at
//              the end of a tile, hands the accumulator to the epilogue;
//      warps 2-5: the epilogue: tcgen05.ld of their 32 TMEM lanes (rows),
//              C = alpha * acc + beta * C, then release the accumulator.
//   Every wait is bounded; all roles meet at one exit where the MMA thread
//   has waited for its MMAs and warp 1 frees the TMEM.
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "sgemm.h"
#include "sgemm_internal.h"

namespace sg {
namespace tf32x3 {

constexpr int BM = 128, BK = 32;
constexpr int THREADS = 192;
constexpr int A_BYTES = BM * BK * 4;        // 16 KB

// Tile width BN (the MMA's N) and ring depth. Two accumulators of BN TMEM
// columns each, so the epilogue of one tile overlaps the MMAs of the next.
// CL: CTAs per thread-block cluster. With CL = 2 the two CTAs of a cluster
// work on neighbouring tiles of one tile row (columns 2j and 2j + 1) and
// share its A: each loads one of A_hi / A_lo and multicasts it into both
// CTAs' stage, so A is read from L2 once per pair instead of twice.
template <int BN_, int STAGES_, int CL_ = 1>
struct TcCfg {
    static constexpr int BN = BN_, STAGES = STAGES_, CL = CL_;
    static_assert(CL == 1 || CL == 2, "CTAs per cluster");
    static constexpr int B_BYTES = BN * BK * 4;
    static constexpr int STAGE_BYTES = 2 * A_BYTES + 2 * B_BYTES;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + 256;
    static_assert(BN == 128 || BN == 256, "MMA N");
    static_assert(SMEM_BYTES <= 227 * 1024, "ring too large");
    // Instruction descriptor of kind::tf32: D FP32 (bits 4-5 = 1), A and B
    // TF32 (bits 7-9 and 10-12 = 2), both K-major (bits 15, 16 = 0), N >> 3
    // in bits 17-22, M >> 4 in bits 24-28.
    static constexpr uint32_t IDESC = (1u << 4) | (2u << 7) | (2u << 10) |
                                      (static_cast<uint32_t>(BN >> 3) << 17) |
                                      (static_cast<uint32_t>(BM >> 4) << 24);
};

struct Params {
    int M, N, K;
    int tiles_m, tiles_n, k_tiles, group_m;
    int c_vec;
    float* C;
    long long ldc;
    float alpha, beta;
    unsigned long long timeout_ns;
    int* status;
    // CTA-pair kernel only: items [0, full_items) are whole 256 x 256 tiles;
    // the half_items after them cover the remaining tiles as 256 x 128
    // halves (two per tile), so a short last wave takes half as long.
    int full_items, half_items;
};

// ---- tcgen05 helpers ---------------------------------------------------------

// Shared-memory operand descriptor for a K-major tile with the 128-byte
// swizzle: rows of 128 bytes, 8-row (1024-byte) swizzle atoms stacked along
// M/N. Fields: start address >> 4 (bits 0-13), leading byte offset >> 4
// (bits 16-29; not used by swizzled K-major layouts, set to 1), stride byte
// offset >> 4 (bits 32-45: 1024 bytes between 8-row groups), descriptor
// version 1 (bits 46-47), swizzle mode 2 = 128-byte (bits 61-63).
__device__ __forceinline__ uint64_t desc_k_sw128(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>(1u) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t acc) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}"
                 :: "r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}

// The same arrive, on the barrier at offset bar in every CTA of the cluster
// named in mask (bit r: CTA rank r).
__device__ __forceinline__ void mma_commit_mc(uint32_t bar, uint16_t mask) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
                 " [%0], %1;" :: "r"(bar), "h"(mask) : "memory");
}

// 2-D TMA tile load multicast to the same shared-memory offset (dst, and the
// barrier bar that counts the bytes) in every CTA of the cluster named in
// mask. x * 4 bytes is a multiple of 16 (x is a multiple of BK).
__device__ __forceinline__ void tma_load_2d_mc(uint32_t dst, const void* desc, uint32_t bar,
                                               int32_t x, int32_t y, uint16_t mask) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".multicast::cluster [%0], [%1, {%3, %4}], [%2], %5;"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(desc)), "r"(bar), "r"(x), "r"(y), "h"(mask)
        : "memory");
}

// Arrive once on bar when every tcgen05.mma this thread issued has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(bar) : "memory");
}

__device__ __forceinline__ void fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive FP32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
                   "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
                   "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
                   "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ float to_tf32(float x) {
    uint32_t h;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(h) : "f"(x));
    return __uint_as_float(h);
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Params& p, int code) {
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

__device__ __forceinline__ void tile_of(int t, const Params& p, int& tm, int& tn) {
    const int per_group = p.group_m * p.tiles_n;
    const int g = t / per_group;
    const int first = g * p.group_m;
    const int gm = min(p.tiles_m - first, p.group_m);
    const int r = t - g * per_group;
    tm = first + r % gm;
    tn = r / gm;
}

// ---- split pre-passes ---------------------------------------------------------
// The call splits A, then B, then runs the MMA kernel. The B split reads
// only the caller's B and writes its own buffers, so it is launched by
// programmatic stream serialisation and runs alongside the A split (both
// let the next kernel be scheduled as soon as they start); it waits for the
// A split at its very end, so that the MMA kernel, waiting for the B split
// in turn, finds both done. In a kernel launched the ordinary way
// griddep_wait returns at once.

// hi/lo (rows x ldd) <- src (rows x cols, row stride lds), zeros in the
// padding columns [cols, ldd). ldd is a multiple of 4, so every thread writes
// one float4 of each output; it reads a float4 too when `vec` (src 16-byte
// aligned and lds % 4 == 0), else four scalars. blockIdx.y walks rows.
__global__ void split_rows_kernel(const float* __restrict__ src, long long lds, float* __restrict__ hi,
                                  float* __restrict__ lo, long long ldd, int rows, int cols, int vec) {
    griddep_launch_dependents();
    const int quads = static_cast<int>(ldd >> 2);
    for (long long r = blockIdx.y; r < rows; r += gridDim.y) {
        const float* srow = src + r * lds;
        for (int q = blockIdx.x * blockDim.x + threadIdx.x; q < quads; q += blockDim.x * gridDim.x) {
            const int c = 4 * q;
            float4 x;
            if (vec && c + 3 < cols) {
                x = *reinterpret_cast<const float4*>(srow + c);
            } else {
                x.x = c < cols ? srow[c] : 0.0f;
                x.y = c + 1 < cols ? srow[c + 1] : 0.0f;
                x.z = c + 2 < cols ? srow[c + 2] : 0.0f;
                x.w = c + 3 < cols ? srow[c + 3] : 0.0f;
            }
            const float4 h = make_float4(to_tf32(x.x), to_tf32(x.y), to_tf32(x.z), to_tf32(x.w));
            const float4 l = make_float4(to_tf32(x.x - h.x), to_tf32(x.y - h.y), to_tf32(x.z - h.z),
                                         to_tf32(x.w - h.w));
            *reinterpret_cast<float4*>(hi + r * ldd + c) = h;
            *reinterpret_cast<float4*>(lo + r * ldd + c) = l;
        }
    }
    griddep_wait();
}

// hiT/loT (cols x ldd) <- transpose of src (rows x cols, row stride lds):
// hiT[j][k] = split(src[k][j]); zeros for k in [rows, ldd). 64 x 64 tiles
// through shared memory: 16 consecutive threads read one source row as
// float4 (scalars where src is not 16-byte aligned or lds % 4 != 0, and at
// the column edge), then write one hi and one lo row as float4 along k (ldd
// is a multiple of 4). blockIdx.x walks column tiles, blockIdx.y row tiles.
constexpr int kSplitTile = 64;

__global__ void __launch_bounds__(256) split_transpose_kernel(const float* __restrict__ src,
                                                              long long lds,
                                                              float* __restrict__ hiT,
                                                              float* __restrict__ loT,
                                                              long long ldd, int rows, int cols) {
    __shared__ float tile[kSplitTile][kSplitTile + 1];
    griddep_launch_dependents();
    const bool vec = (reinterpret_cast<uintptr_t>(src) % 16 == 0) && (lds % 4 == 0);
    const long long n0 = static_cast<long long>(blockIdx.x) * kSplitTile;
    const long long tiles_k = (ldd + kSplitTile - 1) / kSplitTile;
    const int t = threadIdx.x;
    for (long long tk = blockIdx.y; tk < tiles_k; tk += gridDim.y) {
        const long long k0 = tk * kSplitTile;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int q = t + 256 * j;
            const int kk = q >> 4, nn = (q & 15) * 4;
            const long long k = k0 + kk, n = n0 + nn;
            float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (k < rows) {
                const float* sp = src + k * lds + n;
                if (vec && n + 3 < cols) {
                    v = *reinterpret_cast<const float4*>(sp);
                } else {
                    if (n < cols) v.x = sp[0];
                    if (n + 1 < cols) v.y = sp[1];
                    if (n + 2 < cols) v.z = sp[2];
                    if (n + 3 < cols) v.w = sp[3];
                }
            }
            tile[kk][nn] = v.x;
            tile[kk][nn + 1] = v.y;
            tile[kk][nn + 2] = v.z;
            tile[kk][nn + 3] = v.w;
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int q = t + 256 * j;
            const int nn = q >> 4, kk = (q & 15) * 4;
            const long long n = n0 + nn, k = k0 + kk;
            if (n < cols && k < ldd) {
                float h[4], l[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float x = tile[kk + e][nn];
                    h[e] = to_tf32(x);
                    l[e] = to_tf32(x - h[e]);
                }
                const long long o = n * ldd + k;
                *reinterpret_cast<float4*>(hiT + o) = make_float4(h[0], h[1], h[2], h[3]);
                *reinterpret_cast<float4*>(loT + o) = make_float4(l[0], l[1], l[2], l[3]);
            }
        }
        __syncthreads();
    }
    griddep_wait();
}

// ---- the tensor-core kernel ---------------------------------------------------

template <class T>
__global__ void __launch_bounds__(THREADS, 1)
tf32x3_kernel(const __grid_constant__ CUtensorMap tmAh, const __grid_constant__ CUtensorMap tmAl,
              const __grid_constant__ CUtensorMap tmBh, const __grid_constant__ CUtensorMap tmBl,
              const Params p) {
    constexpr int BN = T::BN, STAGES = T::STAGES, B_BYTES = T::B_BYTES;
    constexpr int STAGE_BYTES = T::STAGE_BYTES, TMEM_COLS = T::TMEM_COLS;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t s0 = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
    // barriers: full[2], empty[2], acc_full[2], acc_empty[2], done; then the TMEM address
    const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * STAGES;
    const uint32_t accf0 = empty0 + 8 * STAGES, acce0 = accf0 + 16, done_bar = acce0 + 16;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            // With CL = 2 a stage is free once both CTAs' MMAs have read
            // it: the multicast A halves land in both.
            mbar_init(empty0 + 8 * s, T::CL);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf0 + 8 * b, 1);
            mbar_init(acce0 + 8 * b, 128);
        }
        mbar_init(done_bar, 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_u32(tmem_slot)), "r"(TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;
    // The peer's multicast copies and commits target this CTA's barriers:
    // both CTAs initialise theirs before either issues one.
    if (T::CL > 1) cluster_sync();

    // Work items: tiles, or with CL = 2 pairs of horizontally adjacent
    // tiles, one per CTA of the cluster (a CTA whose tile lies past the last
    // column loads zeros and writes nothing, but still loads its A half).
    const int rank = T::CL > 1 ? static_cast<int>(cluster_ctarank()) : 0;
    const int first_item = T::CL > 1 ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
    const int item_step = static_cast<int>(gridDim.x) / T::CL;
    Params q = p;
    if (T::CL > 1) q.tiles_n = (p.tiles_n + 1) / 2;
    const int num_tiles = q.tiles_m * q.tiles_n;
    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&tmAh);
            tma_prefetch_desc(&tmAl);
            tma_prefetch_desc(&tmBh);
            tma_prefetch_desc(&tmBl);
            int s = 0;
            uint32_t ph = 0;
            int issued = 0;
            bool ok = true;
            for (int t = first_item; t < num_tiles && ok; t += item_step) {
                int tm, tn;
                tile_of(t, q, tm, tn);
                tn = tn * T::CL + rank;
                for (int kt = 0; kt < p.k_tiles; ++kt) {
                    if (!wait_bar(empty0 + 8 * s, ph ^ 1u, p, STATUS_PRODUCER_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full = full0 + 8 * s;
                    const uint32_t st = s0 + s * STAGE_BYTES;
                    mbar_arrive_expect_tx(full, STAGE_BYTES);
                    if (T::CL > 1) {
                        // Rank 0 brings A_hi, rank 1 A_lo, each into both CTAs.
                        tma_load_2d_mc(st + rank * A_BYTES, rank ? &tmAl : &tmAh, full, kt * BK,
                                       tm * BM, 0x3);
                    } else {
                        tma_load_2d(st, &tmAh, full, kt * BK, tm * BM);
                        tma_load_2d(st + A_BYTES, &tmAl, full, kt * BK, tm * BM);
                    }
                    tma_load_2d(st + 2 * A_BYTES, &tmBh, full, kt * BK, tn * BN);
                    tma_load_2d(st + 2 * A_BYTES + B_BYTES, &tmBl, full, kt * BK, tn * BN);
                    ++issued;
                    if (++s == STAGES) { s = 0; ph ^= 1u; }
                }
            }
            if (!ok) {
                // Let this thread's copies land before the CTA can exit.
                const int n = issued < STAGES ? issued : STAGES;
                int ss = s;
                uint32_t pp = ph;
                for (int i = 0; i < n; ++i) {
                    if (--ss < 0) { ss = STAGES - 1; pp ^= 1u; }
                    wait_bar(full0 + 8 * ss, pp, p, STATUS_DRAIN_TIMEOUT);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int it = 0;
            bool ok = true;
            for (int t = first_item; t < num_tiles && ok; t += item_step, ++it) {
                const int b = it & 1;
                const uint32_t acc_phase = static_cast<uint32_t>((it >> 1) & 1);
                // Wait until the epilogue has emptied this accumulator.
                if (!wait_bar(acce0 + 8 * b, acc_phase ^ 1u, p, STATUS_CONSUMER_TIMEOUT)) break;
                fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(b * BN);
                for (int kt = 0; kt < p.k_tiles; ++kt) {
                    if (!wait_bar(full0 + 8 * s, ph, p, STATUS_CONSUMER_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    fence_after();
                    const uint32_t st = s0 + s * STAGE_BYTES;
                    const uint64_t ah = desc_k_sw128(st), al = desc_k_sw128(st + A_BYTES);
                    const uint64_t bh = desc_k_sw128(st + 2 * A_BYTES);
                    const uint64_t bl = desc_k_sw128(st + 2 * A_BYTES + B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BK / 8; ++kk) {
                        // 8 TF32 = 32 bytes further along the swizzled row.
                        const uint64_t off = static_cast<uint64_t>((kk * 32) >> 4);
                        const uint32_t first = (kt == 0 && kk == 0) ? 0u : 1u;
                        mma_tf32(d, ah + off, bh + off, T::IDESC, first);
                        mma_tf32(d, ah + off, bl + off, T::IDESC, 1u);
                        mma_tf32(d, al + off, bh + off, T::IDESC, 1u);
                    }
                    // Stage free once these finish (in both CTAs with CL = 2).
                    if (T::CL > 1) mma_commit_mc(empty0 + 8 * s, 0x3);
                    else mma_commit(empty0 + 8 * s);
                    if (++s == STAGES) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                mma_commit(accf0 + 8 * b);               // accumulator ready
            }
            // Every MMA this thread issued has finished before TMEM is freed.
            mma_commit(done_bar);
            wait_bar(done_bar, 0, p, STATUS_DRAIN_TIMEOUT);
        }
    } else {
        // Epilogue warpgroup: warp w reads TMEM lanes 32 (w % 4) .. + 31.
        const int wq = warp & 3;
        int it = 0;
        for (int t = first_item; t < num_tiles; t += item_step, ++it) {
            const int b = it & 1;
            const uint32_t acc_phase = static_cast<uint32_t>((it >> 1) & 1);
            if (!wait_bar(accf0 + 8 * b, acc_phase, p, STATUS_CONSUMER_TIMEOUT)) break;
            __syncwarp();          // tcgen05.ld is warp-collective: reconverge first
            fence_after();
            int tm, tn;
            tile_of(t, q, tm, tn);
            tn = tn * T::CL + rank;
            const int m = tm * BM + 32 * wq + lane;
            const bool row_ok = m < p.M;
            float* crow = p.C + static_cast<long long>(row_ok ? m : 0) * p.ldc;
            const bool use_c = p.beta != 0.0f;
            for (int ch = 0; ch < BN / 32; ++ch) {
                float v[32];
                tmem_ld32(tmem + (static_cast<uint32_t>(32 * wq) << 16) +
                              static_cast<uint32_t>(b * BN + ch * 32), v);
                if (!row_ok) continue;
                const int n0 = tn * BN + ch * 32;
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    const int n = n0 + j;
                    float o[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) o[e] = p.alpha * v[j + e];
                    if (p.c_vec && n + 3 < p.N) {
                        float4* cp = reinterpret_cast<float4*>(crow + n);
                        if (use_c) {
                            const float4 c = *cp;
                            o[0] = fmaf(p.beta, c.x, o[0]);
                            o[1] = fmaf(p.beta, c.y, o[1]);
                            o[2] = fmaf(p.beta, c.z, o[2]);
                            o[3] = fmaf(p.beta, c.w, o[3]);
                        }
                        *cp = make_float4(o[0], o[1], o[2], o[3]);
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            if (n + e < p.N) {
                                float out = o[e];
                                if (use_c) out = fmaf(p.beta, crow[n + e], out);
                                crow[n + e] = out;
                            }
                        }
                    }
                }
            }
            fence_before();
            mbar_arrive(acce0 + 8 * b);                 // accumulator may be reused
        }
    }

    // Single exit: every role is done (or gave up after its bounded waits),
    // the MMA thread has seen its MMAs finish; free the TMEM.
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                     :: "r"(tmem), "r"(TMEM_COLS) : "memory");
    }
    // No CTA leaves while its peer may still multicast into its shared
    // memory or arrive on its barriers; every role of both CTAs gets here
    // (all of their waits are bounded).
    if (T::CL > 1) cluster_sync();
}

// ---- CTA pairs on one 256 x 256 tile: tcgen05.mma.cta_group::2 -----------------

// The two CTAs of a cluster of two (ranks 0 and 1, a CTA pair) share one
// 256 x 256 output tile. Each holds in its shared memory the 128 rows of A
// (hi and lo) for its half of the tile's rows and the 128 rows of B^T (hi and
// lo) for its half of the tile's columns; one thread of rank 0 issues
// tcgen05.mma.cta_group::2 (M 256, N 256, K 8), which reads A and B from both
// CTAs at the same shared-memory offsets and leaves rows 0..127 of the
// accumulator in rank 0's TMEM and rows 128..255 in rank 1's. Per stage a CTA
// thus loads 64 KB for 128 x 256 outputs, half what one CTA on a 128 x 128
// tile needs per output, and three stages still fit (192 KB).
//   * both producers (warp 0, one thread) wait on their own "empty" barrier
//     (released by rank 0's MMA commit, multicast to both CTAs) and TMA their
//     four tiles into their own stage, completing the bytes on rank 0's
//     "full" barrier (cp.async.bulk.tensor .cta_group::2), which rank 0's
//     producer armed for both CTAs' bytes;
//   * rank 0's MMA thread (warp 1) waits on "full", issues the MMAs and
//     commits: the stage's "empty" in both CTAs, and at the end of a tile the
//     accumulator's "full" in both CTAs;
//   * both epilogues (warps 2-5) read their 128 TMEM lanes and write their
//     rows of C, then arrive on rank 0's accumulator-"empty" barrier, which
//     counts both CTAs' 256 threads.
// Both CTAs allocate the same 512 TMEM columns (two 256-column accumulators)
// with tcgen05.alloc.cta_group::2 and free them after a cluster barrier that
// follows the last MMA's completion.
namespace pair {
constexpr int TILE = 256;                         // M and N of the pair's tile
constexpr int HALF = 128;                         // rows of A and of B^T per CTA
constexpr int STAGES = 3;
constexpr int B_BYTES = HALF * BK * 4;            // 16 KB
constexpr int STAGE_BYTES = 2 * A_BYTES + 2 * B_BYTES;   // 64 KB
constexpr int TMEM_COLS = 2 * TILE;               // 512: all of a CTA's TMEM
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + 256;
static_assert(SMEM_BYTES <= 227 * 1024, "ring too large");
// kind::tf32, D FP32, A and B TF32 K-major, N = 256 (N >> 3 in bits 17-22),
// M = 256 (M >> 4 in bits 24-28).
constexpr uint32_t IDESC = (1u << 4) | (2u << 7) | (2u << 10) |
                           (static_cast<uint32_t>(TILE >> 3) << 17) |
                           (static_cast<uint32_t>(TILE >> 4) << 24);
// The same with N = 128, for the half tiles (each CTA then holds 64 rows
// of B^T).
constexpr uint32_t IDESC_HALF = (1u << 4) | (2u << 7) | (2u << 10) |
                                (static_cast<uint32_t>((TILE / 2) >> 3) << 17) |
                                (static_cast<uint32_t>(TILE >> 4) << 24);
constexpr int HALF_B_BYTES = (HALF / 2) * BK * 4;        // 8 KB of B^T per CTA
}  // namespace pair

// Item i of the CTA-pair kernel: a whole 256 x 256 tile, or one 256 x 128
// half of a tile; `col` is the first column of C it covers, `width` 256 or
// 128.
__device__ __forceinline__ void pair_item(int i, const Params& q, int& tm, int& col,
                                          int& width) {
    int tn;
    if (i < q.full_items) {
        tile_of(i, q, tm, tn);
        col = tn * pair::TILE;
        width = pair::TILE;
    } else {
        const int h = i - q.full_items;
        tile_of(q.full_items + h / 2, q, tm, tn);
        col = tn * pair::TILE + (h & 1) * (pair::TILE / 2);
        width = pair::TILE / 2;
    }
}

__device__ __forceinline__ void mma_tf32_pair(uint32_t d_tmem, uint64_t a, uint64_t b,
                                              uint32_t idesc, uint32_t acc) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}"
                 :: "r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}

// Arrive once on the barrier at offset bar in each CTA of the pair named in
// mask when every tcgen05.mma this thread issued has completed.
__device__ __forceinline__ void mma_commit_pair_mc(uint32_t bar, uint16_t mask) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster"
                 ".multicast::cluster.b64 [%0], %1;" :: "r"(bar), "h"(mask) : "memory");
}

// The same, on this CTA's barrier only.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(bar) : "memory");
}

// 2-D TMA tile load into this CTA's shared memory at dst whose bytes complete
// on the barrier at cluster address bar, which may be in either CTA of the
// pair. x * 4 bytes is a multiple of 16 (x is a multiple of BK).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void* desc, uint32_t bar,
                                                 int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(desc)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

__global__ void __launch_bounds__(THREADS, 1)
tf32x3_pair_kernel(const __grid_constant__ CUtensorMap tmAh, const __grid_constant__ CUtensorMap tmAl,
                   const __grid_constant__ CUtensorMap tmBh, const __grid_constant__ CUtensorMap tmBl,
                   const __grid_constant__ CUtensorMap tmBh64,
                   const __grid_constant__ CUtensorMap tmBl64, const Params p) {
    using namespace pair;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t s0 = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
    // barriers: full[3], empty[3], acc_full[2], acc_empty[2], done; then the TMEM address
    const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * STAGES;
    const uint32_t accf0 = empty0 + 8 * STAGES, acce0 = accf0 + 16, done_bar = acce0 + 16;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            // "full" (used in rank 0): rank 0's producer arms it for both
            // CTAs' bytes; "empty": rank 0's MMA commit.
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf0 + 8 * b, 1);
            mbar_init(acce0 + 8 * b, 2 * 128);   // both CTAs' epilogue threads (rank 0's)
        }
        mbar_init(done_bar, 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_u32(tmem_slot)), "r"(TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;
    // Both CTAs' barriers exist before the peer completes bytes or arrives on
    // them, or the MMA commits to them.
    cluster_sync();
    // Launched behind the split passes (programmatic stream serialisation):
    // nothing above touched global memory; wait for them here.
    griddep_wait();

    Params q = p;
    q.tiles_m = (p.M + TILE - 1) / TILE;
    q.tiles_n = (p.N + TILE - 1) / TILE;
    const int num_tiles = p.full_items + p.half_items;
    const int first_item = static_cast<int>(cluster_id_x());
    const int item_step = static_cast<int>(gridDim.x) / 2;
    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&tmAh);
            tma_prefetch_desc(&tmAl);
            tma_prefetch_desc(&tmBh);
            tma_prefetch_desc(&tmBl);
            if (p.half_items > 0) {
                tma_prefetch_desc(&tmBh64);
                tma_prefetch_desc(&tmBl64);
            }
            // Rank 0's "full" barriers, as cluster addresses.
            const uint32_t full_r0 = mapa_shared(full0, 0);
            int s = 0;
            uint32_t ph = 0;
            // A producer that gives up has waited the whole time limit for a
            // stage to be released, far longer than any copy it issued
            // before takes to land; the copies are done by then.
            for (int t = first_item; t < num_tiles; t += item_step) {
                int tm, col, width;
                pair_item(t, q, tm, col, width);
                const bool half = width < TILE;
                const int a_row = tm * TILE + static_cast<int>(rank) * HALF;
                // Each CTA holds half of the item's columns of B (as rows of B^T).
                const int b_row = col + static_cast<int>(rank) * (width / 2);
                const uint32_t bytes = 2 * (2 * A_BYTES + 2 * (half ? HALF_B_BYTES : B_BYTES));
                SG_DCHECK(p, tm >= 0 && tm < q.tiles_m && col >= 0 && col < q.tiles_n * TILE);
                const CUtensorMap* mbh = half ? &tmBh64 : &tmBh;
                const CUtensorMap* mbl = half ? &tmBl64 : &tmBl;
                bool ok = true;
                for (int kt = 0; kt < p.k_tiles; ++kt) {
                    if (!wait_bar(empty0 + 8 * s, ph ^ 1u, p, STATUS_PRODUCER_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    if (leader) mbar_arrive_expect_tx(full0 + 8 * s, bytes);
                    const uint32_t st = s0 + s * STAGE_BYTES;
                    const uint32_t bar = full_r0 + 8 * s;
                    tma_load_2d_pair(st, &tmAh, bar, kt * BK, a_row);
                    tma_load_2d_pair(st + A_BYTES, &tmAl, bar, kt * BK, a_row);
                    tma_load_2d_pair(st + 2 * A_BYTES, mbh, bar, kt * BK, b_row);
                    tma_load_2d_pair(st + 2 * A_BYTES + B_BYTES, mbl, bar, kt * BK, b_row);
                    if (++s == STAGES) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
            }
        }
    } else if (warp == 1) {
        if (leader && lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int it = 0;
            bool ok = true;
            for (int t = first_item; t < num_tiles && ok; t += item_step, ++it) {
                const int b = it & 1;
                const uint32_t acc_phase = static_cast<uint32_t>((it >> 1) & 1);
                // Wait until both CTAs' epilogues have emptied this accumulator.
                if (!wait_bar(acce0 + 8 * b, acc_phase ^ 1u, p, STATUS_CONSUMER_TIMEOUT)) break;
                fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(b * TILE);
                const uint32_t idesc = t < p.full_items ? IDESC : IDESC_HALF;
                for (int kt = 0; kt < p.k_tiles; ++kt) {
                    if (!wait_bar(full0 + 8 * s, ph, p, STATUS_CONSUMER_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    fence_after();
                    const uint32_t st = s0 + s * STAGE_BYTES;
                    const uint64_t ah = desc_k_sw128(st), al = desc_k_sw128(st + A_BYTES);
                    const uint64_t bh = desc_k_sw128(st + 2 * A_BYTES);
                    const uint64_t bl = desc_k_sw128(st + 2 * A_BYTES + B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BK / 8; ++kk) {
                        const uint64_t off = static_cast<uint64_t>((kk * 32) >> 4);
                        const uint32_t first = (kt == 0 && kk == 0) ? 0u : 1u;
                        mma_tf32_pair(d, ah + off, bh + off, idesc, first);
                        mma_tf32_pair(d, ah + off, bl + off, idesc, 1u);
                        mma_tf32_pair(d, al + off, bh + off, idesc, 1u);
                    }
                    // The stage is free in both CTAs once these finish.
                    mma_commit_pair_mc(empty0 + 8 * s, 0x3);
                    if (++s == STAGES) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                mma_commit_pair_mc(accf0 + 8 * b, 0x3);   // accumulator ready in both
            }
            // Every MMA issued has finished before the TMEM is freed.
            mma_commit_pair(done_bar);
            wait_bar(done_bar, 0, p, STATUS_DRAIN_TIMEOUT);
        }
    } else {
        // Epilogue warpgroup: warp w reads TMEM lanes 32 (w % 4) .. + 31, which
        // hold rows 128 rank + 32 (w % 4) .. of the pair's tile.
        const int wq = warp & 3;
        const uint32_t acce_r0 = mapa_shared(acce0, 0);
        int it = 0;
        for (int t = first_item; t < num_tiles; t += item_step, ++it) {
            const int b = it & 1;
            const uint32_t acc_phase = static_cast<uint32_t>((it >> 1) & 1);
            if (!wait_bar(accf0 + 8 * b, acc_phase, p, STATUS_CONSUMER_TIMEOUT)) break;
            __syncwarp();          // tcgen05.ld is warp-collective: reconverge first
            fence_after();
            int tm, col, width;
            pair_item(t, q, tm, col, width);
            const int m = tm * TILE + static_cast<int>(rank) * HALF + 32 * wq + lane;
            const bool row_ok = m < p.M;
            float* crow = p.C + static_cast<long long>(row_ok ? m : 0) * p.ldc;
            const bool use_c = p.beta != 0.0f;
            SG_DCHECK(p, b * TILE + width <= TMEM_COLS && (width == TILE || width == TILE / 2));
            for (int ch = 0; ch < width / 32; ++ch) {
                float v[32];
                tmem_ld32(tmem + (static_cast<uint32_t>(32 * wq) << 16) +
                              static_cast<uint32_t>(b * TILE + ch * 32), v);
                if (!row_ok) continue;
                const int n0 = col + ch * 32;
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    const int n = n0 + j;
                    float o[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) o[e] = p.alpha * v[j + e];
                    if (p.c_vec && n + 3 < p.N) {
                        float4* cp = reinterpret_cast<float4*>(crow + n);
                        if (use_c) {
                            const float4 c = *cp;
                            o[0] = fmaf(p.beta, c.x, o[0]);
                            o[1] = fmaf(p.beta, c.y, o[1]);
                            o[2] = fmaf(p.beta, c.z, o[2]);
                            o[3] = fmaf(p.beta, c.w, o[3]);
                        }
                        *cp = make_float4(o[0], o[1], o[2], o[3]);
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            if (n + e < p.N) {
                                float out = o[e];
                                if (use_c) out = fmaf(p.beta, crow[n + e], out);
                                crow[n + e] = out;
                            }
                        }
                    }
                }
            }
            fence_before();
            // This accumulator may be reused once both CTAs' threads arrive.
            if (leader) mbar_arrive(acce0 + 8 * b);
            else mbar_arrive_remote(acce_r0 + 8 * b);
        }
    }

    // Single exit: every role is done (or gave up after its bounded waits);
    // rank 0's MMA thread has seen its last MMA finish before it got here, and
    // the cluster barrier makes the peer wait for that too before the TMEM of
    // both CTAs is freed; no CTA leaves while its peer may still arrive on its
    // barriers.
    fence_before();
    __syncthreads();
    cluster_sync();
    fence_after();
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;"
                     :: "r"(tmem), "r"(TMEM_COLS) : "memory");
    }
    cluster_sync();
}

// ---- the TF32 tensor-core ceiling -----------------------------------------------

// One CTA per SM (its shared memory keeps a second one off the SM). One
// thread issues `iters` x 4 back-to-back tcgen05.mma.kind::tf32 (M 128, N BN,
// K 8; the instruction shape and descriptors of tf32x3_kernel) on a 128 x 32
// A tile and a BN x 32 B tile of zeros resident in shared memory, all into
// one TMEM accumulator, then commits and waits (bounded) for them before the
// TMEM is freed. Nothing is read from or written to global memory except
// the status word on a time-out: the rate is the tensor pipe's alone.
constexpr int kPeakSmem = 160 * 1024;

template <int BN>
__global__ void __launch_bounds__(128, 1) tf32_mma_peak_kernel(long long iters, Params p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    constexpr int TILE_BYTES = A_BYTES + BN * BK * 4;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + TILE_BYTES);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);
    const int warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < TILE_BYTES / 16; i += blockDim.x)
        reinterpret_cast<float4*>(smem)[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(bar), 1);
        fence_barrier_init();
    }
    // The zeros written by the threads above must be visible to the tensor
    // core's (async-proxy) reads of the operands.
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_u32(tmem_slot)), "r"(BN) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;
    if (threadIdx.x == 0) {
        constexpr uint32_t IDESC = (1u << 4) | (2u << 7) | (2u << 10) |
                                   (static_cast<uint32_t>(BN >> 3) << 17) |
                                   (static_cast<uint32_t>(BM >> 4) << 24);
        const uint32_t s0 = smem_u32(smem);
        const uint64_t a = desc_k_sw128(s0), b = desc_k_sw128(s0 + A_BYTES);
        for (long long it = 0; it < iters; ++it) {
#pragma unroll
            for (int kk = 0; kk < BK / 8; ++kk) {
                const uint64_t off = static_cast<uint64_t>((kk * 32) >> 4);
                mma_tf32(tmem, a + off, b + off, IDESC, (it == 0 && kk == 0) ? 0u : 1u);
            }
        }
        mma_commit(smem_u32(bar));
        wait_bar(smem_u32(bar), 0, p, STATUS_DRAIN_TIMEOUT);
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 0) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                     :: "r"(tmem), "r"(BN) : "memory");
    }
}

bool encode(CUtensorMap* map, const float* base, int64_t rows, int64_t cols, int64_t ld, int box_rows,
            PFN_cuTensorMapEncodeTiled_v12000 enc) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 4};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Kernel variant. By default CTA pairs on 256 x 256 tiles (tcgen05
// cta_group::2) when those tiles fill every pair the GPU runs at once, else
// clusters of two CTAs that share A by multicast (128 x 128 tiles, 3 stages)
// wherever a tile row holds two tiles, else one CTA per tile. The
// environment variable SGEMM_3XTF32_TILE forces one:
// "128x128c2", "128x128" (one CTA per tile), "128x256" (2 stages) or
// "256x256" (CTA pairs on one tile, tcgen05.mma.cta_group::2).
// Measured on GB300 (clusters against single CTAs, same box, interleaved):
// 4096^3 0.571 against 0.581 ms, 8192x14336x4096 3.52 against 3.58 ms,
// 4093x5120x1531 0.322 against 0.380 ms, 2048^3 even.
enum { VARIANT_AUTO = 0, VARIANT_WIDE = 1, VARIANT_PAIR = 2, VARIANT_SINGLE = 3, VARIANT_MMA2 = 4 };

int tile_variant(const DeviceInfo*) {
    static const int v = [] {
        const char* env = std::getenv("SGEMM_3XTF32_TILE");
        if (env == nullptr) return static_cast<int>(VARIANT_AUTO);
        if (std::strcmp(env, "128x256") == 0) return static_cast<int>(VARIANT_WIDE);
        if (std::strcmp(env, "128x128c2") == 0) return static_cast<int>(VARIANT_PAIR);
        if (std::strcmp(env, "128x128") == 0) return static_cast<int>(VARIANT_SINGLE);
        if (std::strcmp(env, "256x256") == 0) return static_cast<int>(VARIANT_MMA2);
        return static_cast<int>(VARIANT_AUTO);
    }();
    return v;
}

template <class T>
cudaError_t launch(const DeviceInfo* dev, const float* a_hi, const float* a_lo, const float* b_hi,
                   const float* b_lo, int64_t kp, Params p, cudaStream_t stream) {
    // Once per device (device_info admits indexes below 64). Host threads
    // that race here both set the same attribute, which is harmless; the
    // flag itself is atomic.
    static std::atomic<bool> attr_set[64] = {};
    if (!attr_set[dev->device].load(std::memory_order_acquire)) {
        const cudaError_t e = cudaFuncSetAttribute(tf32x3_kernel<T>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   T::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set[dev->device].store(true, std::memory_order_release);
    }
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    CUtensorMap mah, mal, mbh, mbl;
    if (!(encode(&mah, a_hi, p.M, p.K, kp, BM, enc) && encode(&mal, a_lo, p.M, p.K, kp, BM, enc) &&
          encode(&mbh, b_hi, p.N, p.K, kp, T::BN, enc) && encode(&mbl, b_lo, p.N, p.K, kp, T::BN, enc)))
        return cudaErrorInvalidValue;
    p.tiles_n = (p.N + T::BN - 1) / T::BN;
    if (T::CL == 1) {
        const int64_t tiles = static_cast<int64_t>(p.tiles_m) * p.tiles_n;
        const int grid = static_cast<int>(tiles < dev->sm_count ? tiles : dev->sm_count);
        tf32x3_kernel<T><<<grid, THREADS, T::SMEM_BYTES, stream>>>(mah, mal, mbh, mbl, p);
        return cudaGetLastError();
    }
    // Clusters of T::CL CTAs, as many as the GPU runs at once (a cluster
    // sits whole in one GPC), each a persistent worker over tile pairs.
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = T::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = T::CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    static std::atomic<int> max_clusters[64] = {};
    int ncl = max_clusters[dev->device].load(std::memory_order_relaxed);
    if (ncl <= 0) {
        cfg.gridDim = dim3(T::CL);
        const cudaError_t e = cudaOccupancyMaxActiveClusters(&ncl, tf32x3_kernel<T>, &cfg);
        if (e != cudaSuccess) return e;
        if (ncl <= 0) return cudaErrorInvalidConfiguration;
        max_clusters[dev->device].store(ncl, std::memory_order_relaxed);
    }
    const int64_t items = static_cast<int64_t>(p.tiles_m) * ((p.tiles_n + T::CL - 1) / T::CL);
    const int clusters = static_cast<int>(items < ncl ? items : ncl);
    cfg.gridDim = dim3(static_cast<unsigned>(clusters * T::CL));
    return cudaLaunchKernelEx(&cfg, tf32x3_kernel<T>, mah, mal, mbh, mbl, p);
}

// How many clusters of the CTA-pair kernel the device runs at once (a
// cluster sits whole in one GPC), queried once per device; 0 if none fits.
int pair_clusters(const DeviceInfo* dev) {
    static std::atomic<int> max_clusters[64] = {};
    int ncl = max_clusters[dev->device].load(std::memory_order_acquire);
    if (ncl != 0) return ncl < 0 ? 0 : ncl;
    ncl = -1;
    if (cudaFuncSetAttribute(tf32x3_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             pair::SMEM_BYTES) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.blockDim = dim3(THREADS);
        cfg.dynamicSmemBytes = pair::SMEM_BYTES;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cfg.gridDim = dim3(2);
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, tf32x3_pair_kernel, &cfg) == cudaSuccess && n > 0)
            ncl = n;
    }
    (void)cudaGetLastError();
    max_clusters[dev->device].store(ncl, std::memory_order_release);
    return ncl < 0 ? 0 : ncl;
}

// The CTA-pair kernel on 256 x 256 tiles (tcgen05.mma.cta_group::2).
cudaError_t launch_pair(const DeviceInfo* dev, const float* a_hi, const float* a_lo,
                        const float* b_hi, const float* b_lo, int64_t kp, Params p,
                        cudaStream_t stream) {
    const int ncl = pair_clusters(dev);
    if (ncl <= 0) return cudaErrorInvalidConfiguration;
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    CUtensorMap mah, mal, mbh, mbl, mbh64, mbl64;
    // Boxes of BK x 128 rows: each CTA loads its half of the tile's rows of
    // A and of B^T; boxes of 64 rows of B^T for the half tiles.
    if (!(encode(&mah, a_hi, p.M, p.K, kp, pair::HALF, enc) &&
          encode(&mal, a_lo, p.M, p.K, kp, pair::HALF, enc) &&
          encode(&mbh, b_hi, p.N, p.K, kp, pair::HALF, enc) &&
          encode(&mbl, b_lo, p.N, p.K, kp, pair::HALF, enc) &&
          encode(&mbh64, b_hi, p.N, p.K, kp, pair::HALF / 2, enc) &&
          encode(&mbl64, b_lo, p.N, p.K, kp, pair::HALF / 2, enc)))
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = pair::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (pdl_enabled()) {
        // Scheduled while the split passes finish; it waits for them on the
        // device before its first global-memory access.
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 2;
    }
    const int64_t tiles = ((p.M + pair::TILE - 1) / pair::TILE) *
                          static_cast<int64_t>((p.N + pair::TILE - 1) / pair::TILE);
    if (tiles > 0x3fffffffll) return cudaErrorInvalidValue;
    // A last wave that is at most half full is run as half tiles: the pairs
    // then take half as long over it (4096^3: 256 tiles on 76 pairs, 3.5
    // waves of work instead of 4).
    const int64_t rest = tiles % ncl;
    const bool split = tiles > ncl && rest > 0 && 2 * rest <= ncl;
    p.full_items = static_cast<int>(split ? tiles - rest : tiles);
    p.half_items = static_cast<int>(split ? 2 * rest : 0);
    const int64_t items = static_cast<int64_t>(p.full_items) + p.half_items;
    const int clusters = static_cast<int>(items < ncl ? items : ncl);
    cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters));
    return cudaLaunchKernelEx(&cfg, tf32x3_pair_kernel, mah, mal, mbh, mbl, mbh64, mbl64, p);
}

}  // namespace tf32x3
}  // namespace sg

using namespace sg;

namespace {

int run_3xtf32(int opa, int opb, int64_t M, int64_t N, int64_t K, float alpha, const float* A,
               int64_t lda, const float* B, int64_t ldb, float beta, float* C, int64_t ldc,
               cudaStream_t stream) {
    int rc = check_args_ex(opa, opb, M, N, K, alpha, A, lda, B, ldb, C, ldc);
    if (rc != SGEMM_OK) return rc;
    if (M == 0 || N == 0) return SGEMM_OK;
    // Short reductions (the dropped lo*lo terms are not covered by the bound
    // below K = 3), alpha == 0 and K == 0 go to the FFMA path.
    if (K < 16 || alpha == 0.0f)
        return sgemm_ex(opa, opb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
    const DeviceInfo* dev = nullptr;
    if ((rc = device_info(&dev)) != SGEMM_OK) return rc;
    int* status = nullptr;
    cudaMemPool_t pool = nullptr;
    if ((rc = device_memory_handles(dev, &status, &pool)) != SGEMM_OK) return rc;
    using namespace tf32x3;
    const int64_t kp = (K + 3) & ~int64_t{3};
    const size_t a_bytes = static_cast<size_t>(M) * static_cast<size_t>(kp) * 4;
    const size_t b_bytes = static_cast<size_t>(N) * static_cast<size_t>(kp) * 4;
    const size_t a_pad = (a_bytes + 255) & ~size_t{255}, b_pad = (b_bytes + 255) & ~size_t{255};
    void* w = nullptr;
    if (cudaMallocFromPoolAsync(&w, 2 * a_pad + 2 * b_pad, pool, stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return sgemm_ex(opa, opb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
    }
    unsigned char* ws = static_cast<unsigned char*>(w);
    float* a_hi = reinterpret_cast<float*>(ws);
    float* a_lo = reinterpret_cast<float*>(ws + a_pad);
    float* b_hi = reinterpret_cast<float*>(ws + 2 * a_pad);
    float* b_lo = reinterpret_cast<float*>(ws + 2 * a_pad + b_pad);
    // Each split writes a K-major (rows x kp) hi/lo pair: a row-wise split
    // of an operand already stored K-major (A, or a transposed B), a
    // transposing split otherwise (B, or a transposed A).
    // The A split is launched the ordinary way (after whatever the caller
    // queued before), the B split alongside it (programmatic stream
    // serialisation, see the split kernels).
    auto split_kmajor = [&](const float* X, int64_t ldx, float* hi, float* lo, int64_t rows,
                            bool pdl) {
        const int vec = ((reinterpret_cast<uintptr_t>(X) % 16) == 0 && (ldx % 4) == 0) ? 1 : 0;
        const int64_t quads = kp / 4;
        const int gx = static_cast<int>(quads < 256 * 8 ? (quads + 255) / 256 : 8);
        const int gy = static_cast<int>(rows < 8192 ? rows : 8192);
        return launch_kernel(split_rows_kernel, dim3(gx, gy), dim3(256), 0, stream, pdl, 1, X,
                             static_cast<long long>(ldx), hi, lo, static_cast<long long>(kp),
                             static_cast<int>(rows), static_cast<int>(K), vec);
    };
    auto split_transposed = [&](const float* X, int64_t ldx, float* hi, float* lo, int64_t cols,
                                bool pdl) {
        const int64_t tiles_k = (kp + kSplitTile - 1) / kSplitTile;
        const dim3 grid(static_cast<unsigned>((cols + kSplitTile - 1) / kSplitTile),
                        static_cast<unsigned>(tiles_k < 65535 ? tiles_k : 65535));
        return launch_kernel(split_transpose_kernel, grid, dim3(256), 0, stream, pdl, 1, X,
                             static_cast<long long>(ldx), hi, lo, static_cast<long long>(kp),
                             static_cast<int>(K), static_cast<int>(cols));
    };
    const bool pdl = pdl_enabled();
    cudaError_t e = opa ? split_transposed(A, lda, a_hi, a_lo, M, false)
                        : split_kmajor(A, lda, a_hi, a_lo, M, false);
    if (e == cudaSuccess)
        e = opb ? split_kmajor(B, ldb, b_hi, b_lo, N, pdl) : split_transposed(B, ldb, b_hi, b_lo, N, pdl);
    if (e == cudaSuccess) {
        Params p;
        std::memset(&p, 0, sizeof(p));
        p.M = static_cast<int>(M);
        p.N = static_cast<int>(N);
        p.K = static_cast<int>(K);
        p.tiles_m = static_cast<int>((M + BM - 1) / BM);
        p.k_tiles = static_cast<int>((K + BK - 1) / BK);
        // Tiles walk 16 tile-rows at a time: at 4096^3 0.552 ms against
        // 0.556 ms with 8 and 0.561 / 0.562 ms with 4 / 32 (GB300).
        p.group_m = 16;
        p.c_vec = ((reinterpret_cast<uintptr_t>(C) % 16) == 0 && (ldc % 4) == 0) ? 1 : 0;
        p.C = C;
        p.ldc = ldc;
        p.alpha = alpha;
        p.beta = beta;
        p.timeout_ns = wait_timeout_ns();
        p.status = status;
        int v = tile_variant(dev);
        if (v == VARIANT_AUTO) {
            // 256 x 256 tiles on CTA pairs (tcgen05.mma.cta_group::2) once
            // they fill every pair the GPU runs at once; below that the
            // 128 x 128 tiles keep more SMs busy (1024^3: 16 such tiles,
            // 49.9 against 37.8 us). Measured on GB300: 4096^3 0.511 against
            // 0.566 ms, 8192 x 14336 x 4096 2.84 against 3.53 ms, 4093 x 5120
            // x 1531 0.279 against 0.314 ms, the same bits.
            const int64_t tiles256 = ((M + pair::TILE - 1) / pair::TILE) *
                                     ((N + pair::TILE - 1) / pair::TILE);
            const int ncl = pair_clusters(dev);
            if (ncl > 0 && tiles256 >= ncl) v = VARIANT_MMA2;
            else v = N > 128 ? VARIANT_PAIR : VARIANT_SINGLE;
        }
        switch (v) {
            case VARIANT_WIDE:
                e = launch<TcCfg<256, 2>>(dev, a_hi, a_lo, b_hi, b_lo, kp, p, stream);
                break;
            case VARIANT_PAIR:
                e = launch<TcCfg<128, 3, 2>>(dev, a_hi, a_lo, b_hi, b_lo, kp, p, stream);
                break;
            case VARIANT_MMA2:
                e = launch_pair(dev, a_hi, a_lo, b_hi, b_lo, kp, p, stream);
                break;
            default:
                e = launch<TcCfg<128, 3>>(dev, a_hi, a_lo, b_hi, b_lo, kp, p, stream);
                break;
        }
    }
    cudaFreeAsync(w, stream);
    if (e != cudaSuccess) return cuda_fail(e, SGEMM_ERR_LAUNCH);
    return SGEMM_OK;
}

}  // namespace

extern "C" int sgemm_3xtf32(int64_t M, int64_t N, int64_t K, float alpha, const float* A,
                            int64_t lda, const float* B, int64_t ldb, float beta, float* C,
                            int64_t ldc, cudaStream_t stream) {
    return run_3xtf32(0, 0, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
}

extern "C" int sgemm_3xtf32_ex(int opa, int opb, int64_t M, int64_t N, int64_t K, float alpha,
                               const float* A, int64_t lda, const float* B, int64_t ldb,
                               float beta, float* C, int64_t ldc, cudaStream_t stream) {
    return run_3xtf32(opa, opb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
}

extern "C" int sgemm_tf32_mma_peak(int n, double target_ms, double* tflops, double* ms,
                                   double* flops, cudaStream_t stream) {
    using namespace sg::tf32x3;
    if (n != 128 && n != 256) return SGEMM_ERR_INVALID_VALUE;
    if (!(target_ms >= 1.0) || target_ms > 60000.0) return SGEMM_ERR_INVALID_VALUE;
    const DeviceInfo* dev = nullptr;
    int rc = device_info(&dev);
    if (rc != SGEMM_OK) return rc;
    int* status = nullptr;
    cudaMemPool_t pool = nullptr;
    if ((rc = device_memory_handles(dev, &status, &pool)) != SGEMM_OK) return rc;
    auto kernel = n == 256 ? &tf32_mma_peak_kernel<256> : &tf32_mma_peak_kernel<128>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kPeakSmem);
    if (e != cudaSuccess) return cuda_fail(e, SGEMM_ERR_CUDA);
    Params p;
    std::memset(&p, 0, sizeof(p));
    p.status = status;
    // A run is calibrated below 60 s; its single wait is allowed twice that.
    p.timeout_ns = 120000000000ull;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if ((e = cudaEventCreate(&e0)) != cudaSuccess || (e = cudaEventCreate(&e1)) != cudaSuccess) {
        if (e0) cudaEventDestroy(e0);
        return cuda_fail(e, SGEMM_ERR_CUDA);
    }
    const int grid = dev->sm_count;
    auto run = [&](long long iters, float* out_ms) -> cudaError_t {
        cudaError_t err = cudaEventRecord(e0, stream);
        if (err != cudaSuccess) return err;
        kernel<<<grid, 128, kPeakSmem, stream>>>(iters, p);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
        if ((err = cudaEventRecord(e1, stream)) != cudaSuccess) return err;
        if ((err = cudaEventSynchronize(e1)) != cudaSuccess) return err;
        return cudaEventElapsedTime(out_ms, e0, e1);
    };
    float t = 0.0f;
    long long iters = 1024;
    int result = SGEMM_OK;
    // Calibrate: grow until a launch takes >= 5 ms, then scale to the target.
    for (;;) {
        if ((e = run(iters, &t)) != cudaSuccess) { result = SGEMM_ERR_LAUNCH; break; }
        if (t >= 5.0f || iters > (1ll << 36)) break;
        iters *= 4;
    }
    if (result == SGEMM_OK) {
        long long want = static_cast<long long>(static_cast<double>(iters) * target_ms / t);
        if (want < 1) want = 1;
        // Warm-up of the same length, then the timed launch.
        if ((e = run(want, &t)) != cudaSuccess || (e = run(want, &t)) != cudaSuccess) {
            result = SGEMM_ERR_LAUNCH;
        } else {
            // 2 M N K FLOP per MMA (M 128, K 8), 4 MMAs per iteration.
            const double f = 2.0 * BM * n * 8.0 * 4.0 * static_cast<double>(want) * grid;
            if (tflops) *tflops = f / (static_cast<double>(t) * 1e-3) / 1e12;
            if (ms) *ms = t;
            if (flops) *flops = f;
        }
    }
    if (result != SGEMM_OK) cuda_fail(e, result);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    return result;
}
