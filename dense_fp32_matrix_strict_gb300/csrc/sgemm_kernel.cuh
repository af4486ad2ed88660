// sgemm_kernel.cuh — the warp-specialised strict-FP32 SGEMM kernel for sm_103a.
//
// C = alpha * A * B + beta * C, row-major A (M x K, lda), B (K x N, ldb),
// C (M x N, ldc); every multiply-add is one FFMA on the FP32 CUDA cores.
//
// Structure (one persistent CTA per SM, static tile schedule):
//   * producer warp(s) fill an S-deep ring of shared-memory stages, each a
//     BM x BK tile of A and a BK x BN tile of B. An operand whose base and
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
// The pages this follows ("The road to a fast GEMM": sections "v4:
// two-dimensional register tiling", "v5: vectorized loads", "Where to go
// next" on double buffering, multi-stage pipelines and warp tiling; the
// Tinyforge README on BK = 16 + padding and XOR swizzling; the T4 article's
// "Tiling" section on zero-filled tails) use __syncthreads double buffering
// on sm_75..sm_89. Here the ring is deeper, the barriers are mbarriers, the
// loads are TMA where the strides allow it, and A stays row-major in shared
// memory with the 128-byte TMA swizzle instead of a transposing store: each
// lane reads float4 runs along k for its 8 rows, which costs the same number
// of shared loads per FFMA as a transposed copy.
//
// Every mbarrier wait is bounded (globaltimer): on timeout the thread sets a
// bit in the device status word, lets its own copies in flight land (again
// bounded) and returns. Nothing spins forever.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "ptx.cuh"

namespace sg {

enum LoadMode : int { LOAD_TMA = 0, LOAD_CPASYNC = 1 };

// Status bits written by the kernel when a bounded wait gives up.
enum : int {
    STATUS_CONSUMER_TIMEOUT = 1,
    STATUS_PRODUCER_TIMEOUT = 2,
    STATUS_DRAIN_TIMEOUT = 4,
};

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
};

// Kernel configuration. LMAP: lane mapping (lane_grid); XPF: prefetch the
// next stage's first fragments during the current stage's last k-group;
// FORDER: FMA form of the outer product (0: scalar FFMA rows outer, 1: scalar
// columns outer, 2: packed FFMA2 over column pairs).
// ISSUE: 0 = dedicated producer warp(s); 1 = when both operands load by TMA,
// consumer thread 0 issues the refills itself (no producer warp, so 256
// threads and up to 255 registers per thread).
template <int BM_, int BN_, int BK_, int STAGES_, int A_MODE_, int B_MODE_, int LMAP_ = 0,
          int XPF_ = 0, int FORDER_ = 0, int ISSUE_ = 0>
struct Cfg {
    static constexpr int BM = BM_, BN = BN_, BK = BK_, STAGES = STAGES_;
    static constexpr int A_MODE = A_MODE_, B_MODE = B_MODE_;
    static constexpr int LMAP = LMAP_, XPF = XPF_, FORDER = FORDER_;
    static constexpr bool INLINE =
        (ISSUE_ == 1) && (A_MODE_ == LOAD_TMA) && (B_MODE_ == LOAD_TMA);
    static_assert(BK == 32, "A rows are one 128-byte swizzle span");
    static_assert(BM % 32 == 0 && BN % 64 == 0, "warp tile is 32 x 64");
    static constexpr int WARPS_M = BM / 32, WARPS_N = BN / 64;
    static constexpr int CONSUMER_WARPS = WARPS_M * WARPS_N;
    static constexpr int CONSUMERS = CONSUMER_WARPS * 32;
    static constexpr bool ANY_CP = (A_MODE == LOAD_CPASYNC) || (B_MODE == LOAD_CPASYNC);
    static constexpr bool ANY_TMA = (A_MODE == LOAD_TMA) || (B_MODE == LOAD_TMA);
    // cp.async producers: one warp per SM sub-partition so the copy
    // instructions do not all land on one scheduler.
    static constexpr int PRODUCER_WARPS = INLINE ? 0 : (ANY_CP ? 4 : 1);
    static constexpr int THREADS = CONSUMERS + 32 * PRODUCER_WARPS;
    static constexpr int A_BYTES = BM * BK * 4;
    static constexpr int B_BYTES = BK * BN * 4;
    static constexpr uint32_t TX_BYTES =
        (A_MODE == LOAD_TMA ? A_BYTES : 0) + (B_MODE == LOAD_TMA ? B_BYTES : 0);
    static constexpr uint32_t FULL_COUNT = (ANY_TMA ? 1 : 0) + (ANY_CP ? 32 * PRODUCER_WARPS : 0);
    static constexpr int SMEM_BYTES = 1024 /* alignment slack */ + STAGES * (A_BYTES + B_BYTES)
                                      + 2 * STAGES * 8;
    static_assert(SMEM_BYTES <= 227 * 1024, "ring does not fit in 227 KB of shared memory");
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

// Byte offset of A element (row r, column k) inside one stage: 128-byte rows,
// 16-byte chunk index XOR (r mod 8) — the TMA 128B swizzle pattern.
__device__ __forceinline__ uint32_t a_swz(int r, int k) {
    return static_cast<uint32_t>(r * 128 + ((((k >> 2) ^ r) & 7) << 4) + ((k & 3) << 2));
}

template <class C>
__device__ __forceinline__ void producer(const CUtensorMap* tmA, const CUtensorMap* tmB,
                                         const GemmParams& p, uint32_t sA, uint32_t sB,
                                         uint32_t full0, uint32_t empty0, int pw, int lane) {
    const int num_tiles = p.tiles_m * p.tiles_n;
    const bool tma_thread = C::ANY_TMA && pw == 0 && lane == 0;
    if (!C::ANY_CP && !tma_thread) return;
    if (tma_thread) {
        if (C::A_MODE == LOAD_TMA) tma_prefetch_desc(tmA);
        if (C::B_MODE == LOAD_TMA) tma_prefetch_desc(tmB);
    }
    int s = 0;
    uint32_t ph = 0;
    int issued = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
        int tm, tn;
        tile_coords(t, p, tm, tn);
        const int m0 = tm * C::BM, n0 = tn * C::BN;
        for (int kt = 0; kt < p.k_tiles; ++kt) {
            if (!wait_bounded(empty0 + 8 * s, ph ^ 1u, p, STATUS_PRODUCER_TIMEOUT)) {
                ok = false;
                break;
            }
            const uint32_t full = full0 + 8 * s;
            const uint32_t dA = sA + s * C::A_BYTES, dB = sB + s * C::B_BYTES;
            const int k0 = kt * C::BK;
            if (tma_thread) {
                mbar_arrive_expect_tx(full, C::TX_BYTES);
                if (C::A_MODE == LOAD_TMA) tma_load_2d(dA, tmA, full, k0, m0);
                if (C::B_MODE == LOAD_TMA) tma_load_2d(dB, tmB, full, n0, k0);
            }
            if (C::A_MODE == LOAD_CPASYNC) {
                // One row of BK = 32 floats per warp instruction, lane = k.
                const int k = k0 + lane;
                for (int r = pw; r < C::BM; r += C::PRODUCER_WARPS) {
                    const int m = m0 + r;
                    const bool v = (m < p.M) && (k < p.K);
                    const float* src = v ? p.A + (long long)m * p.lda + k : p.A;
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
                        cp_async_4(dB + (kr * C::BN + nn) * 4, src, v);
                    }
                }
            }
            if (C::ANY_CP) cp_async_mbar_arrive_noinc(full);
            ++issued;
            if (++s == C::STAGES) { s = 0; ph ^= 1u; }
        }
    }
    if (!ok) {
        // Let the copies this thread started land before the CTA can exit:
        // wait (bounded) for the last phase of each stage it filled.
        const int n = issued < C::STAGES ? issued : C::STAGES;
        int ss = s;
        uint32_t pp = ph;
        for (int i = 0; i < n; ++i) {
            if (--ss < 0) { ss = C::STAGES - 1; pp ^= 1u; }
            wait_bounded(full0 + 8 * ss, pp, p, STATUS_DRAIN_TIMEOUT);
        }
    }
    if (C::ANY_CP) asm volatile("cp.async.wait_all;" ::: "memory");
}

// Lane -> (tr, tc) in the 4 x 8 lane grid of a 32 x 64 warp tile. The
// mapping decides which lanes share a shared-memory quarter-warp phase:
//   0: tr = lane / 8, tc = lane % 8   (a phase reads 1 A row, 8 B float4)
//   1: tr = lane % 4, tc = lane / 4   (a phase reads 4 A rows, 2 B float4)
//   2: 2 x 4 blocks per phase          (a phase reads 2 A rows, 4 B float4)
template <int LMAP>
__device__ __forceinline__ void lane_grid(int lane, int& tr, int& tc) {
    if (LMAP == 0) {
        tr = lane >> 3;
        tc = lane & 7;
    } else if (LMAP == 1) {
        tr = lane & 3;
        tc = lane >> 2;
    } else {
        tr = (lane & 1) | (((lane >> 3) & 1) << 1);
        tc = ((lane >> 1) & 3) | ((lane >> 4) << 2);
    }
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

// One k-step of the 8 x 8 register outer product.
//   FORDER 0/1: scalar FFMA, rows or columns outer.
//   FORDER 2:   packed FFMA2 (fma.rn.f32x2: two IEEE single-precision FMAs,
//               each rounded once, in one instruction): pairs of adjacent
//               columns share one instruction with the row's A value in both
//               lanes. Every output still sees the same FMA sequence, so the
//               result is bit-identical to the scalar forms.
template <int FORDER>
__device__ __forceinline__ void outer_product(float (&acc)[8][8], const float4 (&a)[8], int kk,
                                              const float4& b0, const float4& b1) {
    const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
    if (FORDER == 2) {
        const float2 bp[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w),
                              make_float2(b1.x, b1.y), make_float2(b1.z, b1.w)};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float av = lane_of(a[i], kk);
            const float2 aa = make_float2(av, av);
#pragma unroll
            for (int jp = 0; jp < 4; ++jp) {
                float2 c = make_float2(acc[i][2 * jp], acc[i][2 * jp + 1]);
                c = __ffma2_rn(aa, bp[jp], c);
                acc[i][2 * jp] = c.x;
                acc[i][2 * jp + 1] = c.y;
            }
        }
    } else if (FORDER == 0) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float av = lane_of(a[i], kk);
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av, bv[j], acc[i][j]);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i][j] = fmaf(lane_of(a[i], kk), bv[j], acc[i][j]);
    }
}

// Inline refill (Cfg::INLINE): load stage g of this CTA's sequence into ring
// slot `slot` by TMA, completing on that slot's full barrier.
template <class C>
__device__ __forceinline__ void issue_stage(const CUtensorMap* tmA, const CUtensorMap* tmB,
                                            const GemmParams& p, uint32_t sA, uint32_t sB,
                                            uint32_t full0, int g, int slot) {
    const int i = g / p.k_tiles;
    const int kt = g - i * p.k_tiles;
    int tm, tn;
    tile_coords(static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x), p, tm, tn);
    const uint32_t full = full0 + 8 * slot;
    mbar_arrive_expect_tx(full, C::TX_BYTES);
    tma_load_2d(sA + slot * C::A_BYTES, tmA, full, kt * C::BK, tm * C::BM);
    tma_load_2d(sB + slot * C::B_BYTES, tmB, full, tn * C::BN, kt * C::BK);
}

template <class C>
__device__ __forceinline__ void consumer(const CUtensorMap* tmA, const CUtensorMap* tmB,
                                         const GemmParams& p, const uint8_t* sA_ptr,
                                         const uint8_t* sB_ptr, uint32_t full0, uint32_t empty0,
                                         int warp, int lane) {
    const uint32_t sA_u32 = smem_u32(sA_ptr), sB_u32 = smem_u32(sB_ptr);
    const int num_tiles = p.tiles_m * p.tiles_n;
    const int wm = warp % C::WARPS_M, wn = warp / C::WARPS_M;
    int tr, tc;
    lane_grid<C::LMAP>(lane, tr, tc);
    const int row_base = wm * 32 + tr;        // rows row_base + 4 i, i = 0..7
    const int col_base = wn * 64 + 4 * tc;    // cols col_base + {0..3} and + 32 + {0..3}
    constexpr int KQ = C::BK / 4;

    // Stage sequence of this CTA: k-tile kt of its i-th tile is stage
    // i * k_tiles + kt, held in ring slot (stage mod STAGES).
    const int my_tiles = (num_tiles - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                         static_cast<int>(gridDim.x);
    const int total = my_tiles * p.k_tiles;
    const bool issuer = C::INLINE && threadIdx.x == 0;
    if (issuer) {
        tma_prefetch_desc(tmA);
        tma_prefetch_desc(tmB);
        for (int g = 0; g < total && g < C::STAGES; ++g)
            issue_stage<C>(tmA, tmB, p, sA_u32, sB_u32, full0, g, g);
    }
    int g = 0;
    int s = 0;
    uint32_t ph = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
        int tm, tn;
        tile_coords(t, p, tm, tn);
        float acc[8][8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

        // With XPF, the first k-group of each stage (and its first B row) is
        // loaded while the previous stage's last k-group is multiplied.
        float4 a_pre[8];
        float4 b_pre0, b_pre1;
        if (C::XPF) {
            if (!wait_bounded(full0 + 8 * s, ph, p, STATUS_CONSUMER_TIMEOUT)) return;
            const uint8_t* a_st = sA_ptr + s * C::A_BYTES + row_base * 128;
            const uint8_t* b_st = sB_ptr + s * C::B_BYTES + col_base * 4;
            load_a_group(a_pre, a_st, 0, tr);
            b_pre0 = *reinterpret_cast<const float4*>(b_st);
            b_pre1 = *reinterpret_cast<const float4*>(b_st + 32 * 4);
        }

        for (int kt = 0; kt < p.k_tiles; ++kt) {
            if (!C::XPF) {
                if (!wait_bounded(full0 + 8 * s, ph, p, STATUS_CONSUMER_TIMEOUT)) return;
            }
            const uint8_t* a_st = sA_ptr + s * C::A_BYTES + row_base * 128;
            const uint8_t* b_st = sB_ptr + s * C::B_BYTES + col_base * 4;
            int s_next = s + 1;
            uint32_t ph_next = ph;
            if (s_next == C::STAGES) { s_next = 0; ph_next ^= 1u; }
#pragma unroll
            for (int kq = 0; kq < KQ; ++kq) {
                float4 a[8];
                if (C::XPF && kq == 0) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) a[i] = a_pre[i];
                } else {
                    load_a_group(a, a_st, kq, tr);
                }
                if (C::XPF && kq == KQ - 1 && kt + 1 < p.k_tiles) {
                    if (!wait_bounded(full0 + 8 * s_next, ph_next, p, STATUS_CONSUMER_TIMEOUT))
                        return;
                    const uint8_t* a_nx = sA_ptr + s_next * C::A_BYTES + row_base * 128;
                    const uint8_t* b_nx = sB_ptr + s_next * C::B_BYTES + col_base * 4;
                    load_a_group(a_pre, a_nx, 0, tr);
                    b_pre0 = *reinterpret_cast<const float4*>(b_nx);
                    b_pre1 = *reinterpret_cast<const float4*>(b_nx + 32 * 4);
                }
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    float4 b0, b1;
                    if (C::XPF && kq == 0 && kk == 0) {
                        b0 = b_pre0;
                        b1 = b_pre1;
                    } else {
                        const uint8_t* brow = b_st + (kq * 4 + kk) * C::BN * 4;
                        b0 = *reinterpret_cast<const float4*>(brow);
                        b1 = *reinterpret_cast<const float4*>(brow + 32 * 4);
                    }
                    outer_product<C::FORDER>(acc, a, kk, b0, b1);
                }
            }
            mbar_arrive(empty0 + 8 * s);
            if (issuer && g + C::STAGES < total) {
                // Refill this slot with stage g + STAGES once every consumer
                // has released stage g.
                if (!wait_bounded(empty0 + 8 * s, ph, p, STATUS_PRODUCER_TIMEOUT)) return;
                issue_stage<C>(tmA, tmB, p, sA_u32, sB_u32, full0, g + C::STAGES, s);
            }
            ++g;
            s = s_next;
            ph = ph_next;
        }

        // Epilogue: C = alpha * acc + beta * C, straight from registers.
        const int m0 = tm * C::BM + row_base;
        const int n0 = tn * C::BN + col_base;
        const bool use_c = p.beta != 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int m = m0 + 4 * i;
            if (m >= p.M) continue;
            float* crow = p.C + (long long)m * p.ldc;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int n = n0 + 32 * h;
                float v[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) v[e] = p.alpha * acc[i][4 * h + e];
                if (p.c_vec && n + 3 < p.N) {
                    float4* cp = reinterpret_cast<float4*>(crow + n);
                    if (use_c) {
                        const float4 c = *cp;
                        v[0] = fmaf(p.beta, c.x, v[0]);
                        v[1] = fmaf(p.beta, c.y, v[1]);
                        v[2] = fmaf(p.beta, c.z, v[2]);
                        v[3] = fmaf(p.beta, c.w, v[3]);
                    }
                    *cp = make_float4(v[0], v[1], v[2], v[3]);
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

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
sgemm_ws_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const GemmParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    // 1024-byte alignment: the 128B-swizzle pattern repeats every 8 rows.
    // (Pointer arithmetic on the __shared__ array keeps the shared address
    // space visible to the compiler, so the tile reads stay LDS.)
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* sA = smem;
    uint8_t* sB = smem + C::STAGES * C::A_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sB + C::STAGES * C::B_BYTES);
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = smem_u32(bars + C::STAGES);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full0 + 8 * s, C::FULL_COUNT);
            mbar_init(empty0 + 8 * s, C::CONSUMERS);
        }
        fence_barrier_init();
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (C::PRODUCER_WARPS > 0 && warp >= C::CONSUMER_WARPS) {
        producer<C>(&tmA, &tmB, p, smem_u32(sA), smem_u32(sB), full0, empty0,
                    warp - C::CONSUMER_WARPS, lane);
    } else {
        consumer<C>(&tmA, &tmB, p, sA, sB, full0, empty0, warp, lane);
    }
}

}  // namespace sg
