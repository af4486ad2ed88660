// kernels.h — host-side registry of the compiled SGEMM kernel variants.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "sgemm_kernel.cuh"
#include "sk_fixup.cuh"

namespace sg {

// Launches `kernel` on `stream`. With `pdl` set, by programmatic stream
// serialisation: the kernel may be scheduled while the kernel before it on
// the stream is still running, and waits for it (griddep_wait) before its
// first global-memory access; only used where that earlier kernel is one of
// this library's own, launched by the same call. With `cluster` > 1, in
// thread-block clusters of that many CTAs along x (the grid a multiple).
template <typename... Params, typename... Args>
cudaError_t launch_kernel(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, bool pdl, int cluster, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = static_cast<unsigned>(cluster);
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = static_cast<unsigned>(n);
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

struct KernelEntry {
    const char* name;
    int bm, bn, bk, stages, a_mode, b_mode, threads, smem_bytes;
    // Set attributes, query occupancy: CTAs per SM and, for a cluster
    // variant, how many of its clusters the whole GPU runs at once (0 else).
    cudaError_t (*prepare)(int* ctas_per_sm, int* clusters);
    cudaError_t (*launch)(const CUtensorMap* tmA, const CUtensorMap* tmB, const GemmParams* p,
                          int grid, cudaStream_t stream, bool pdl);
};

template <class C>
cudaError_t ws_prepare(int* ctas_per_sm, int* clusters) {
    cudaError_t e = cudaFuncSetAttribute(sgemm_ws_kernel<C>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, sgemm_ws_kernel<C>,
                                                      C::THREADS, C::SMEM_BYTES);
    *clusters = 0;
    if (e != cudaSuccess || C::CS == 1) return e;
    // Clusters are placed whole inside one GPC, so fewer than SMs / CS of
    // them may fit at once.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C::CS);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C::CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(clusters, sgemm_ws_kernel<C>, &cfg);
}

template <class C>
cudaError_t ws_launch(const CUtensorMap* tmA, const CUtensorMap* tmB, const GemmParams* p,
                      int grid, cudaStream_t stream, bool pdl) {
    return launch_kernel(sgemm_ws_kernel<C>, dim3(grid), dim3(C::THREADS), C::SMEM_BYTES, stream,
                         pdl, C::CS, *tmA, *tmB, *p);
}

// The stream-K fixup for a BM x BN tile: `split` CTAs per stream-K tile.
// Launched the ordinary way: scheduled early behind the persistent GEMM
// (programmatic serialisation), its waiting CTAs cost 0.3-2.4 us on GB300.
template <int BM, int BN>
cudaError_t fixup_launch(const GemmParams* p, int sk_tiles, int split, cudaStream_t stream) {
    sk_fixup_kernel<BM, BN><<<sk_tiles * split, 256, 0, stream>>>(*p, split);
    return cudaGetLastError();
}

// One kernel family: a CTA tile and tuning knobs, instantiated for the four
// (A, B) load-mode pairs of a row-major A and the two B load modes of a
// transposed A (TMA) in mode_index order, plus its stream-K fixup.
constexpr int kModes = 8;

struct KernelFamily {
    const char* name;
    int bm, bn;
    KernelEntry modes[kModes];
    cudaError_t (*fixup)(const GemmParams* p, int sk_tiles, int split, cudaStream_t stream);
    int cs = 1;   // CTAs per cluster sharing one tile (Cfg::CS); grid = tiles x cs
};

// Index into a family's modes: TMA/TMA, CP/TMA, TMA/CP, CP/CP for a
// row-major A; then transposed A (TMA) with B by TMA, with B by cp.async;
// then a row-major A transposed in shared memory, with B by TMA; then the
// transposed-A path on a transposed copy the kernel makes itself (Cfg::FUSED,
// B by TMA; only the 128 x 128 family has it).
constexpr int kModeFused = 7;
inline constexpr int mode_index(int a_mode, int b_mode, int a_t = 0) {
    return a_mode == LOAD_TMA_XP ? 6 : a_t ? 4 + b_mode : a_mode + 2 * b_mode;
}

template <int BM, int BN, int S, int AM, int BMD, int FORDER, int EARLY, int LMAP, int AT = 0,
          int ALOAD = 4, int TN = 8, int KSPLIT = 1, int CS = 1, int FUSED = 0>
constexpr KernelEntry make_entry(const char* name) {
    using C = Cfg<BM, BN, 32, S, AM, BMD, FORDER, EARLY, LMAP, AT, ALOAD, TN, KSPLIT, CS, FUSED>;
    // A variant whose ring does not fit in shared memory is left out (no
    // entry points); the planner never picks it.
    if constexpr (!C::FITS)
        return KernelEntry{name, BM, BN, 32, S, AM, BMD, C::THREADS, C::SMEM_BYTES, nullptr,
                           nullptr};
    else
        return KernelEntry{name, BM, BN, 32, S, AM, BMD, C::THREADS, C::SMEM_BYTES,
                           &ws_prepare<C>, &ws_launch<C>};
}

// A mode a family does not have (never planned).
constexpr KernelEntry no_entry(const char* name, int bm, int bn) {
    return KernelEntry{name, bm, bn, 32, 0, 0, 0, 0, 0, nullptr, nullptr};
}

// The fused transposed-copy mode of a family (kModeFused).
template <int BM, int BN, int S, int FORDER, int EARLY, int LMAP>
constexpr KernelEntry fused_entry(const char* name) {
    return make_entry<BM, BN, S, LOAD_TMA, LOAD_TMA, FORDER, EARLY, LMAP, 1, 4, 8, 1, 1, 1>(name);
}

#define SG_FAMILY_A(NAME, BM, BN, S, FORDER, EARLY, LMAP, ALOAD) \
    SG_FAMILY_AX(NAME, BM, BN, S, FORDER, EARLY, LMAP, ALOAD, no_entry(NAME "_ATtma_Btma", BM, BN))

#define SG_FAMILY_AX(NAME, BM, BN, S, FORDER, EARLY, LMAP, ALOAD, FUSED_ENTRY)             \
    KernelFamily {                                                                          \
        NAME, BM, BN,                                                                       \
            {                                                                               \
                make_entry<BM, BN, S, LOAD_TMA, LOAD_TMA, FORDER, EARLY, LMAP, 0, ALOAD>(     \
                    NAME "_Atma_Btma"),                                                     \
                make_entry<BM, BN, S, LOAD_CPASYNC, LOAD_TMA, FORDER, EARLY, LMAP, 0, ALOAD>( \
                    NAME "_Acp_Btma"),                                                      \
                make_entry<BM, BN, S, LOAD_TMA, LOAD_CPASYNC, FORDER, EARLY, LMAP, 0, ALOAD>( \
                    NAME "_Atma_Bcp"),                                                      \
                make_entry<BM, BN, S, LOAD_CPASYNC, LOAD_CPASYNC, FORDER, EARLY, LMAP, 0,     \
                           ALOAD>(NAME "_Acp_Bcp"),                                         \
                make_entry<BM, BN, S, LOAD_TMA, LOAD_TMA, FORDER, EARLY, LMAP, 1>(            \
                    NAME "_ATtma_Btma"),                                                    \
                make_entry<BM, BN, S, LOAD_TMA, LOAD_CPASYNC, FORDER, EARLY, LMAP, 1>(        \
                    NAME "_ATtma_Bcp"),                                                     \
                make_entry<BM, BN, S, LOAD_TMA_XP, LOAD_TMA, FORDER, EARLY, LMAP>(            \
                    NAME "_Axp_Btma"),                                                      \
                FUSED_ENTRY,                                                                \
            },                                                                              \
            &fixup_launch<BM, BN>                                                           \
    }

// A family with TN columns per lane (see Cfg) in every mode.
#define SG_FAMILY_T(NAME, BM, BN, S, FORDER, EARLY, LMAP, TN)                               \
    KernelFamily {                                                                          \
        NAME, BM, BN,                                                                       \
            {                                                                               \
                make_entry<BM, BN, S, LOAD_TMA, LOAD_TMA, FORDER, EARLY, LMAP, 0, 4, TN>(     \
                    NAME "_Atma_Btma"),                                                     \
                make_entry<BM, BN, S, LOAD_CPASYNC, LOAD_TMA, FORDER, EARLY, LMAP, 0, 4, TN>( \
                    NAME "_Acp_Btma"),                                                      \
                make_entry<BM, BN, S, LOAD_TMA, LOAD_CPASYNC, FORDER, EARLY, LMAP, 0, 4, TN>( \
                    NAME "_Atma_Bcp"),                                                      \
                make_entry<BM, BN, S, LOAD_CPASYNC, LOAD_CPASYNC, FORDER, EARLY, LMAP, 0, 4,  \
                           TN>(NAME "_Acp_Bcp"),                                            \
                make_entry<BM, BN, S, LOAD_TMA, LOAD_TMA, FORDER, EARLY, LMAP, 1, 4, TN>(     \
                    NAME "_ATtma_Btma"),                                                    \
                make_entry<BM, BN, S, LOAD_TMA, LOAD_CPASYNC, FORDER, EARLY, LMAP, 1, 4, TN>( \
                    NAME "_ATtma_Bcp"),                                                     \
                make_entry<BM, BN, S, LOAD_TMA_XP, LOAD_TMA, FORDER, EARLY, LMAP, 0, 4, TN>(  \
                    NAME "_Axp_Btma"),                                                      \
                no_entry(NAME "_ATtma_Btma", BM, BN),                                       \
            },                                                                              \
            &fixup_launch<BM, BN>                                                           \
    }

// A family whose consumer warps come in KSPLIT k-groups, its CTAs in
// clusters of CS sharing one tile (see Cfg).
#define SG_FAMILY_KC(NAME, BM, BN, S, KS, CS)                                               \
    KernelFamily {                                                                          \
        NAME, BM, BN,                                                                       \
            {                                                                               \
                make_entry<BM, BN, S, LOAD_TMA, LOAD_TMA, 3, 1, 0, 0, 4, 8, KS, CS>(          \
                    NAME "_Atma_Btma"),                                                     \
                make_entry<BM, BN, S, LOAD_CPASYNC, LOAD_TMA, 3, 1, 0, 0, 4, 8, KS, CS>(      \
                    NAME "_Acp_Btma"),                                                      \
                make_entry<BM, BN, S, LOAD_TMA, LOAD_CPASYNC, 3, 1, 0, 0, 4, 8, KS, CS>(      \
                    NAME "_Atma_Bcp"),                                                      \
                make_entry<BM, BN, S, LOAD_CPASYNC, LOAD_CPASYNC, 3, 1, 0, 0, 4, 8, KS, CS>(  \
                    NAME "_Acp_Bcp"),                                                       \
                make_entry<BM, BN, S, LOAD_TMA, LOAD_TMA, 3, 1, 0, 1, 4, 8, KS, CS>(          \
                    NAME "_ATtma_Btma"),                                                    \
                make_entry<BM, BN, S, LOAD_TMA, LOAD_CPASYNC, 3, 1, 0, 1, 4, 8, KS, CS>(      \
                    NAME "_ATtma_Bcp"),                                                     \
                make_entry<BM, BN, S, LOAD_TMA_XP, LOAD_TMA, 3, 1, 0, 0, 4, 8, KS, CS>(       \
                    NAME "_Axp_Btma"),                                                      \
                no_entry(NAME "_ATtma_Btma", BM, BN),                                       \
            },                                                                              \
            &fixup_launch<BM, BN>, CS                                                       \
    }

#define SG_FAMILY_K(NAME, BM, BN, S, KS) SG_FAMILY_KC(NAME, BM, BN, S, KS, 1)

#define SG_FAMILY(NAME, BM, BN, S, FORDER, EARLY, LMAP) \
    SG_FAMILY_A(NAME, BM, BN, S, FORDER, EARLY, LMAP, 4)

// The same with the fused transposed-copy mode.
#define SG_FAMILY_FUSED(NAME, BM, BN, S, FORDER, EARLY, LMAP)    \
    SG_FAMILY_AX(NAME, BM, BN, S, FORDER, EARLY, LMAP, 4,        \
                 (fused_entry<BM, BN, S, FORDER, EARLY, LMAP>(NAME "_ATtma_Btma")))

// Families, one translation unit each (compiled in parallel). The first
// seven are the ones "auto" chooses between; the rest are tuning
// alternatives that sgemm_set_config can force.
const KernelFamily* family_128x128();
const KernelFamily* family_64x64();
const KernelFamily* family_128x64();
const KernelFamily* family_128x64_k2();
const KernelFamily* family_64x64_k4();
const KernelFamily* family_64x64_k4_c2();
const KernelFamily* family_64x64_k4_c4();
const KernelFamily* const* sweep_families(int* count);

}  // namespace sg
