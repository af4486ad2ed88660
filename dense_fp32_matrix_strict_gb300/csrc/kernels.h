// kernels.h — host-side registry of the compiled SGEMM kernel variants.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "sgemm_kernel.cuh"

namespace sg {

struct KernelEntry {
    const char* name;
    int bm, bn, bk, stages, a_mode, b_mode, threads, smem_bytes;
    cudaError_t (*prepare)(int* ctas_per_sm);   // set attributes, query occupancy
    cudaError_t (*launch)(const CUtensorMap* tmA, const CUtensorMap* tmB, const GemmParams* p,
                          int grid, cudaStream_t stream);
};

template <class C>
cudaError_t ws_prepare(int* ctas_per_sm) {
    cudaError_t e = cudaFuncSetAttribute(sgemm_ws_kernel<C>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, sgemm_ws_kernel<C>,
                                                         C::THREADS, C::SMEM_BYTES);
}

template <class C>
cudaError_t ws_launch(const CUtensorMap* tmA, const CUtensorMap* tmB, const GemmParams* p,
                      int grid, cudaStream_t stream) {
    sgemm_ws_kernel<C><<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(*tmA, *tmB, *p);
    return cudaGetLastError();
}

#define SG_WS_ENTRY(NAME, BM, BN, S, AM, BMD)                                              \
    KernelEntry {                                                                          \
        NAME, BM, BN, 32, S, AM, BMD, Cfg<BM, BN, 32, S, AM, BMD>::THREADS,                \
            Cfg<BM, BN, 32, S, AM, BMD>::SMEM_BYTES, &ws_prepare<Cfg<BM, BN, 32, S, AM, BMD>>, \
            &ws_launch<Cfg<BM, BN, 32, S, AM, BMD>>                                        \
    }

// Each returns its table (4 entries: A/B load modes TMA/TMA, CP/TMA, TMA/CP,
// CP/CP, in that order). Defined in one translation unit per CTA tile.
const KernelEntry* ws_kernels_128x128();
const KernelEntry* ws_kernels_64x64();

// Index into a 4-entry table.
inline int mode_index(int a_mode, int b_mode) { return a_mode + 2 * b_mode; }

}  // namespace sg
