// sgemm_internal.h — the allocation-free planning and launch core shared by
// the C-ABI entry points (argument checks, per-device kernel set-up, kernel
// and schedule choice, TMA descriptors, launches). Nothing here allocates
// device memory: the caller passes the status word and the stream-K
// workspace.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "kernels.h"

namespace sg {

constexpr int kMaxFamilies = 32;

// What the planner needs to know about the current device. Filled once per
// device by device_info(): properties, kernel attributes, occupancy, and
// the TMA encoder entry point. No device memory is allocated.
struct DeviceInfo {
    int device = -1;
    int sm_count = 0;
    int ctas_per_sm[kMaxFamilies][4] = {};
};

struct Plan {
    int kind = 0;                 // 0: nothing to do, 1: C = beta * C, 2: GEMM
    const KernelFamily* fam = nullptr;
    const KernelEntry* k = nullptr;
    CUtensorMap tmA, tmB;
    GemmParams p;
    int grid = 0;
    int sk_tiles = 0;             // tiles finished by the stream-K fixup
    size_t ws_bytes = 0;          // stream-K workspace the launch needs
};

// Validates the arguments of sgemm (SGEMM_OK or SGEMM_ERR_INVALID_VALUE).
int check_args(int64_t M, int64_t N, int64_t K, float alpha, const float* A, int64_t lda,
               const float* B, int64_t ldb, const float* C, int64_t ldc);

// Per-device set-up of the current device (once, under a lock).
int device_info(const DeviceInfo** out);

// Chooses kernel, load modes, grid and schedule. allow_sk = false forces the
// data-parallel schedule (no workspace); otherwise ws_bytes tells the caller
// how much workspace to pass to launch_plan.
int make_plan(const DeviceInfo* dev, int64_t M, int64_t N, int64_t K, float alpha,
              const float* A, int64_t lda, const float* B, int64_t ldb, float beta,
              const float* C, int64_t ldc, bool allow_sk, Plan* pl);

// Enqueues the plan on `stream`. status: device status word; ws: at least
// pl->ws_bytes of device memory (may be null when ws_bytes == 0).
int launch_plan(Plan* pl, int* status, float* ws, cudaStream_t stream);

// Human-readable plan name into buf ("none", "scale", or the kernel name,
// with "+sk" when the stream-K tail is used).
void plan_name(const Plan& pl, char* buf, int buflen);

// Records a CUDA error for sgemm_last_cuda_error and returns `code`.
int cuda_fail(cudaError_t e, int code);

}  // namespace sg
