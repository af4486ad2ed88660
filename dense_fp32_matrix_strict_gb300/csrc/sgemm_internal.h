// sgemm_internal.h — the allocation-free planning and launch core shared by
// the C-ABI entry points (argument checks, per-device kernel set-up, kernel
// and schedule choice, TMA descriptors, launches). Nothing here allocates
// device memory: the caller passes the status word and the stream-K
// workspace.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cudaTypedefs.h>
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
    int ctas_per_sm[kMaxFamilies][kModes] = {};
    int clusters[kMaxFamilies][kModes] = {};   // co-resident clusters (cluster variants)
};

struct Plan {
    int kind = 0;                 // 0: nothing to do, 1: C = beta * C, 2: GEMM
    const KernelFamily* fam = nullptr;
    const KernelEntry* k = nullptr;
    CUtensorMap tmA, tmB;
    GemmParams p;
    int grid = 0;
    int sms = 0;                  // SMs of the device (grid of the packing copies)
    int sk_tiles = 0;             // stream-K tiles (split across CTAs)
    // Split tiles finished by the separate fixup kernel (":fixup") instead
    // of inside the GEMM kernel.
    bool sk_fixup = false;
    // Operand transposition: a_t, A stored K x M (loaded as [BK][BM] boxes);
    // b_t, B stored N x K (transposed into the packed B buffer first).
    bool a_t = false, b_t = false;
    // a_pre: a row-major A copied transposed (K x lda_pack) into the packed
    // A buffer, then read through the transposed-A kernel path.
    bool a_pre = false;
    // a_fused (with a_pre): that copy is made inside the GEMM kernel by its
    // transposer warps (Cfg::FUSED), unit by unit with a flag per unit after
    // the copy at offset at_flags_off of the packed A buffer, instead of by
    // a kernel before it. Not used for a call being captured into a graph
    // (a replay would see the flags its previous run left).
    bool a_fused = false;
    size_t at_flags_off = 0;
    // b_fused (with b_t and pack_b): the row-major copy of the transposed B
    // made inside the GEMM kernel the same way, its flags at offset
    // bt_flags_off of the packed B buffer.
    bool b_fused = false;
    size_t bt_flags_off = 0;
    // a_xp: a row-major A transposed in shared memory by the kernel's
    // transposer warps (mode LOAD_TMA_XP).
    bool a_xp = false;
    // Operands TMA cannot describe in place (base or row stride not 16-byte
    // aligned) but worth it: copied first to an aligned workspace buffer
    // with row stride ld_pack (a multiple of 4 floats).
    bool pack_a = false, pack_b = false;
    int64_t lda_pack = 0, ldb_pack = 0;
    // Workspace the launch needs: [packed A | packed B | stream-K slots],
    // each region a multiple of 256 bytes.
    size_t pack_a_bytes = 0, pack_b_bytes = 0, sk_bytes = 0;
    size_t ws_bytes = 0;
};

// Validates the arguments of sgemm (SGEMM_OK or SGEMM_ERR_INVALID_VALUE);
// the _ex form those of sgemm_ex (opa, opb: 0 as stored, 1 transposed).
int check_args(int64_t M, int64_t N, int64_t K, float alpha, const float* A, int64_t lda,
               const float* B, int64_t ldb, const float* C, int64_t ldc);
int check_args_ex(int opa, int opb, int64_t M, int64_t N, int64_t K, float alpha, const float* A,
                  int64_t lda, const float* B, int64_t ldb, const float* C, int64_t ldc);

// Per-device set-up of the current device (once, under a lock).
int device_info(const DeviceInfo** out);

// Chooses kernel, load modes, grid and schedule. allow_sk = false forces the
// data-parallel schedule; allow_pack = false never copies an operand to an
// aligned buffer. ws_bytes tells the caller how much workspace to pass to
// launch_plan (0 when both are false).
int make_plan(const DeviceInfo* dev, int64_t M, int64_t N, int64_t K, float alpha,
              const float* A, int64_t lda, const float* B, int64_t ldb, float beta,
              const float* C, int64_t ldc, bool allow_sk, bool allow_pack, Plan* pl);
// The same for transposed operands. A transposed B always needs the packing
// copy, a transposed A whenever TMA cannot read it in place: with
// allow_pack = false those return SGEMM_ERR_CUDA (allocation failure).
int make_plan_ex(const DeviceInfo* dev, int opa, int opb, int64_t M, int64_t N, int64_t K,
                 float alpha, const float* A, int64_t lda, const float* B, int64_t ldb,
                 float beta, const float* C, int64_t ldc, bool allow_sk, bool allow_pack,
                 Plan* pl);

// Enqueues the plan on `stream`. status: device status word; ws: at least
// pl->ws_bytes of 256-byte-aligned device memory (may be null when
// ws_bytes == 0).
int launch_plan(Plan* pl, int* status, float* ws, cudaStream_t stream);

// Turns copies made inside the GEMM kernel (a_fused, b_fused) into copies by
// kernels of their own, same GEMM kernel otherwise; for calls captured into
// a CUDA graph.
void unfuse_plan(Plan* pl);

// Human-readable plan name into buf ("none", "scale", or the kernel name,
// with "+packA" / "+packB" for operands copied to aligned buffers, "+packAT"
// for the transposed copy of A by a kernel of its own, "+packATfused" for
// that copy made inside the GEMM kernel, "+packBT" / "+packBTfused" the same
// for the row-major copy of a transposed B, "+sk" when the stream-K tail is
// used and finished in the kernel, "+skfix" when the fixup kernel finishes
// it).
void plan_name(const Plan& pl, char* buf, int buflen);

// The return code of a status word: SGEMM_ERR_DEVICE_TIMEOUT for any
// time-out bit, else SGEMM_ERR_DEVICE_CHECK for a schedule or index bit,
// else SGEMM_OK.
int status_code(int bits);

// Records a CUDA error for sgemm_last_cuda_error and returns `code`.
int cuda_fail(cudaError_t e, int code);

// The status word and the workspace pool of the regular entry points on the
// current device (allocated on first use).
int device_memory_handles(const DeviceInfo* dev, int** status, cudaMemPool_t* pool);

// cuTensorMapEncodeTiled, resolved by device_info().
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// Current limit of the kernels' bounded waits.
unsigned long long wait_timeout_ns();

// Whether kernels that follow one of the same call's own kernels on the
// stream are launched by programmatic stream serialisation (on unless the
// environment variable SGEMM_PDL is "0" when first asked).
bool pdl_enabled();

}  // namespace sg
