// sgemm_noalloc.cu — sgemm_noalloc: the same SGEMM as sgemm, for callers
// that must not allocate device memory.
//
// sgemm allocates on a device twice in its life: a status word (cudaMalloc,
// on the first call) and, for problems whose last wave of tiles is split
// across the SMs, a stream-K workspace (cudaMallocFromPoolAsync, per call).
// Some callers cannot allow either: programs whose device memory is owned
// by another allocator that must account for every byte, and real-time
// paths that may not take an allocator's locks. sgemm_noalloc serves them:
// it runs the same kernels with the same schedule, but its status word and
// stream-K partial sums live in one fixed scratch array compiled into this
// file.
//
// The scratch is a file-scope __device__ array of kScratchBytes (32 MiB).
// Every GPU that loads this library's module holds it until the process
// exits. Host code cannot use the array's name as a device address, so the
// first call on each device, with that device current, asks the runtime for
// the address with cudaGetSymbolAddress and caches it. That first call also
// performs the library's per-device kernel set-up; it should therefore come
// before any stream capture starts.
//
// All calls on a device share the array and it keeps the last call's
// contents: every partial-sum slot a launch reads was written earlier in the
// same launch, so nothing needs clearing per call; the status word is zero
// when the module loads, collects the time-out bits of every later call, and
// is read and cleared by sgemm_noalloc_check_status (a copy to a host
// variable and a memset on the caller's stream, nothing allocated). Calls
// that overlap on the GPU (for example on two streams without ordering
// between them) race on the array and may produce wrong results: serialise
// them.
#include <cstddef>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "sgemm.h"
#include "sgemm_internal.h"

// Status word (first 256 bytes) + stream-K partial-sum slots.
constexpr size_t kScratchBytes = size_t{32} << 20;
constexpr size_t kScratchStatusBytes = 256;
constexpr size_t kScratchWorkspaceBytes = kScratchBytes - kScratchStatusBytes;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

namespace sg {
namespace {

constexpr int kMaxScratchDevices = 64;

struct ScratchSlot {
    bool ready = false;
    unsigned char* ptr = nullptr;   // device address of g_noalloc_scratch
};

std::mutex g_scratch_mu;
ScratchSlot g_scratch_slot[kMaxScratchDevices];

// Device address of the scratch array on `dev`, which must be current.
int scratch_address(int dev, unsigned char** out) {
    if (dev < 0 || dev >= kMaxScratchDevices) return SGEMM_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchSlot& s = g_scratch_slot[dev];
    if (!s.ready) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr)
            return cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidSymbol, SGEMM_ERR_CUDA);
        s.ptr = static_cast<unsigned char*>(p);
        s.ready = true;
    }
    *out = s.ptr;
    return SGEMM_OK;
}

}  // namespace
}  // namespace sg

using namespace sg;

extern "C" int sgemm_noalloc(int64_t M, int64_t N, int64_t K, float alpha, const float* A,
                             int64_t lda, const float* B, int64_t ldb, float beta, float* C,
                             int64_t ldc, cudaStream_t stream) {
    int rc = check_args(M, N, K, alpha, A, lda, B, ldb, C, ldc);
    if (rc != SGEMM_OK) return rc;
    if (M == 0 || N == 0) return SGEMM_OK;
    const DeviceInfo* dev = nullptr;
    if ((rc = device_info(&dev)) != SGEMM_OK) return rc;
    unsigned char* scratch = nullptr;
    if ((rc = scratch_address(dev->device, &scratch)) != SGEMM_OK) return rc;
    Plan pl;
    // No packed copies of unaligned operands here: they would not fit the
    // scratch for large problems, so such operands keep the cp.async loads.
    if ((rc = make_plan(dev, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, true, false, &pl)) !=
        SGEMM_OK)
        return rc;
    // The stream-K workspace must fit in the fixed scratch: 2 slots of
    // 128 x 128 floats per SM, 19.5 MB on a 152-SM GB300.
    if (pl.ws_bytes > kScratchWorkspaceBytes) return SGEMM_ERR_INVALID_VALUE;
    int* status = reinterpret_cast<int*>(scratch);
    float* ws = pl.ws_bytes > 0 ? reinterpret_cast<float*>(scratch + kScratchStatusBytes) : nullptr;
    return launch_plan(&pl, status, ws, stream);
}

extern "C" int sgemm_noalloc_check_status(cudaStream_t stream, int* bits) {
    const DeviceInfo* dev = nullptr;
    int rc = device_info(&dev);
    if (rc != SGEMM_OK) return rc;
    unsigned char* scratch = nullptr;
    if ((rc = scratch_address(dev->device, &scratch)) != SGEMM_OK) return rc;
    int* status = reinterpret_cast<int*>(scratch);
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, SGEMM_ERR_CUDA);
    int v = 0;
    if ((e = cudaMemcpyAsync(&v, status, sizeof(int), cudaMemcpyDeviceToHost, stream)) !=
            cudaSuccess ||
        (e = cudaMemsetAsync(status, 0, sizeof(int), stream)) != cudaSuccess ||
        (e = cudaStreamSynchronize(stream)) != cudaSuccess)
        return cuda_fail(e, SGEMM_ERR_CUDA);
    if (bits != nullptr) *bits = v;
    return status_code(v);
}
