// sgemm_api.cu — the C ABI: argument checks, per-device set-up, kernel plan
// (CTA tile, TMA or cp.async per operand, persistent grid, data-parallel +
// stream-K schedule), TMA descriptor encoding, and launches on the caller's
// stream.
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "sgemm.h"
#include "sgemm_internal.h"

namespace sg {

namespace {

constexpr int kMaxDevices = 64;
constexpr int kStatusBytes = 256;

// All compiled kernel families: [0] 128x128, [1] 64x64, [2] 128x64,
// [3] 128x64 in two k-groups, [4] 64x64 in four k-groups and [5], [6] the
// same in clusters of 2 and 4 CTAs are what "auto" chooses between; the
// rest are tuning alternatives.
struct Registry {
    const KernelFamily* fam[kMaxFamilies];
    int count = 0;
    Registry() {
        fam[count++] = family_128x128();
        fam[count++] = family_64x64();
        fam[count++] = family_128x64();
        fam[count++] = family_128x64_k2();
        fam[count++] = family_64x64_k4();
        fam[count++] = family_64x64_k4_c2();
        fam[count++] = family_64x64_k4_c4();
        int n = 0;
        const KernelFamily* const* sw = sweep_families(&n);
        for (int i = 0; i < n && count < kMaxFamilies; ++i) fam[count++] = sw[i];
    }
};

const Registry& registry() {
    static const Registry r;
    return r;
}

struct DeviceSlot {
    bool ready = false;
    int error = SGEMM_OK;
    DeviceInfo info;
};

// Memory the regular entry points own on a device: the status word and a
// library-private stream-ordered pool for stream-K workspaces.
struct DeviceMemory {
    bool ready = false;
    int* status = nullptr;
    cudaMemPool_t pool = nullptr;
};

std::mutex g_mu;
DeviceSlot g_dev[kMaxDevices];
DeviceMemory g_mem[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
bool g_env_read = false;

// Forced configuration: family index (-1 = auto); cp = force cp.async loads;
// sk = -1 auto, 0 never use the stream-K tail.
std::atomic<int> g_force_family{-1};
std::atomic<int> g_force_cp{0};
// at = -1 auto, 0 never, 1 always copy a row-major A transposed (K x M) into
// the workspace and run the transposed-A kernel on it.
std::atomic<int> g_force_at{-1};
std::atomic<int> g_force_sk{-1};
// fx = 1: split tiles finished by the separate fixup kernel instead of in
// the GEMM kernel (":fixup").
std::atomic<int> g_force_fx{0};
std::atomic<unsigned long long> g_timeout_ns{2000000000ull};
// Flag value of the next launch that finishes split tiles in the kernel or
// makes an operand copy itself: unique per launch in this process and never
// 0. The flags sit in recycled pool memory that may hold anything a call left
// there (operand copies, partial sums), so a value a stale word could equal
// by chance must not be easy to hit: the upper half starts as a quiet-NaN
// pattern with an unusual payload (0x7fc5a5a5), the lower half counts.
std::atomic<unsigned long long> g_sk_tag{0x7fc5a5a500000001ull};

thread_local int t_last_cuda_error = 0;

// Per-shape configuration rules (sgemm_set_shape_config), consulted by
// make_plan only while the global configuration is "auto". An autotuning
// sweep installs the fastest configuration it measured for each shape here.
// A configuration choice: family index (-1 auto), cp.async forced, stream-K
// (-1 auto, 0 never), how a row-major A reaches the consumers (-1 auto, 0 as
// stored, 1 through a transposed copy in HBM, 2 transposed in shared memory).
struct Config {
    int family = -1, cp = 0, sk = -1, at = -1, fx = 0;
    bool is_auto() const { return family < 0 && cp == 0 && sk < 0 && at < 0 && fx == 0; }
};

struct ShapeRule {
    int64_t M, N, K;
    Config cfg;
};
constexpr int kMaxShapeRules = 256;
std::mutex g_rules_mu;
ShapeRule g_rules[kMaxShapeRules];
int g_nrules = 0;

bool shape_rule(int64_t M, int64_t N, int64_t K, Config* cfg) {
    std::lock_guard<std::mutex> lock(g_rules_mu);
    for (int i = 0; i < g_nrules; ++i) {
        const ShapeRule& r = g_rules[i];
        if (r.M == M && r.N == N && r.K == K) {
            *cfg = r.cfg;
            return true;
        }
    }
    return false;
}

// "<family>[:cpasync][:dp][:at|:atcopy|:noat|:xp][:fixup]" with <family> one
// of auto, 128x128, 64x64, 128x64 or a registry name. ":at" takes the
// transposed copy of A (made inside the GEMM kernel where the family can),
// ":atcopy" the same copy made by a kernel of its own.
int parse_config(const char* name, Config* out) {
    if (name == nullptr) return SGEMM_ERR_INVALID_VALUE;
    char buf[128];
    std::strncpy(buf, name, sizeof(buf) - 1);
    buf[sizeof(buf) - 1] = '\0';
    int want_cp = 0, want_sk = -1, want_at = -1, want_fx = 0;
    char* mod = std::strchr(buf, ':');
    if (mod != nullptr) *mod++ = '\0';
    while (mod != nullptr) {
        char* next = std::strchr(mod, ':');
        if (next != nullptr) *next++ = '\0';
        if (std::strcmp(mod, "cpasync") == 0) want_cp = 1;
        else if (std::strcmp(mod, "dp") == 0) want_sk = 0;
        else if (std::strcmp(mod, "at") == 0) want_at = 1;
        else if (std::strcmp(mod, "noat") == 0) want_at = 0;
        else if (std::strcmp(mod, "xp") == 0) want_at = 2;
        else if (std::strcmp(mod, "atcopy") == 0) want_at = 3;
        else if (std::strcmp(mod, "fixup") == 0) want_fx = 1;
        else return SGEMM_ERR_INVALID_VALUE;
        mod = next;
    }
    int f = -2;
    if (std::strcmp(buf, "auto") == 0 || buf[0] == '\0') f = -1;
    else if (std::strcmp(buf, "128x128") == 0) f = 0;
    else if (std::strcmp(buf, "64x64") == 0) f = 1;
    else if (std::strcmp(buf, "128x64") == 0) f = 2;
    else {
        const Registry& r = registry();
        for (int i = 0; i < r.count; ++i)
            if (std::strcmp(buf, r.fam[i]->name) == 0) f = i;
    }
    if (f == -2) return SGEMM_ERR_INVALID_VALUE;
    out->family = f;
    out->cp = want_cp;
    out->sk = want_sk;
    out->at = want_at;
    out->fx = want_fx;
    return SGEMM_OK;
}

void set_global_config(const Config& c) {
    g_force_family = c.family;
    g_force_cp = c.cp;
    g_force_sk = c.sk;
    g_force_at = c.at;
    g_force_fx = c.fx;
}

void read_env_locked() {
    if (g_env_read) return;
    g_env_read = true;
    const char* env = std::getenv("SGEMM_FORCE_CONFIG");
    Config c;
    if (env != nullptr && parse_config(env, &c) == SGEMM_OK) set_global_config(c);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// [lo, hi) byte range of a rows x cols matrix with leading dimension ld.
void extent(const void* p, int64_t rows, int64_t cols, int64_t ld, uintptr_t* lo, uintptr_t* hi) {
    *lo = reinterpret_cast<uintptr_t>(p);
    *hi = *lo + static_cast<uintptr_t>(((rows - 1) * ld + cols) * 4);
}

// 2-D row-major fp32 tensor map: rows x cols, row stride ld floats, box of
// box_rows x box_cols, optional 128-byte swizzle. Returns false if the
// driver rejects it.
bool encode_2d(CUtensorMap* map, const float* base, int64_t rows, int64_t cols, int64_t ld,
               int box_rows, int box_cols, bool swizzle128) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 4};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool tma_ok(const float* p, int64_t ld, int64_t rows, int64_t cols) {
    return aligned(p, 16) && (ld % 4) == 0 && ld < ((int64_t)1 << 38) && rows >= 1 && cols >= 1 &&
           rows <= 0xffffffffll && cols <= 0xffffffffll;
}

// C = beta * C over an M x N matrix (beta == 0 writes zeros, never reads C).
__global__ void scale_kernel(float* __restrict__ C, long long ldc, int M, int N, float beta) {
    for (long long m = blockIdx.y; m < M; m += gridDim.y) {
        float* row = C + m * ldc;
        for (int n = blockIdx.x * blockDim.x + threadIdx.x; n < N; n += blockDim.x * gridDim.x)
            row[n] = (beta == 0.0f) ? 0.0f : beta * row[n];
    }
}

// dst (rows x ldd, ldd = cols rounded up to 4) <- src (rows x cols, row
// stride lds, any alignment), one float4 of dst per thread per step; the
// padding columns get zeros. HBM-bound: one read and one write of the
// operand.
__global__ void pack_rows_kernel(const float* __restrict__ src, long long lds,
                                 float* __restrict__ dst, long long ldd, int rows, int cols) {
    griddep_wait();
    griddep_launch_dependents();
    const int quads = (cols + 3) >> 2;
    const long long total = static_cast<long long>(rows) * quads;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long r = i / quads;
        const int c = static_cast<int>(i - r * quads) * 4;
        const float* s = src + r * lds + c;
        float4 v;
        v.x = s[0];
        v.y = c + 1 < cols ? s[1] : 0.0f;
        v.z = c + 2 < cols ? s[2] : 0.0f;
        v.w = c + 3 < cols ? s[3] : 0.0f;
        *reinterpret_cast<float4*>(dst + r * ldd + c) = v;
    }
}

// dst (C x ldd, ldd = R rounded up to 4) <- the transpose of src (R x C, row
// stride lds): dst[c][r] = src[r][c], zeros in the padding columns r >= R.
// A block moves a 64 x 64 tile through shared memory (one padding column
// against bank conflicts): float4 reads along src rows when src allows them,
// float4 writes along dst rows (ldd is a multiple of 4 and dst 16-byte
// aligned), so both sides stay coalesced in 16-byte pieces. HBM-bound: one
// read and one write of the operand.
constexpr int kTpTile = 64;

__global__ void __launch_bounds__(256) transpose_pack_kernel(const float* __restrict__ src,
                                                             long long lds, float* __restrict__ dst,
                                                             long long ldd, int R, int C) {
    __shared__ float tile[kTpTile][kTpTile + 1];
    griddep_wait();
    griddep_launch_dependents();
    const bool vec = (reinterpret_cast<uintptr_t>(src) % 16 == 0) && (lds % 4 == 0);
    const long long c0 = static_cast<long long>(blockIdx.x) * kTpTile;
    const long long tiles_r = (ldd + kTpTile - 1) / kTpTile;
    const int t = threadIdx.x;
    for (long long tr = blockIdx.y; tr < tiles_r; tr += gridDim.y) {
        const long long r0 = tr * kTpTile;
        // 64 rows x 16 float4 of src; 16 consecutive threads read one row.
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int q = t + 256 * j;
            const int rr = q >> 4, cc = (q & 15) * 4;
            const long long r = r0 + rr, c = c0 + cc;
            float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (r < R) {
                const float* sp = src + r * lds + c;
                if (vec && c + 3 < C) {
                    v = *reinterpret_cast<const float4*>(sp);
                } else {
                    if (c < C) v.x = sp[0];
                    if (c + 1 < C) v.y = sp[1];
                    if (c + 2 < C) v.z = sp[2];
                    if (c + 3 < C) v.w = sp[3];
                }
            }
            tile[rr][cc] = v.x;
            tile[rr][cc + 1] = v.y;
            tile[rr][cc + 2] = v.z;
            tile[rr][cc + 3] = v.w;
        }
        __syncthreads();
        // 64 dst rows (src columns) x 16 float4 along r.
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int q = t + 256 * j;
            const int cc = q >> 4, rr = (q & 15) * 4;
            const long long c = c0 + cc, r = r0 + rr;
            if (c < C && r < ldd)
                *reinterpret_cast<float4*>(dst + c * ldd + r) =
                    make_float4(tile[rr][cc], tile[rr + 1][cc], tile[rr + 2][cc], tile[rr + 3][cc]);
        }
        __syncthreads();
    }
}

// Launches transpose_pack_kernel for an R x C source.
cudaError_t launch_transpose_pack(const float* src, long long lds, float* dst, long long ldd,
                                  int R, int C, cudaStream_t stream, bool pdl) {
    const long long tiles_r = (ldd + kTpTile - 1) / kTpTile;
    const dim3 grid(static_cast<unsigned>((C + kTpTile - 1) / kTpTile),
                    static_cast<unsigned>(tiles_r < 65535 ? tiles_r : 65535));
    return launch_kernel(transpose_pack_kernel, grid, dim3(256), 0, stream, pdl, 1, src, lds,
                         dst, ldd, R, C);
}

size_t align256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

__global__ void wait_timeout_kernel(GemmParams p) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) wait_bounded(b, 0, p, STATUS_CONSUMER_TIMEOUT);
}

// The status word and workspace pool of the current device (allocated on
// first use).
int device_memory(const DeviceInfo* info, DeviceMemory** out) {
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceMemory& m = g_mem[info->device];
    if (m.ready) {
        *out = &m;
        return SGEMM_OK;
    }
    cudaError_t e;
    void* status = nullptr;
    if ((e = cudaMalloc(&status, kStatusBytes)) != cudaSuccess) return cuda_fail(e, SGEMM_ERR_CUDA);
    if ((e = cudaMemset(status, 0, kStatusBytes)) != cudaSuccess ||
        (e = cudaDeviceSynchronize()) != cudaSuccess) {
        cudaFree(status);
        return cuda_fail(e, SGEMM_ERR_CUDA);
    }
    cudaMemPoolProps props;
    std::memset(&props, 0, sizeof(props));
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = info->device;
    cudaMemPool_t pool = nullptr;
    if ((e = cudaMemPoolCreate(&pool, &props)) != cudaSuccess) {
        cudaFree(status);
        return cuda_fail(e, SGEMM_ERR_CUDA);
    }
    // Keep freed workspace in the pool instead of returning it at every
    // synchronisation.
    uint64_t keep = UINT64_MAX;
    cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
    m.status = static_cast<int*>(status);
    m.pool = pool;
    m.ready = true;
    *out = &m;
    return SGEMM_OK;
}

}  // namespace

// A kernel that follows a packing copy of the same call is launched by
// programmatic stream serialisation (it is scheduled while the copy
// finishes and waits for it on the device), unless the environment variable
// SGEMM_PDL is "0" when the library first launches. On GB300 this saves
// ~1.5 us of the 4096^3 call (transposing copy of A, then the GEMM).
bool pdl_enabled() {
    static const bool on = [] {
        const char* v = std::getenv("SGEMM_PDL");
        return !(v != nullptr && std::strcmp(v, "0") == 0);
    }();
    return on;
}

int status_code(int bits) {
    if (bits & (STATUS_CONSUMER_TIMEOUT | STATUS_PRODUCER_TIMEOUT | STATUS_DRAIN_TIMEOUT))
        return SGEMM_ERR_DEVICE_TIMEOUT;
    if (bits != 0) return SGEMM_ERR_DEVICE_CHECK;
    return SGEMM_OK;
}

int cuda_fail(cudaError_t e, int code) {
    t_last_cuda_error = static_cast<int>(e);
    return code;
}

int check_args(int64_t M, int64_t N, int64_t K, float alpha, const float* A, int64_t lda,
               const float* B, int64_t ldb, const float* C, int64_t ldc) {
    return check_args_ex(0, 0, M, N, K, alpha, A, lda, B, ldb, C, ldc);
}

int check_args_ex(int opa, int opb, int64_t M, int64_t N, int64_t K, float alpha, const float* A,
                  int64_t lda, const float* B, int64_t ldb, const float* C, int64_t ldc) {
    const int64_t kMax = 0x7fffffff;
    if ((opa != 0 && opa != 1) || (opb != 0 && opb != 1)) return SGEMM_ERR_INVALID_VALUE;
    if (M < 0 || N < 0 || K < 0 || M > kMax || N > kMax || K > kMax) return SGEMM_ERR_INVALID_VALUE;
    // Stored shapes: A is M x K (K x M when transposed), B is K x N (N x K).
    const int64_t a_rows = opa ? K : M, a_cols = opa ? M : K;
    const int64_t b_rows = opb ? N : K, b_cols = opb ? K : N;
    if (lda < (a_cols > 1 ? a_cols : 1) || ldb < (b_cols > 1 ? b_cols : 1) ||
        ldc < (N > 1 ? N : 1))
        return SGEMM_ERR_INVALID_VALUE;
    // Offsets up to rows * ld must fit comfortably in int64 bytes.
    const int64_t kOff = (int64_t)1 << 60;
    if ((a_rows > 0 && lda > kOff / a_rows) || (b_rows > 0 && ldb > kOff / b_rows) ||
        (M > 0 && ldc > kOff / M))
        return SGEMM_ERR_INVALID_VALUE;
    if (M == 0 || N == 0) return SGEMM_OK;
    if (C == nullptr || !aligned(C, 4)) return SGEMM_ERR_INVALID_VALUE;
    const bool reads_ab = (alpha != 0.0f) && (K > 0);
    if (reads_ab) {
        if (A == nullptr || B == nullptr || !aligned(A, 4) || !aligned(B, 4))
            return SGEMM_ERR_INVALID_VALUE;
        uintptr_t clo, chi, lo, hi;
        extent(C, M, N, ldc, &clo, &chi);
        extent(A, a_rows, a_cols, lda, &lo, &hi);
        if (lo < chi && clo < hi) return SGEMM_ERR_INVALID_VALUE;
        extent(B, b_rows, b_cols, ldb, &lo, &hi);
        if (lo < chi && clo < hi) return SGEMM_ERR_INVALID_VALUE;
    }
    return SGEMM_OK;
}

int device_info(const DeviceInfo** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, SGEMM_ERR_CUDA);
    if (dev < 0 || dev >= kMaxDevices) return SGEMM_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_mu);
    read_env_locked();
    DeviceSlot& st = g_dev[dev];
    if (st.ready) {
        *out = &st.info;
        return SGEMM_OK;
    }
    if (st.error != SGEMM_OK) return st.error;
    int major = 0, minor = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return cuda_fail(e, SGEMM_ERR_CUDA);
    if (major != 10 || minor != 3) {
        st.error = SGEMM_ERR_UNSUPPORTED_DEVICE;
        return st.error;
    }
    if (g_encode == nullptr) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
            return cuda_fail(e == cudaSuccess ? cudaErrorNotSupported : e, SGEMM_ERR_CUDA);
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    const Registry& reg = registry();
    for (int f = 0; f < reg.count; ++f) {
        for (int m = 0; m < kModes; ++m) {
            int n = 0, ncl = 0;
            const KernelEntry& ke = reg.fam[f]->modes[m];
            e = ke.prepare != nullptr ? ke.prepare(&n, &ncl) : cudaSuccess;
            // A cluster variant of which no cluster fits is as unusable.
            if (e == cudaSuccess && reg.fam[f]->cs > 1 && ncl <= 0) n = 0;
            if (e != cudaSuccess || n <= 0) {
                // The 128 x 128 and 64 x 64 families must work in their
                // row-major and transposed-A modes; the in-smem transpose
                // mode, the 128 x 64 family (which "auto" then skips) and a
                // tuning alternative that cannot run here are only marked
                // unusable.
                if (f < 2 && m < 6)
                    return cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidConfiguration,
                                     SGEMM_ERR_CUDA);
                (void)cudaGetLastError();
                n = 0;
                ncl = 0;
            }
            st.info.ctas_per_sm[f][m] = n;
            st.info.clusters[f][m] = ncl;
        }
    }
    st.info.device = dev;
    st.info.sm_count = sms;
    st.ready = true;
    *out = &st.info;
    return SGEMM_OK;
}

int make_plan(const DeviceInfo* dev, int64_t M, int64_t N, int64_t K, float alpha,
              const float* A, int64_t lda, const float* B, int64_t ldb, float beta,
              const float* C, int64_t ldc, bool allow_sk, bool allow_pack, Plan* pl) {
    return make_plan_ex(dev, 0, 0, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, allow_sk,
                        allow_pack, pl);
}

int make_plan_ex(const DeviceInfo* dev, int opa, int opb, int64_t M, int64_t N, int64_t K,
                 float alpha, const float* A, int64_t lda, const float* B, int64_t ldb,
                 float beta, const float* C, int64_t ldc, bool allow_sk, bool allow_pack,
                 Plan* pl) {
    pl->a_t = opa != 0;
    pl->b_t = opb != 0;
    if (M == 0 || N == 0) {
        pl->kind = 0;
        return SGEMM_OK;
    }
    if (alpha == 0.0f || K == 0) {
        pl->kind = 1;
        GemmParams& p = pl->p;
        std::memset(&p, 0, sizeof(p));
        p.M = static_cast<int>(M);
        p.N = static_cast<int>(N);
        p.C = const_cast<float*>(C);
        p.ldc = ldc;
        p.beta = beta;
        return SGEMM_OK;
    }
    pl->kind = 2;
    const int sms = dev->sm_count;
    pl->sms = sms;
    Config cfg;
    cfg.family = g_force_family.load();
    cfg.cp = g_force_cp.load();
    cfg.sk = g_force_sk.load();
    cfg.at = g_force_at.load();
    cfg.fx = g_force_fx.load();
    if (cfg.is_auto()) shape_rule(M, N, K, &cfg);
    pl->sk_fixup = cfg.fx != 0;
    int fi = cfg.family;
    const int force_cp_flag = cfg.cp;
    const int force_sk = cfg.sk;
    // Under "auto" the choice below also decides whether the stream-K tail
    // is used; a forced family keeps the fixed rule further down.
    bool sk_decided = false;
    if (fi < 0) {
        sk_decided = true;
        auto cdiv = [](int64_t a, int64_t b) { return (a + b - 1) / b; };
        const int64_t kt = cdiv(K, 32);
        const double dkt = static_cast<double>(kt);
        const int64_t nsm = sms;
        const bool sk_possible = allow_sk && force_sk != 0;
        const int64_t tiles128 = cdiv(M, 128) * cdiv(N, 128);
        const int64_t tiles128x64 = cdiv(M, 128) * cdiv(N, 64);
        const int64_t tiles64 = cdiv(M, 64) * cdiv(N, 64);
        // A transposed A always goes by TMA (in place or packed); a
        // transposed B is always copied to the row-major layout first.
        const bool a_tma = opa ? true : (tma_ok(A, lda, M, K) || (allow_pack && N >= 256));
        const bool b_tma = opb ? true : (tma_ok(B, ldb, K, N) || (allow_pack && M >= 256));
        const bool tma_both = force_cp_flag == 0 && a_tma && b_tma;
        const int mi_tt = mode_index(LOAD_TMA, LOAD_TMA, opa);
        if (!tma_both && tiles128 * kt < 2 * nsm) {
            // Operands only cp.async can read, below two 128 x 128 x 32
            // k-iterations per SM: the 64 x 64 tile, with the stream-K tail
            // only if its own k-iterations still give every SM two.
            fi = 1;
            if (!(sk_possible && tiles64 * kt >= 2 * nsm)) allow_sk = false;
        } else {
            // Each candidate's cost in units of one 128 x 128 x 32
            // k-iteration of a CTA alone on its SM (~2.3 us on GB300), fitted
            // to sweeps on GB300 (152 SMs); the launch itself (~7 us) is
            // common to all and left out. Per k-iteration of one tile: a
            // 128 x 64 CTA alone on its SM 0.63 units, two co-resident ones
            // 1.06 for both; 128 x 64 in two k-groups 0.54; 64 x 64 in four
            // k-groups 0.31. The stream-K tail adds its partial sums and
            // their hand-over. Finished inside the kernel: ~2 units plus
            // ~0.26 for every segment of a split tile beyond two (the
            // finishing CTA reads one slot per segment; fitted on GB300 to
            // 1024^3, 2048^3, 512 x 2048 x 1024, 256^2 x 8192, 200 x 300 x
            // 6000 and 130 x 72 x 4100 across the three tile families).
            // With the separate fixup kernel: ~5 units for 128 x 128 tiles
            // and ~4 for 64 x 64 (taken as 6 and 4, so that a tie goes to
            // whole tiles).
            const double inf = 1e300;
            int best_f = 0;
            bool best_sk = false;
            double best_c = inf;
            auto offer = [&](int f, bool sk, double c) {
                if (c < best_c) {
                    best_f = f;
                    best_sk = sk;
                    best_c = c;
                }
            };
            // Whole waves of tiles plus, with the stream-K tail, the last
            // partial wave's k-iterations spread over the CTAs (the schedule
            // further down: ranges at least kt/32 iterations long).
            auto sk_ctas = [&](int64_t tiles, int64_t cap) {
                const int64_t S = (tiles % cap) * kt;
                int64_t G = S / cdiv(kt, 32);
                if (G > cap) G = cap;
                if (G < 1) G = 1;
                return G;
            };
            auto sk_iters = [&](int64_t tiles, int64_t cap) {
                const int64_t S = (tiles % cap) * kt;
                return static_cast<double>((tiles / cap) * kt + cdiv(S, sk_ctas(tiles, cap)));
            };
            // The hand-over cost of the tail finished inside the kernel.
            auto sk_handover = [&](int64_t tiles, int64_t cap) {
                const int64_t parts = cdiv(sk_ctas(tiles, cap), tiles % cap) + 1;
                return 2.0 + 0.26 * static_cast<double>(parts > 2 ? parts - 2 : 0);
            };
            const bool fix = cfg.fx != 0;
            const int64_t cap128 = static_cast<int64_t>(dev->ctas_per_sm[0][0]) * nsm;
            if (cap128 > 0) {
                offer(0, false, static_cast<double>(cdiv(tiles128, cap128)) * dkt + 1);
                if (sk_possible && tiles128 % cap128 != 0)
                    offer(0, true, sk_iters(tiles128, cap128) +
                                       (fix ? 6.0 : sk_handover(tiles128, cap128)));
            }
            if (tma_both) {
                if (dev->ctas_per_sm[2][mi_tt] >= 2)
                    offer(2, false,
                          tiles128x64 <= nsm
                              ? 0.63 * dkt
                              : static_cast<double>(cdiv(tiles128x64, 2 * nsm)) * 1.06 * dkt);
                const int64_t cap_k2 = static_cast<int64_t>(dev->ctas_per_sm[3][mi_tt]) * nsm;
                if (cap_k2 > 0) {
                    offer(3, false, static_cast<double>(cdiv(tiles128x64, cap_k2)) * 0.54 * dkt);
                    if (sk_possible && !fix && tiles128x64 % cap_k2 != 0)
                        offer(3, true, sk_iters(tiles128x64, cap_k2) * 0.54 +
                                           sk_handover(tiles128x64, cap_k2));
                }
                const int64_t cap_k4 = static_cast<int64_t>(dev->ctas_per_sm[4][mi_tt]) * nsm;
                if (cap_k4 > 0) {
                    offer(4, false, static_cast<double>(cdiv(tiles64, cap_k4)) * 0.31 * dkt);
                    if (sk_possible && tiles64 % cap_k4 != 0)
                        offer(4, true, sk_iters(tiles64, cap_k4) * 0.31 +
                                           (fix ? 4.0 : sk_handover(tiles64, cap_k4)));
                }
                // The same tile in clusters of cs CTAs that split each tile's
                // k-tiles: a cs-th of the k-loop per CTA, plus the hand-over of
                // the partial sums through distributed shared memory (~0.8
                // units with 2 CTAs, ~1.25 with 4). Only when all the
                // clusters run at once: a second wave of clusters measured
                // slower than the plain tile (640^3: 30.8 against 20.9 us).
                for (int f = 5; f <= 6; ++f) {
                    const int64_t cs = registry().fam[f]->cs;
                    const int64_t ncl = dev->clusters[f][mi_tt];
                    if (dev->ctas_per_sm[f][mi_tt] <= 0 || tiles64 > ncl) continue;
                    offer(f, false,
                          0.31 * static_cast<double>(cdiv(kt, cs)) + (cs == 2 ? 0.8 : 1.25));
                }
            }
            fi = best_f;
            if (!best_sk) allow_sk = false;
        }
    }
    const KernelFamily* fam = registry().fam[fi];
    pl->fam = fam;
    const int bm = fam->bm, bn = fam->bn, bk = 32;
    const bool force_cp = force_cp_flag != 0;
    // How a row-major A reaches the consumers. The transposed-A read
    // ([BK][BM] stages, two float4 per lane and k-step) keeps the FMA pipe
    // busier than the row-major read (90 % against 83 % of active cycles at
    // 4096^3 on GB300). Two ways to get there: a transposed copy of A in the
    // workspace ("a_pre", then the transposed-A kernel), or the in-smem
    // transpose (mode 6, transposer warps in the kernel, no copy), possible
    // for an A TMA can read in place, when B goes by TMA too and the family
    // has the variant.
    const bool b_will_tma = pl->b_t ? true : (tma_ok(B, ldb, K, N) || (allow_pack && M >= 256));
    const bool xp_possible = !pl->a_t && !force_cp && tma_ok(A, lda, M, K) && b_will_tma &&
                             dev->ctas_per_sm[fi][mode_index(LOAD_TMA_XP, LOAD_TMA)] > 0;
    // Either way beats reading the row-major A as stored. Measured on GB300
    // against that: the HBM copy saves ~8.5 % of the main loop (2MNK FLOP at
    // ~66 TFLOP/s), ~3.6 % more than the in-smem transpose, but costs ~5 us
    // of launch and allocation plus one read and one write of A at ~6 TB/s.
    // "auto" takes the copy where its extra saving pays for it, else the
    // in-smem transpose where possible (not for the two-CTA 128 x 64 tile,
    // where it gains nothing).
    const double mk = static_cast<double>(M) * static_cast<double>(K);
    const double t_main = 2.0 * mk * static_cast<double>(N) / 66e12;
    const double copy_cost = 5e-6 + 8.0 * mk / 6e12;
    const bool copy_ok = !pl->a_t && allow_pack && !force_cp;
    // The transposer warps add a step between a stage landing and its use,
    // which a work item of fewer than 4 k-iterations does not hide: 256^3 in
    // clusters of 4 CTAs (2 k-iterations each) took 11.0 us with it and
    // 10.3 us reading the row-major A (GB300); from 8 k-iterations on the
    // two were even or the transpose ahead (640^3: 21.3 against 22.6 us).
    const int64_t item_kt = ((K + 31) / 32 + fam->cs - 1) / fam->cs;
    const bool xp_auto = xp_possible && fi != 2 && item_kt >= 4;
    pl->a_pre = false;
    pl->a_xp = false;
    if (cfg.at == 1 || cfg.at == 3) {
        pl->a_pre = copy_ok;
    } else if (cfg.at == 2) {
        pl->a_xp = xp_possible;
    } else if (cfg.at < 0) {
        if (xp_auto) {
            pl->a_pre = copy_ok && 0.036 * t_main > copy_cost;
            pl->a_xp = !pl->a_pre;
        } else {
            pl->a_pre = copy_ok && 0.085 * t_main > copy_cost;
        }
        // A row-major A that TMA cannot read in place and that would be
        // copied to an aligned buffer anyway (N >= 256, below) is better
        // copied transposed: the same one HBM pass, then the transposed-A
        // read (GB300: 1024x1024x1023 50.5 against 51.6 us, 768x768x767
        // 28.7 against 29.8 us, 2048x1024x1023 80.0 against 84.2 us), where
        // the main loop is long enough for its ~8.5 % to matter (0.085
        // t_main > 1 us); on shorter ones the transposed copy came out slower
        // (300x512x1001: 24.6 against 22.6 us).
        const bool a_packs_anyway =
            !pl->a_t && allow_pack && !force_cp && N >= 256 && !tma_ok(A, lda, M, K);
        if (a_packs_anyway && 0.085 * t_main > 1e-6) pl->a_pre = copy_ok;
    }
    std::memset(&pl->tmA, 0, sizeof(CUtensorMap));
    std::memset(&pl->tmB, 0, sizeof(CUtensorMap));
    int a_mode = LOAD_CPASYNC, b_mode = LOAD_CPASYNC;
    pl->pack_a = pl->pack_b = false;
    pl->pack_a_bytes = pl->pack_b_bytes = 0;
    // Copies are described to the driver against a placeholder address first
    // (to make sure it accepts the shape) and encoded again on the real
    // workspace buffer at launch.
    const float* kPlaceholder = reinterpret_cast<const float*>(uintptr_t{1} << 20);
    pl->a_fused = false;
    pl->at_flags_off = 0;
    if (pl->a_pre) {
        const int64_t ld = (M + 3) & ~int64_t{3};
        if (tma_ok(kPlaceholder, ld, K, M) &&
            encode_2d(&pl->tmA, kPlaceholder, K, M, ld, bk, bm, false)) {
            a_mode = LOAD_TMA;
            pl->pack_a = true;
            pl->lda_pack = ld;
            pl->pack_a_bytes = align256(static_cast<size_t>(K) * static_cast<size_t>(ld) * 4);
        } else {
            pl->a_pre = false;
        }
    }
    if (pl->a_pre) {
        // (A is loaded from the transposed copy.)
    } else if (!pl->a_t) {
        if (!force_cp && tma_ok(A, lda, M, K) && encode_2d(&pl->tmA, A, M, K, lda, bm, bk, true))
            a_mode = LOAD_TMA;
    } else {
        // Transposed A (stored K x M): [BK][BM] boxes, no swizzle, TMA only
        // (":cpasync" does not apply to it).
        if (tma_ok(A, lda, K, M) && encode_2d(&pl->tmA, A, K, M, lda, bk, bm, false))
            a_mode = LOAD_TMA;
    }
    if (!pl->b_t && !force_cp && tma_ok(B, ldb, K, N) &&
        encode_2d(&pl->tmB, B, K, N, ldb, bk, bn, false))
        b_mode = LOAD_TMA;
    // An operand TMA cannot describe in place is copied once to an aligned
    // buffer when the GEMM reads it often enough (A is read once per
    // 128-column tile of C, B once per 128-row tile): from 256 columns (rows)
    // the 4-byte cp.async loads it saves cost more than the extra pass. A
    // transposed A has no cp.async path, so it is always copied then.
    if (!pl->a_t && !pl->a_pre && a_mode != LOAD_TMA && allow_pack && !force_cp && N >= 256) {
        const int64_t ld = (K + 3) & ~int64_t{3};
        if (tma_ok(kPlaceholder, ld, M, K) && encode_2d(&pl->tmA, kPlaceholder, M, K, ld, bm, bk, true)) {
            a_mode = LOAD_TMA;
            pl->pack_a = true;
            pl->lda_pack = ld;
            pl->pack_a_bytes = align256(static_cast<size_t>(M) * static_cast<size_t>(ld) * 4);
        }
    }
    if (pl->a_t && a_mode != LOAD_TMA) {
        if (!allow_pack) return cuda_fail(cudaErrorMemoryAllocation, SGEMM_ERR_CUDA);
        const int64_t ld = (M + 3) & ~int64_t{3};
        if (!(tma_ok(kPlaceholder, ld, K, M) &&
              encode_2d(&pl->tmA, kPlaceholder, K, M, ld, bk, bm, false)))
            return cuda_fail(cudaErrorInvalidValue, SGEMM_ERR_LAUNCH);
        a_mode = LOAD_TMA;
        pl->pack_a = true;
        pl->lda_pack = ld;
        pl->pack_a_bytes = align256(static_cast<size_t>(K) * static_cast<size_t>(ld) * 4);
    }
    if (pl->b_t) {
        // Transposed B (stored N x K): transposed once into a row-major K x N
        // buffer. Read in place it would sit in shared memory as [BN][BK],
        // and the packed FFMA2 needs two adjacent columns at one k in one
        // register pair; the copy costs one HBM pass of B instead.
        if (!allow_pack) return cuda_fail(cudaErrorMemoryAllocation, SGEMM_ERR_CUDA);
        const int64_t ld = (N + 3) & ~int64_t{3};
        pl->pack_b = true;
        pl->ldb_pack = ld;
        pl->pack_b_bytes = align256(static_cast<size_t>(K) * static_cast<size_t>(ld) * 4);
        if (!force_cp && tma_ok(kPlaceholder, ld, K, N) &&
            encode_2d(&pl->tmB, kPlaceholder, K, N, ld, bk, bn, false))
            b_mode = LOAD_TMA;
    } else if (b_mode != LOAD_TMA && allow_pack && !force_cp && M >= 256) {
        const int64_t ld = (N + 3) & ~int64_t{3};
        if (tma_ok(kPlaceholder, ld, K, N) && encode_2d(&pl->tmB, kPlaceholder, K, N, ld, bk, bn, false)) {
            b_mode = LOAD_TMA;
            pl->pack_b = true;
            pl->ldb_pack = ld;
            pl->pack_b_bytes = align256(static_cast<size_t>(K) * static_cast<size_t>(ld) * 4);
        }
    }
    if (pl->a_xp) {
        if (a_mode == LOAD_TMA && b_mode == LOAD_TMA) a_mode = LOAD_TMA_XP;
        else pl->a_xp = false;
    }
    int mi = mode_index(a_mode, b_mode, (pl->a_t || pl->a_pre) ? 1 : 0);
    // The transposed copy made inside the GEMM kernel, where the family has
    // that mode with the same CTAs per SM (so grid and schedule are those of
    // the copy by a separate kernel) and ":atcopy" does not ask otherwise:
    // the copy's ~20-28 us at 4096^3 then overlap the first tiles' work. The
    // flags (one per unit of BK k-rows x BM columns) follow the copy.
    // The same for the row-major copy of a transposed B, when A is read
    // through the transposed-A path anyway (its copy made here too, or A
    // given transposed and read in place). Both only with a first wave of
    // whole tiles: the tail's CTAs start all along the k-range at once and
    // would wait for units the round-robin has not reached (1024^3 forced to
    // it: 62.6 against 47.5 us).
    pl->b_fused = false;
    pl->bt_flags_off = 0;
    const int64_t tiles_all = ((M + bm - 1) / bm) * ((N + bn - 1) / bn);
    const bool fuse_ok = cfg.at != 3 && b_mode == LOAD_TMA &&
                         dev->ctas_per_sm[fi][kModeFused] > 0 &&
                         dev->ctas_per_sm[fi][kModeFused] == dev->ctas_per_sm[fi][mi] &&
                         tiles_all >= static_cast<int64_t>(dev->ctas_per_sm[fi][kModeFused]) * sms;
    if (fuse_ok && pl->a_pre) {
        const size_t units = static_cast<size_t>((M + bm - 1) / bm) *
                             static_cast<size_t>((K + bk - 1) / bk);
        pl->a_fused = true;
        pl->at_flags_off = pl->pack_a_bytes;
        pl->pack_a_bytes += align256(units * 8);
        mi = kModeFused;
    }
    if (fuse_ok && pl->b_t && pl->pack_b &&
        (pl->a_fused || (pl->a_t && !pl->pack_a && a_mode == LOAD_TMA))) {
        const size_t units = static_cast<size_t>((N + bn - 1) / bn) *
                             static_cast<size_t>((K + bk - 1) / bk);
        pl->b_fused = true;
        pl->bt_flags_off = pl->pack_b_bytes;
        pl->pack_b_bytes += align256(units * 8);
        mi = kModeFused;
    }
    pl->k = &fam->modes[mi];

    GemmParams& p = pl->p;
    std::memset(&p, 0, sizeof(p));
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.tiles_m = static_cast<int>((M + bm - 1) / bm);
    p.tiles_n = static_cast<int>((N + bn - 1) / bn);
    p.k_tiles = static_cast<int>((K + bk - 1) / bk);
    // Tile rows per raster group. The time hardly depends on it (8, 16 and 32
    // within 0.1 % at 4096^3, 8192x14336x4096 and 4093x5120x1531 on GB300),
    // the DRAM traffic does: at 4096^3 one launch read 318 MB with 8, 273 MB
    // with 16 (B's column blocks are re-read once per group) and 521 MB with
    // 32 (the whole of A per wave no longer stays in L2).
    p.group_m = 16;
    p.c_vec = (aligned(C, 16) && (ldc % 4) == 0) ? 1 : 0;
    p.A = A;
    p.B = B;
    p.C = const_cast<float*>(C);
    p.lda = lda;
    p.ldb = ldb;
    p.ldc = ldc;
    p.alpha = alpha;
    p.beta = beta;
    p.timeout_ns = g_timeout_ns.load();
    const int64_t tiles = static_cast<int64_t>(p.tiles_m) * p.tiles_n;
    if (tiles > 0x7fffffffll) return SGEMM_ERR_INVALID_VALUE;
    if (dev->ctas_per_sm[fi][mi] <= 0) return cuda_fail(cudaErrorInvalidConfiguration, SGEMM_ERR_LAUNCH);
    const int64_t cap = static_cast<int64_t>(dev->ctas_per_sm[fi][mi]) * sms;
    if (fam->cs > 1) {
        // One tile per cluster of fam->cs CTAs (each a share of its k-tiles),
        // clusters in as many waves as it takes; no stream-K tail.
        const int64_t g = tiles * fam->cs;
        if (g > 0x7fffffffll) return SGEMM_ERR_INVALID_VALUE;
        p.dp_tiles = static_cast<int>(tiles);
        p.sk_ctas = 0;
        p.sk_iters = 0;
        pl->grid = static_cast<int>(g);
        pl->sk_tiles = 0;
        pl->sk_bytes = 0;
        pl->ws_bytes = pl->pack_a_bytes + pl->pack_b_bytes;
        return SGEMM_OK;
    }

    // Schedule: whole waves data-parallel; the last, partial wave's
    // k-iterations spread over the CTAs (stream-K) unless it is nearly full.
    const int64_t waves = tiles / cap, rest = tiles % cap;
    const bool use_sk = allow_sk && force_sk != 0 && rest != 0 &&
                        (sk_decided || waves == 0 || rest * 10 < cap * 9);
    if (!use_sk) {
        p.dp_tiles = static_cast<int>(tiles);
        p.sk_ctas = 0;
        p.sk_iters = 0;
        pl->grid = static_cast<int>(tiles < cap ? tiles : cap);
        pl->sk_tiles = 0;
        pl->sk_bytes = 0;
        pl->ws_bytes = pl->pack_a_bytes + pl->pack_b_bytes;
        return SGEMM_OK;
    }
    const int64_t S = rest * p.k_tiles;
    // A range is at least k_tiles / 32 iterations long, so no tile has more
    // than 34 partial segments (the fixup handles up to kSkMaxParts).
    const int64_t min_len = (p.k_tiles + 31) / 32;
    int64_t G = S / min_len;
    if (G > cap) G = cap;
    if (G < 1) G = 1;
    p.dp_tiles = static_cast<int>(waves * cap);
    p.sk_ctas = static_cast<int>(G);
    p.sk_iters = S;
    p.sk_fixup = pl->sk_fixup ? 1 : 0;
    pl->grid = static_cast<int>(waves > 0 ? cap : G);
    pl->sk_tiles = static_cast<int>(rest);
    // Slots of BM x BN floats: one per CTA when split tiles are finished in
    // the kernel (followed by one 8-byte flag per CTA), two per CTA for the
    // fixup kernel.
    const size_t slot_bytes = static_cast<size_t>(bm) * bn * sizeof(float);
    pl->sk_bytes = pl->sk_fixup ? static_cast<size_t>(2 * G) * slot_bytes
                                : static_cast<size_t>(G) * slot_bytes +
                                      align256(static_cast<size_t>(G) * 8);
    pl->ws_bytes = pl->pack_a_bytes + pl->pack_b_bytes + pl->sk_bytes;
    return SGEMM_OK;
}

int launch_plan(Plan* pl, int* status, float* ws, cudaStream_t stream) {
    cudaError_t e = cudaSuccess;
    if (pl->kind == 0) return SGEMM_OK;
    if (pl->kind == 1) {
        const GemmParams& p = pl->p;
        const int bx = p.N < 256 * 16 ? (p.N + 255) / 256 : 16;
        const int by = p.M < 4096 ? p.M : 4096;
        scale_kernel<<<dim3(bx, by), 256, 0, stream>>>(p.C, p.ldc, p.M, p.N, p.beta);
        e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, SGEMM_ERR_LAUNCH);
        return SGEMM_OK;
    }
    pl->p.status = status;
    if (pl->ws_bytes > 0 && ws == nullptr) return SGEMM_ERR_INVALID_VALUE;
    unsigned char* w = reinterpret_cast<unsigned char*>(ws);
    GemmParams& p = pl->p;
    const int pack_grid = 16 * (pl->sms > 0 ? pl->sms : 1);
    // True once a kernel of this call is on the stream: the next one may
    // then be launched by programmatic serialisation behind it.
    const bool pdl = pdl_enabled();
    bool prior = false;
    p.at_src = nullptr;
    p.at_lds = 0;
    p.at_flags = nullptr;
    p.at_tag = 0;
    p.bt_src = nullptr;
    p.bt_lds = 0;
    p.bt_flags = nullptr;
    if (pl->a_fused || pl->b_fused) {
        unsigned long long tag = g_sk_tag.fetch_add(1);
        if (tag == 0) tag = g_sk_tag.fetch_add(1);   // after a wrap-around
        p.at_tag = tag;
    }
    if (pl->pack_a) {
        float* a2 = reinterpret_cast<float*>(w);
        if (pl->a_pre && pl->a_fused) {
            // The GEMM kernel's transposer warps write the transpose of the
            // row-major A (M x K) into a2 (K x lda_pack) themselves.
            p.at_src = p.A;
            p.at_lds = p.lda;
            p.at_flags = reinterpret_cast<unsigned long long*>(w + pl->at_flags_off);
        } else if (pl->a_pre) {
            // Row-major A (M x K) -> its transpose (K x lda_pack).
            e = launch_transpose_pack(p.A, p.lda, a2, pl->lda_pack, p.M, p.K, stream, false);
        } else {
            // A transposed keeps its stored (K x M) layout in the copy.
            const int rows = pl->a_t ? p.K : p.M, cols = pl->a_t ? p.M : p.K;
            e = launch_kernel(pack_rows_kernel, dim3(pack_grid), dim3(256), 0, stream, false, 1,
                              p.A, p.lda, a2, pl->lda_pack, rows, cols);
        }
        if (e != cudaSuccess) return cuda_fail(e, SGEMM_ERR_LAUNCH);
        prior = !pl->a_fused;
        const bool kt = pl->a_t || pl->a_pre;
        const bool ok = kt ? encode_2d(&pl->tmA, a2, p.K, p.M, pl->lda_pack, 32, pl->fam->bm, false)
                           : encode_2d(&pl->tmA, a2, p.M, p.K, pl->lda_pack, pl->fam->bm, 32, true);
        if (!ok) return cuda_fail(cudaErrorInvalidValue, SGEMM_ERR_LAUNCH);
        p.A = a2;
        p.lda = pl->lda_pack;
    }
    if (pl->pack_b) {
        float* b2 = reinterpret_cast<float*>(w + pl->pack_a_bytes);
        if (pl->b_t && pl->b_fused) {
            // The GEMM kernel's transposer warps write the row-major copy of
            // B (stored N x K) into b2 (K x ldb_pack) themselves.
            p.bt_src = p.B;
            p.bt_lds = p.ldb;
            p.bt_flags = reinterpret_cast<unsigned long long*>(w + pl->pack_a_bytes +
                                                                 pl->bt_flags_off);
        } else if (pl->b_t) {
            // B stored N x K -> row-major K x ldb_pack.
            e = launch_transpose_pack(p.B, p.ldb, b2, pl->ldb_pack, p.N, p.K, stream,
                                      pdl && prior);
        } else {
            e = launch_kernel(pack_rows_kernel, dim3(pack_grid), dim3(256), 0, stream, pdl && prior,
                              1, p.B, p.ldb, b2, pl->ldb_pack, p.K, p.N);
        }
        if (e != cudaSuccess) return cuda_fail(e, SGEMM_ERR_LAUNCH);
        if (!pl->b_fused) prior = true;
        if (!encode_2d(&pl->tmB, b2, p.K, p.N, pl->ldb_pack, 32, pl->fam->bn, false))
            return cuda_fail(cudaErrorInvalidValue, SGEMM_ERR_LAUNCH);
        p.B = b2;
        p.ldb = pl->ldb_pack;
    }
    p.ws = pl->sk_bytes > 0
               ? reinterpret_cast<float*>(w + pl->pack_a_bytes + pl->pack_b_bytes)
               : nullptr;
    p.sk_flags = nullptr;
    p.sk_tag = 0;
    if (pl->sk_bytes > 0 && !pl->sk_fixup) {
        p.sk_flags = reinterpret_cast<unsigned long long*>(
            w + pl->pack_a_bytes + pl->pack_b_bytes +
            static_cast<size_t>(p.sk_ctas) * pl->fam->bm * pl->fam->bn * sizeof(float));
        unsigned long long tag = g_sk_tag.fetch_add(1);
        if (tag == 0) tag = g_sk_tag.fetch_add(1);   // after a wrap-around
        p.sk_tag = tag;
    }
    e = pl->k->launch(&pl->tmA, &pl->tmB, &pl->p, pl->grid, stream, pdl && prior);
    if (e == cudaSuccess && pl->sk_tiles > 0 && pl->sk_fixup) {
        // Enough fixup CTAs for about two per SM, at most 8 per tile.
        const int want = (2 * pl->sms + pl->sk_tiles - 1) / pl->sk_tiles;
        const int split = want < 1 ? 1 : (want > 8 ? 8 : want);
        e = pl->fam->fixup(&pl->p, pl->sk_tiles, split, stream);
    }
    if (e != cudaSuccess) return cuda_fail(e, SGEMM_ERR_LAUNCH);
    return SGEMM_OK;
}

void unfuse_plan(Plan* pl) {
    if (!pl->a_fused && !pl->b_fused) return;
    pl->a_fused = false;
    pl->b_fused = false;
    pl->k = &pl->fam->modes[mode_index(LOAD_TMA, LOAD_TMA, 1)];
}

void plan_name(const Plan& pl, char* buf, int buflen) {
    if (buf == nullptr || buflen <= 0) return;
    if (pl.kind == 0) std::snprintf(buf, static_cast<size_t>(buflen), "none");
    else if (pl.kind == 1) std::snprintf(buf, static_cast<size_t>(buflen), "scale");
    else std::snprintf(buf, static_cast<size_t>(buflen), "%s%s%s%s", pl.k->name,
                       pl.pack_a ? (pl.a_pre ? (pl.a_fused ? "+packATfused" : "+packAT") : "+packA")
                                 : "",
                       pl.pack_b ? (pl.b_t ? (pl.b_fused ? "+packBTfused" : "+packBT") : "+packB")
                                 : "",
                       pl.sk_tiles > 0 ? (pl.sk_fixup ? "+skfix" : "+sk") : "");
}

int device_memory_handles(const DeviceInfo* dev, int** status, cudaMemPool_t* pool) {
    DeviceMemory* mem = nullptr;
    const int rc = device_memory(dev, &mem);
    if (rc != SGEMM_OK) return rc;
    *status = mem->status;
    *pool = mem->pool;
    return SGEMM_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() { return g_encode; }

unsigned long long wait_timeout_ns() { return g_timeout_ns.load(); }

int launch_selftest_wait(unsigned long long timeout_ns, int* status, cudaStream_t stream) {
    GemmParams p;
    std::memset(&p, 0, sizeof(p));
    p.timeout_ns = timeout_ns;
    p.status = status;
    wait_timeout_kernel<<<1, 32, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, SGEMM_ERR_LAUNCH);
    return SGEMM_OK;
}

}  // namespace sg

using namespace sg;

namespace {

int run_sgemm(int opa, int opb, int64_t M, int64_t N, int64_t K, float alpha, const float* A,
              int64_t lda, const float* B, int64_t ldb, float beta, float* C, int64_t ldc,
              cudaStream_t stream) {
    int rc = check_args_ex(opa, opb, M, N, K, alpha, A, lda, B, ldb, C, ldc);
    if (rc != SGEMM_OK) return rc;
    if (M == 0 || N == 0) return SGEMM_OK;
    const DeviceInfo* dev = nullptr;
    if ((rc = device_info(&dev)) != SGEMM_OK) return rc;
    DeviceMemory* mem = nullptr;
    if ((rc = device_memory(dev, &mem)) != SGEMM_OK) return rc;
    Plan pl;
    if ((rc = make_plan_ex(dev, opa, opb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, true, true,
                           &pl)) != SGEMM_OK)
        return rc;
    float* ws = nullptr;
    if (pl.ws_bytes > 0) {
        // Stream-ordered workspace (packed operands, stream-K slots) from the
        // library's pool: concurrent calls on different streams never share
        // it, and stream capture records it as an allocation node.
        void* w = nullptr;
        if (cudaMallocFromPoolAsync(&w, pl.ws_bytes, mem->pool, stream) != cudaSuccess) {
            (void)cudaGetLastError();
            if ((rc = make_plan_ex(dev, opa, opb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                                   false, false, &pl)) != SGEMM_OK)
                return rc;
        } else {
            ws = static_cast<float*>(w);
        }
    }
    if (pl.a_fused || pl.b_fused) {
        // A graph replays its flag value: with the fused copy a replay could
        // take the previous run's flags for its own, so a call being captured
        // makes the copy with a kernel of its own.
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
            (void)cudaGetLastError();
            cap = cudaStreamCaptureStatusActive;
        }
        if (cap != cudaStreamCaptureStatusNone) unfuse_plan(&pl);
    }
    rc = launch_plan(&pl, mem->status, ws, stream);
    if (ws != nullptr) cudaFreeAsync(ws, stream);
    return rc;
}

int plan_sgemm(int opa, int opb, int64_t M, int64_t N, int64_t K, float alpha, const float* A,
               int64_t lda, const float* B, int64_t ldb, float beta, const float* C, int64_t ldc,
               char* buf, int buflen, int* grid) {
    int rc = check_args_ex(opa, opb, M, N, K, alpha, A, lda, B, ldb, C, ldc);
    if (rc != SGEMM_OK) return rc;
    Plan pl;
    if (M != 0 && N != 0) {
        const DeviceInfo* dev = nullptr;
        if ((rc = device_info(&dev)) != SGEMM_OK) return rc;
        if ((rc = make_plan_ex(dev, opa, opb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, true,
                               true, &pl)) != SGEMM_OK)
            return rc;
    }
    plan_name(pl, buf, buflen);
    if (grid != nullptr) *grid = pl.kind == 2 ? pl.grid : 0;
    return SGEMM_OK;
}

}  // namespace

extern "C" int sgemm(int64_t M, int64_t N, int64_t K, float alpha, const float* A, int64_t lda,
                     const float* B, int64_t ldb, float beta, float* C, int64_t ldc,
                     cudaStream_t stream) {
    return run_sgemm(0, 0, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
}

extern "C" int sgemm_ex(int opa, int opb, int64_t M, int64_t N, int64_t K, float alpha,
                        const float* A, int64_t lda, const float* B, int64_t ldb, float beta,
                        float* C, int64_t ldc, cudaStream_t stream) {
    return run_sgemm(opa, opb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
}

extern "C" int sgemm_plan(int64_t M, int64_t N, int64_t K, float alpha, const float* A,
                          int64_t lda, const float* B, int64_t ldb, float beta, const float* C,
                          int64_t ldc, char* buf, int buflen, int* grid) {
    return plan_sgemm(0, 0, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, buf, buflen, grid);
}

extern "C" int sgemm_plan_ex(int opa, int opb, int64_t M, int64_t N, int64_t K, float alpha,
                             const float* A, int64_t lda, const float* B, int64_t ldb, float beta,
                             const float* C, int64_t ldc, char* buf, int buflen, int* grid) {
    return plan_sgemm(opa, opb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, buf, buflen, grid);
}

extern "C" int sgemm_check_status(cudaStream_t stream, int* bits) {
    const DeviceInfo* dev = nullptr;
    int rc = device_info(&dev);
    if (rc != SGEMM_OK) return rc;
    DeviceMemory* mem = nullptr;
    if ((rc = device_memory(dev, &mem)) != SGEMM_OK) return rc;
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, SGEMM_ERR_CUDA);
    int v = 0;
    if ((e = cudaMemcpyAsync(&v, mem->status, sizeof(int), cudaMemcpyDeviceToHost, stream)) != cudaSuccess ||
        (e = cudaMemsetAsync(mem->status, 0, sizeof(int), stream)) != cudaSuccess ||
        (e = cudaStreamSynchronize(stream)) != cudaSuccess)
        return cuda_fail(e, SGEMM_ERR_CUDA);
    if (bits != nullptr) *bits = v;
    return status_code(v);
}

extern "C" const char* sgemm_error_string(int code) {
    switch (code) {
        case SGEMM_OK: return "success";
        case SGEMM_ERR_INVALID_VALUE: return "invalid argument";
        case SGEMM_ERR_UNSUPPORTED_DEVICE: return "unsupported device (need compute capability 10.3)";
        case SGEMM_ERR_LAUNCH: return "kernel launch failed";
        case SGEMM_ERR_DEVICE_TIMEOUT: return "a bounded wait inside a kernel timed out";
        case SGEMM_ERR_CUDA: return "CUDA runtime error";
        case SGEMM_ERR_DEVICE_CHECK: return "a device-side schedule or index check failed";
        default: return "unknown error code";
    }
}

extern "C" int sgemm_last_cuda_error(void) { return t_last_cuda_error; }

extern "C" int sgemm_set_config(const char* name) {
    Config c;
    int rc = parse_config(name, &c);
    if (rc != SGEMM_OK) return rc;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        g_env_read = true;   // an explicit choice overrides the environment
    }
    set_global_config(c);
    return SGEMM_OK;
}

extern "C" int sgemm_set_shape_config(int64_t M, int64_t N, int64_t K, const char* name) {
    if (M < 0 || N < 0 || K < 0) return SGEMM_ERR_INVALID_VALUE;
    Config c;
    if (name != nullptr) {
        const int rc = parse_config(name, &c);
        if (rc != SGEMM_OK) return rc;
    }
    std::lock_guard<std::mutex> lock(g_rules_mu);
    int slot = -1;
    for (int i = 0; i < g_nrules; ++i)
        if (g_rules[i].M == M && g_rules[i].N == N && g_rules[i].K == K) slot = i;
    if (c.is_auto()) {
        // "auto" (or NULL) removes the rule.
        if (slot >= 0) g_rules[slot] = g_rules[--g_nrules];
        return SGEMM_OK;
    }
    if (slot < 0) {
        if (g_nrules == kMaxShapeRules) return SGEMM_ERR_INVALID_VALUE;
        slot = g_nrules++;
    }
    g_rules[slot] = ShapeRule{M, N, K, c};
    return SGEMM_OK;
}

extern "C" int sgemm_clear_shape_configs(void) {
    std::lock_guard<std::mutex> lock(g_rules_mu);
    g_nrules = 0;
    return SGEMM_OK;
}

extern "C" int sgemm_config_names(char* buf, int buflen) {
    if (buf == nullptr || buflen <= 0) return SGEMM_ERR_INVALID_VALUE;
    const Registry& r = registry();
    size_t used = 0;
    buf[0] = '\0';
    for (int i = 0; i < r.count; ++i) {
        const size_t n = std::strlen(r.fam[i]->name);
        if (used + n + 2 > static_cast<size_t>(buflen)) return SGEMM_ERR_INVALID_VALUE;
        if (i > 0) buf[used++] = ',';
        std::memcpy(buf + used, r.fam[i]->name, n);
        used += n;
        buf[used] = '\0';
    }
    return SGEMM_OK;
}

extern "C" int sgemm_set_wait_timeout_ns(uint64_t ns) {
    if (ns < 1000) return SGEMM_ERR_INVALID_VALUE;
    g_timeout_ns = ns;
    return SGEMM_OK;
}

extern "C" int sgemm_selftest_wait_timeout(uint64_t timeout_ns, cudaStream_t stream) {
    if (timeout_ns < 1000 || timeout_ns > 10000000000ull) return SGEMM_ERR_INVALID_VALUE;
    const DeviceInfo* dev = nullptr;
    int rc = device_info(&dev);
    if (rc != SGEMM_OK) return rc;
    DeviceMemory* mem = nullptr;
    if ((rc = device_memory(dev, &mem)) != SGEMM_OK) return rc;
    return launch_selftest_wait(timeout_ns, mem->status, stream);
}

// Used by fp32_peak.cu.
int sgemm_internal_device_ready() {
    const DeviceInfo* dev = nullptr;
    return device_info(&dev);
}
int sgemm_internal_sm_count() {
    const DeviceInfo* dev = nullptr;
    if (device_info(&dev) != SGEMM_OK) return 0;
    return dev->sm_count;
}
void sgemm_internal_set_cuda_error(int e) { t_last_cuda_error = e; }
