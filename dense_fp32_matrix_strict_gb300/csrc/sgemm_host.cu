// sgemm_host.cu — C = alpha * A * B + beta * C with A, B and C in HOST
// memory. The host<->device copies run on two library-owned streams and
// overlap the GEMMs of row blocks of C on the caller's stream:
//
//   h2d stream:  A block 0 (and C block 0 when beta != 0), B in column
//                chunks, then A block 1, ... each block into one of two
//                device buffers;
//   caller's stream: block 0's GEMM one column chunk at a time as B's chunks
//                land, then the GEMM of block i once its inputs have landed;
//   d2h stream:  block i of C back to the host once its GEMM is done.
//
// A block's buffers are reused two blocks later, after its GEMM (A) and its
// copy back (C) have finished. The call is ordered on the caller's stream
// like the device entry points: the copies start after the work already
// queued there, and the stream reaches the end of the call only when the
// last block of C is in host memory.
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "sgemm.h"
#include "sgemm_internal.h"

namespace sg {
namespace {

constexpr int kMaxHostDevices = 64;

struct CopyStreams {
    bool ready = false;
    cudaStream_t h2d = nullptr, d2h = nullptr;
};

std::mutex g_copy_mu;
CopyStreams g_copy[kMaxHostDevices];

// The two copy streams of the current device, created on first use.
int copy_streams(int dev, CopyStreams** out) {
    if (dev < 0 || dev >= kMaxHostDevices) return SGEMM_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_copy_mu);
    CopyStreams& c = g_copy[dev];
    if (!c.ready) {
        cudaError_t e = cudaStreamCreateWithFlags(&c.h2d, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&c.d2h, cudaStreamNonBlocking);
        if (e != cudaSuccess) {
            if (c.h2d != nullptr) cudaStreamDestroy(c.h2d);
            c.h2d = c.d2h = nullptr;
            return cuda_fail(e, SGEMM_ERR_CUDA);
        }
        c.ready = true;
    }
    *out = &c;
    return SGEMM_OK;
}

size_t align256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

int64_t round4(int64_t n) { return (n + 3) & ~int64_t{3}; }

// Events of one call; destroyed when the call returns (the driver releases
// an event still pending once it completes).
struct CallEvents {
    static constexpr int kCount = 23;
    cudaEvent_t ev[kCount] = {};
    int made = 0;
    cudaError_t create() {
        for (; made < kCount; ++made) {
            const cudaError_t e = cudaEventCreateWithFlags(&ev[made], cudaEventDisableTiming);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    ~CallEvents() {
        for (int i = 0; i < made; ++i) cudaEventDestroy(ev[i]);
    }
};

}  // namespace
}  // namespace sg

using namespace sg;

extern "C" int sgemm_host(int64_t M, int64_t N, int64_t K, float alpha, const float* A,
                          int64_t lda, const float* B, int64_t ldb, float beta, float* C,
                          int64_t ldc, cudaStream_t stream) {
    int rc = check_args(M, N, K, alpha, A, lda, B, ldb, C, ldc);
    if (rc != SGEMM_OK) return rc;
    if (M == 0 || N == 0) return SGEMM_OK;
    const DeviceInfo* dev = nullptr;
    if ((rc = device_info(&dev)) != SGEMM_OK) return rc;
    int* status = nullptr;
    cudaMemPool_t pool = nullptr;
    if ((rc = device_memory_handles(dev, &status, &pool)) != SGEMM_OK) return rc;
    CopyStreams* cs = nullptr;
    if ((rc = copy_streams(dev->device, &cs)) != SGEMM_OK) return rc;

    const bool reads_ab = alpha != 0.0f && K > 0;
    const bool reads_c = beta != 0.0f;
    // Row blocks: one for problems whose GEMM is too short to hide a copy
    // behind (below 5 GFLOP). Otherwise a short last block (128 to 256 rows,
    // taking any ragged rows), so little of C is left to copy back once the
    // last GEMM ends, and before it blocks of about 1024 rows (at most 8, of
    // mb rows each, a multiple of 128 so the GEMM tiles stay full), the first
    // one shorter where the rows do not divide evenly: the first GEMM starts
    // sooner. On GB300 at 4096^3 (768, 1024, 1024, 1024, 256 rows) this takes
    // ~60 us off the call against four blocks of 1024.
    constexpr int kMaxBlocks = 10;
    int64_t blk_r0[kMaxBlocks], blk_rows[kMaxBlocks];
    int nblk = 1;
    int64_t mb = M;
    blk_r0[0] = 0;
    blk_rows[0] = M;
    if (2.0 * static_cast<double>(M) * static_cast<double>(N) * static_cast<double>(K) >= 5e9 &&
        M >= 256) {
        const int64_t tail = (M % 128 == 0) ? (M >= 512 ? 256 : 128) : 128 + M % 128;
        const int64_t body = M - tail;                      // a multiple of 128, >= 0
        int64_t nb = (body + 1023) / 1024;
        if (nb > 8) nb = 8;
        nblk = 0;
        if (K >= 1024 && !reads_c && body >= 1024 + 768) {
            // The first block arrives in k-slabs (below), so its size no
            // longer delays the first GEMM: 1024 rows, then blocks of up to
            // 2048 (fewer GEMM calls), then 768 rows, whose C copies back
            // while the short last block computes. On GB300: 4096^3 (1024,
            // 2048, 768, 256 rows) 2.210 against 2.226 ms with 768, 3 x 1024,
            // 256; 8192 x 14336 x 4096 13.78 against 13.88 ms. Not when C is
            // read too: a block's buffers are refilled only after its C has
            // gone back, and a 2048-row C in and out takes longer than the
            // 768-row GEMM between them (4093 x 5120 x 1531 with beta != 0:
            // 1.567 against 1.434 ms).
            const int64_t mid = body - 1024 - 768;           // a multiple of 128, >= 0
            int64_t nm = (mid + 2047) / 2048;
            if (nm > kMaxBlocks - 3) nm = kMaxBlocks - 3;    // larger blocks past M ~ 16K
            const int64_t ms = nm > 0 ? ((mid + nm - 1) / nm + 127) / 128 * 128 : 0;
            int64_t r0 = 0;
            blk_r0[nblk] = r0;
            blk_rows[nblk++] = 1024;
            r0 += 1024;
            for (int64_t b = 0; b < nm; ++b) {
                const int64_t rows = (b + 1 < nm) ? ms : mid - (nm - 1) * ms;
                blk_r0[nblk] = r0;
                blk_rows[nblk++] = rows;
                r0 += rows;
            }
            blk_r0[nblk] = r0;
            blk_rows[nblk++] = 768;
            mb = ms > 1024 ? ms : 1024;
            nb = 0;
        } else if (nb > 0) {
            mb = ((body + nb - 1) / nb + 127) / 128 * 128;
            const int64_t head = body - (nb - 1) * mb;      // in (0, mb]
            blk_r0[nblk] = 0;
            blk_rows[nblk++] = head;
            for (int64_t b = 1; b < nb; ++b) {
                blk_r0[nblk] = head + (b - 1) * mb;
                blk_rows[nblk++] = mb;
            }
        } else {
            mb = tail;
        }
        blk_r0[nblk] = body;
        blk_rows[nblk++] = tail;
        if (mb < tail) mb = tail;                           // buffers hold any block
    }
    const int nbuf = nblk > 1 ? 2 : 1;

    // Device copies with leading dimensions rounded up to 4 floats, so that
    // TMA can read them in place.
    const int64_t ldk = round4(K > 0 ? K : 1), ldn = round4(N);
    const size_t b_bytes = reads_ab ? align256(static_cast<size_t>(K) * ldn * 4) : 0;
    const size_t a_bytes = reads_ab ? align256(static_cast<size_t>(mb) * ldk * 4) : 0;
    const size_t c_bytes = align256(static_cast<size_t>(mb) * ldn * 4);
    const size_t total = b_bytes + nbuf * (a_bytes + c_bytes);
    void* w = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&w, total, pool, stream);
    if (e != cudaSuccess) return cuda_fail(e, SGEMM_ERR_CUDA);
    unsigned char* base = static_cast<unsigned char*>(w);
    float* dB = reinterpret_cast<float*>(base);
    float* dA[2] = {reinterpret_cast<float*>(base + b_bytes),
                    reinterpret_cast<float*>(base + b_bytes + a_bytes)};
    float* dC[2] = {reinterpret_cast<float*>(base + b_bytes + nbuf * a_bytes),
                    reinterpret_cast<float*>(base + b_bytes + nbuf * a_bytes + c_bytes)};

    CallEvents evs;
    if ((e = evs.create()) != cudaSuccess) {
        cudaFreeAsync(w, stream);
        return cuda_fail(e, SGEMM_ERR_CUDA);
    }
    cudaEvent_t ev_start = evs.ev[0];
    cudaEvent_t ev_in[2] = {evs.ev[1], evs.ev[2]};      // block inputs landed
    cudaEvent_t ev_done[2] = {evs.ev[3], evs.ev[4]};    // block GEMM finished
    cudaEvent_t ev_out[2] = {evs.ev[5], evs.ev[6]};     // block of C back on the host
    cudaEvent_t* ev_part = evs.ev + 7;   // up to 16: B chunks or k-slabs landed
    // Block 0 starts before all of its inputs are on the device. With
    // several row blocks and K >= 1024 its A rows and B come in k-slabs (512
    // k each, whole k-tiles, at most 16 slabs) and its GEMM runs slab by slab,
    // adding each slab's product to C (beta on the first, 1 after): the first
    // GEMM starts once 512 k of A's first block and of B have landed (10 MB
    // at 4096^3) instead of the block's A and a quarter of B (29 MB). The
    // extra rounding of C between slabs stays inside the error bound. With
    // N >= 2048 and shorter K, B comes in 4 column chunks (whole multiples of
    // 128 columns) and block 0's GEMM runs chunk by chunk.
    const bool kslab = nblk > 1 && reads_ab && K >= 1024;
    int64_t ks = 512;
    if (kslab && (K + ks - 1) / ks > 16) ks = ((K + 15) / 16 + 31) / 32 * 32;
    const int nks = kslab ? static_cast<int>((K + ks - 1) / ks) : 0;
    int nbc = (!kslab && nblk > 1 && N >= 2048 && reads_ab) ? 4 : 1;
    int64_t nc = ((N + nbc - 1) / nbc + 127) / 128 * 128;
    if (nc > N) nc = N;
    nbc = static_cast<int>((N + nc - 1) / nc);

    // On an error part of the pipeline may already be queued on the copy
    // streams: join them into the caller's stream before the workspace goes
    // back to the pool, or, if even that fails, leave it allocated.
    auto release = [&]() {
        if (cudaEventRecord(ev_in[0], cs->h2d) == cudaSuccess &&
            cudaEventRecord(ev_out[0], cs->d2h) == cudaSuccess &&
            cudaStreamWaitEvent(stream, ev_in[0], 0) == cudaSuccess &&
            cudaStreamWaitEvent(stream, ev_out[0], 0) == cudaSuccess)
            cudaFreeAsync(w, stream);
    };
    auto fail = [&](cudaError_t err, int code) {
        release();
        return cuda_fail(err, code);
    };

    if ((e = cudaEventRecord(ev_start, stream)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(cs->h2d, ev_start, 0)) != cudaSuccess)
        return fail(e, SGEMM_ERR_CUDA);

    int last = 0;
    for (int i = 0; i < nblk; ++i) {
        const int j = i & 1;
        const int64_t r0 = blk_r0[i];
        const int64_t rows = blk_rows[i];
        if (i >= 2) {
            // Buffers j: block i - 2's GEMM has read A_j and written C_j, and
            // C_j has been copied back.
            if ((e = cudaStreamWaitEvent(cs->h2d, ev_done[j], 0)) != cudaSuccess ||
                (e = cudaStreamWaitEvent(cs->h2d, ev_out[j], 0)) != cudaSuccess)
                return fail(e, SGEMM_ERR_CUDA);
        }
        if (reads_ab && !(i == 0 && kslab) &&
            (e = cudaMemcpy2DAsync(dA[j], ldk * 4, A + r0 * lda, lda * 4, K * 4, rows,
                                   cudaMemcpyHostToDevice, cs->h2d)) != cudaSuccess)
            return fail(e, SGEMM_ERR_CUDA);
        if (reads_c &&
            (e = cudaMemcpy2DAsync(dC[j], ldn * 4, C + r0 * ldc, ldc * 4, N * 4, rows,
                                   cudaMemcpyHostToDevice, cs->h2d)) != cudaSuccess)
            return fail(e, SGEMM_ERR_CUDA);
        if ((e = cudaEventRecord(ev_in[j], cs->h2d)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(stream, ev_in[j], 0)) != cudaSuccess)
            return fail(e, SGEMM_ERR_CUDA);
        if (i >= 2 && (e = cudaStreamWaitEvent(stream, ev_out[j], 0)) != cudaSuccess)
            return fail(e, SGEMM_ERR_CUDA);
        if (i == 0 && kslab) {
            // A's first block and B in k-slabs; block 0's GEMM follows them
            // slab by slab.
            for (int sl = 0; sl < nks; ++sl) {
                const int64_t k0 = sl * ks;
                const int64_t kl = (K - k0) < ks ? (K - k0) : ks;
                if ((e = cudaMemcpy2DAsync(dA[j] + k0, ldk * 4, A + r0 * lda + k0, lda * 4, kl * 4,
                                           rows, cudaMemcpyHostToDevice, cs->h2d)) != cudaSuccess ||
                    (e = cudaMemcpy2DAsync(dB + k0 * ldn, ldn * 4, B + k0 * ldb, ldb * 4, N * 4, kl,
                                           cudaMemcpyHostToDevice, cs->h2d)) != cudaSuccess ||
                    (e = cudaEventRecord(ev_part[sl], cs->h2d)) != cudaSuccess ||
                    (e = cudaStreamWaitEvent(stream, ev_part[sl], 0)) != cudaSuccess)
                    return fail(e, SGEMM_ERR_CUDA);
                rc = sgemm(rows, N, kl, alpha, dA[j] + k0, ldk, dB + k0 * ldn, ldn,
                           sl == 0 ? beta : 1.0f, dC[j], ldn, stream);
                if (rc != SGEMM_OK) {
                    release();
                    return rc;
                }
            }
        } else if (i == 0 && reads_ab) {
            // B in column chunks behind block 0's inputs; block 0's GEMM
            // follows them chunk by chunk.
            for (int c = 0; c < nbc; ++c) {
                const int64_t c0 = c * nc;
                const int64_t cols = (N - c0) < nc ? (N - c0) : nc;
                if ((e = cudaMemcpy2DAsync(dB + c0, ldn * 4, B + c0, ldb * 4, cols * 4, K,
                                           cudaMemcpyHostToDevice, cs->h2d)) != cudaSuccess ||
                    (e = cudaEventRecord(ev_part[c], cs->h2d)) != cudaSuccess ||
                    (e = cudaStreamWaitEvent(stream, ev_part[c], 0)) != cudaSuccess)
                    return fail(e, SGEMM_ERR_CUDA);
                rc = sgemm(rows, cols, K, alpha, dA[j], ldk, dB + c0, ldn, beta, dC[j] + c0, ldn,
                           stream);
                if (rc != SGEMM_OK) {
                    release();
                    return rc;
                }
            }
        } else {
            rc = sgemm(rows, N, K, alpha, reads_ab ? dA[j] : nullptr, ldk,
                       reads_ab ? dB : nullptr, ldn, beta, dC[j], ldn, stream);
            if (rc != SGEMM_OK) {
                release();
                return rc;
            }
        }
        if ((e = cudaEventRecord(ev_done[j], stream)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(cs->d2h, ev_done[j], 0)) != cudaSuccess ||
            (e = cudaMemcpy2DAsync(C + r0 * ldc, ldc * 4, dC[j], ldn * 4, N * 4, rows,
                                   cudaMemcpyDeviceToHost, cs->d2h)) != cudaSuccess ||
            (e = cudaEventRecord(ev_out[j], cs->d2h)) != cudaSuccess)
            return fail(e, SGEMM_ERR_CUDA);
        last = j;
    }
    // The caller's stream passes the end of the call once the last block of
    // C (and, the d2h stream being in order, every earlier one) is back.
    if ((e = cudaStreamWaitEvent(stream, ev_out[last], 0)) != cudaSuccess)
        return fail(e, SGEMM_ERR_CUDA);
    if ((e = cudaFreeAsync(w, stream)) != cudaSuccess) return cuda_fail(e, SGEMM_ERR_CUDA);
    return SGEMM_OK;
}
