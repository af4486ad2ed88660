/*
 * sgemm.h — C ABI of the GB300 (sm_103a) strict-FP32 SGEMM library
 * (libsgemm_gb300.so).
 *
 * The operation is the one every page on hand-written FP32 SGEMM defines
 * ("Optimizing SGEMM in CUDA", section "What is a SGEMM?"; "The road to a
 * fast GEMM", section "The problem and the ceiling"):
 *
 *     C[i][j] = alpha * sum_{k<K} A[i][k] * B[k][j] + beta * C[i][j]
 *
 * with row-major A (M x K), B (K x N) and C (M x N). The argument order
 * follows those pages' kernels, (M, N, K, alpha, A, B, beta, C), with the
 * leading dimensions cuBLAS-style calls pass beside each matrix ("Optimizing
 * SGEMM in CUDA", section "cuBLAS implementation").
 *
 * Strictness: every product is accumulated by single-rounding FP32 FMAs on
 * the CUDA cores. No TF32, no reduced precision, no fast-math. Summation
 * order is not fixed, so results are not bit-identical to a sequential loop
 * on real-valued inputs; on integer-valued inputs whose partial sums stay
 * below 2^24 they are exact.
 *
 * All pointers are DEVICE pointers on the current CUDA device, owned by the
 * caller. The library keeps per-device set-up state (created on the first
 * call on a device: device properties, kernel attributes, a 256-byte device
 * status word and a private stream-ordered memory pool). Some calls take a
 * workspace from that pool with cudaMallocFromPoolAsync on the call's stream
 * and return it with cudaFreeAsync on the same stream (so concurrent calls
 * on different streams never share it and stream capture records it as an
 * allocation node): a problem whose last wave of tiles is split across all
 * SMs (the stream-K tail: one slot of BM x BN floats, at most 64 KB, and one
 * 8-byte flag per CTA; two slots per CTA when the configuration suffix
 * ":fixup" selects the separate fixup kernel); a row-major A large
 * enough that the kernel runs faster on its transpose (K x M floats, M
 * rounded up to 4, written by the GEMM kernel itself while its first tiles
 * run, with one 8-byte flag per 32 x 128 block of it; by a copy kernel
 * before it when the call is being captured into a CUDA graph); and an
 * operand that TMA cannot load in place (base or leading dimension not
 * 16-byte aligned) but that the kernel reads often enough (A when N >= 256,
 * B when M >= 256), copied to an aligned buffer (rows x cols rounded up to
 * 4 floats). If that allocation fails the call uses none of them.
 */
#ifndef SGEMM_GB300_H
#define SGEMM_GB300_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define SGEMM_API __attribute__((visibility("default")))
#else
#define SGEMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define SGEMM_OK 0
#define SGEMM_ERR_INVALID_VALUE 1      /* an argument violates the contract below      */
#define SGEMM_ERR_UNSUPPORTED_DEVICE 2 /* current device is not compute capability 10.3 */
#define SGEMM_ERR_LAUNCH 3             /* a kernel launch failed; see sgemm_last_cuda_error */
#define SGEMM_ERR_DEVICE_TIMEOUT 4     /* a bounded wait inside a kernel gave up          */
#define SGEMM_ERR_CUDA 5               /* another CUDA runtime call failed               */
#define SGEMM_ERR_DEVICE_CHECK 6       /* a kernel found a schedule or index invariant
                                          broken (index checks: debug build only)    */

/*
 * sgemm — C = alpha * A * B + beta * C (row-major, FP32).
 *
 *   M, N, K   problem size, each in [0, 2^31 - 1].
 *   alpha     scale of the product.
 *   A         M x K, element (i, k) at A[i * lda + k]; lda >= max(1, K).
 *   B         K x N, element (k, j) at B[k * ldb + j]; ldb >= max(1, N).
 *   beta      scale of the old C.
 *   C         M x N, element (i, j) at C[i * ldc + j]; ldc >= max(1, N);
 *             read (when beta != 0) and written in place.
 *   stream    CUDA stream the work is enqueued on (0 = legacy default).
 *
 * Layout and alignment: any leading dimension and any 4-byte-aligned base
 * pointer is accepted. Operands whose base is 16-byte aligned and whose
 * leading dimension is a multiple of 4 are loaded by TMA; others by 4-byte
 * cp.async. Elements between the end of a row and the next row (ld > width)
 * are never read or written.
 *
 * Readings (BLAS conventions; the pages always evaluate beta * C):
 *   - M == 0 or N == 0: nothing is done.
 *   - beta == 0: C is not read (NaN/Inf in C do not propagate).
 *   - alpha == 0 or K == 0: A and B are not read; C = beta * C (zeros if
 *     beta == 0).
 *
 * Errors: returns SGEMM_ERR_INVALID_VALUE, without enqueuing anything, if
 * M, N or K is negative or above 2^31 - 1; an ld is below its minimum or so
 * large that an offset overflows; A or B is NULL while alpha != 0 and K > 0;
 * C is NULL; a pointer is not 4-byte aligned; or the memory of A or B
 * overlaps the memory of C. SGEMM_ERR_UNSUPPORTED_DEVICE if the current
 * device is not sm_103. SGEMM_ERR_LAUNCH if the launch fails (the CUDA
 * error code is kept for sgemm_last_cuda_error).
 *
 * The call is asynchronous: it returns once the kernel is enqueued. Device
 * time-outs are reported later by sgemm_check_status. A, B and C must stay
 * valid until the stream reaches the kernel. A call enqueues one GEMM kernel,
 * preceded by up to two packing copies where its plan says so (sgemm_plan)
 * and, only with the ":fixup" configuration, followed by the stream-K fixup
 * kernel; a GEMM that follows a copy of the same call is launched with
 * programmatic stream serialisation (it waits for the copy on the device),
 * unless the environment variable SGEMM_PDL is "0" when the library first
 * launches.
 *
 * Sharing the GPU: the persistent kernels launch at most as many CTAs as
 * the GPU runs at once, and some CTAs wait (bounded) for others: the CTA
 * that finishes a split tile of the stream-K tail waits for the partial sums
 * of the CTAs that share the tile ("+sk"), and where the GEMM kernel makes
 * an operand copy itself ("+packATfused", "+packBTfused") a CTA waits for
 * blocks of the copy that any CTA may write. A kernel on another stream that
 * holds SMs while this one starts keeps some of its CTAs waiting for an SM
 * until that kernel ends; if that takes longer than the wait limit
 * (sgemm_set_wait_timeout_ns, 2 s by default), the result is incomplete and
 * sgemm_check_status returns SGEMM_ERR_DEVICE_TIMEOUT. Under the
 * configuration "auto:dp:atcopy" (sgemm_set_config) no CTA waits for
 * another (clusters are scheduled whole).
 *
 * Workspace: the pages' kernels need no scratch, so the plainest contract is
 * "nothing allocated per call". This entry point keeps a weaker one: no call
 * grows the library's device memory in steady state or waits to allocate.
 * Scratch (the transposed copy of A, an aligned copy of an operand, the
 * stream-K slots and flags) is borrowed from the library's stream-ordered
 * pool on `stream` and handed back on `stream`; the pool keeps what it
 * returns, so from the second call of a size on the borrow is a pool hit
 * (host bookkeeping only). Callers that can take no allocation at all use
 * sgemm_noalloc.
 */
SGEMM_API int sgemm(int64_t M, int64_t N, int64_t K, float alpha, const float* A, int64_t lda,
          const float* B, int64_t ldb, float beta, float* C, int64_t ldc,
          cudaStream_t stream);

/*
 * sgemm_host — the same operation, arguments and errors as sgemm, with A, B
 * and C in HOST memory (page-locked memory, from cudaHostAlloc or
 * cudaHostRegister, lets the copies overlap the computation; pageable memory
 * works but each copy then blocks). The library copies row blocks of A (and
 * of C when beta != 0) and B to the current device on a copy stream of its
 * own, runs the GEMM of each block on `stream`, and copies each finished
 * block of C back on a second copy stream, so the transfers of one block
 * overlap the GEMMs of others. Problems below 5 GFLOP run as one block.
 * Larger ones end on a short block (128 to 256 rows, taking any ragged rows
 * of M). With K >= 1024 the first block's A rows and B arrive in k-slabs of
 * 512 k and its GEMM runs slab by slab as they land (C then takes one extra
 * rounding per slab, inside the same error bound); with beta == 0 the blocks
 * are then 1024 rows, blocks of up to 2048, and 768 rows before the short
 * one. Otherwise B comes in column chunks behind the first block, whose GEMM
 * runs chunk by chunk, and the blocks are of about 1024 rows (at most 8),
 * the first of them shorter where the rows do not divide evenly. The device
 * buffers come from the library's stream-ordered pool (B, plus two A and
 * two C blocks: 4 (K N + 2 mb (K + N)) bytes, mb the largest block height;
 * SGEMM_ERR_CUDA if the pool cannot supply them). The call is asynchronous
 * and ordered on `stream`: the copies start after the work already queued
 * there, and `stream` passes the end of the call only when all of C is in
 * host memory, so a host read of C must follow a synchronisation of
 * `stream`. Host buffers must stay valid until then. Elements between rows
 * (ld > width) are never read or written. Not part of the pages' design: it
 * is this library's host-resident entry point.
 */
SGEMM_API int sgemm_host(int64_t M, int64_t N, int64_t K, float alpha, const float* A,
                         int64_t lda, const float* B, int64_t ldb, float beta, float* C,
                         int64_t ldc, cudaStream_t stream);

/* Operand transposition flags for the _ex entry points. */
#define SGEMM_OP_N 0   /* the operand as stored (row-major)        */
#define SGEMM_OP_T 1   /* the transpose of the stored matrix        */

/*
 * sgemm_ex — C = alpha * op(A) * op(B) + beta * C with cuBLAS-style
 * transposition flags, in this library's row-major convention. The pages'
 * kernels take square, untransposed, row-major operands only; the Tinyforge
 * README counts transposed operands among the generality cuBLAS offers and
 * its kernels leave out, and "The road to a fast GEMM" (benchmark harness)
 * calls cuBLAS through the transpose identity of row- and column-major
 * storage.
 *
 *   opa == SGEMM_OP_N: op(A) = A, stored M x K, (i, k) at A[i * lda + k],
 *                      lda >= max(1, K).
 *   opa == SGEMM_OP_T: op(A) = A^T, A stored K x M, op(A)(i, k) at
 *                      A[k * lda + i], lda >= max(1, M).
 *   opb == SGEMM_OP_N: op(B) = B, stored K x N, (k, j) at B[k * ldb + j],
 *                      ldb >= max(1, N).
 *   opb == SGEMM_OP_T: op(B) = B^T, B stored N x K, op(B)(k, j) at
 *                      B[j * ldb + k], ldb >= max(1, K).
 *
 * Everything else (sizes, C, readings, errors, asynchrony) is as for sgemm;
 * an opa or opb other than 0 or 1 returns SGEMM_ERR_INVALID_VALUE. A
 * transposed A is read by TMA in its stored layout when its base is 16-byte
 * aligned and lda % 4 == 0, else first copied (in that layout) to an aligned
 * workspace buffer; a transposed B is always transposed into a row-major
 * K x N workspace buffer (one HBM pass over B), by the GEMM kernel itself
 * when A goes through the transposed-A path, else by a copy kernel before
 * it. Those buffers come
 * from the library's stream-ordered pool like the stream-K workspace; if the
 * pool cannot supply one, the call returns SGEMM_ERR_CUDA with
 * cudaErrorMemoryAllocation kept for sgemm_last_cuda_error.
 * sgemm_ex(SGEMM_OP_N, SGEMM_OP_N, ...) is sgemm(...).
 */
SGEMM_API int sgemm_ex(int opa, int opb, int64_t M, int64_t N, int64_t K, float alpha,
                       const float* A, int64_t lda, const float* B, int64_t ldb, float beta,
                       float* C, int64_t ldc, cudaStream_t stream);

/*
 * sgemm_check_status — synchronise `stream`, then read and clear the current
 * device's status word. Returns SGEMM_OK, SGEMM_ERR_DEVICE_TIMEOUT if any
 * kernel since the last check gave up on a bounded wait (its output is then
 * incomplete), SGEMM_ERR_DEVICE_CHECK if a kernel found a schedule invariant
 * broken or, in the library built with -DSGEMM_DEBUG, an index check failed
 * (the result may then be wrong), or SGEMM_ERR_CUDA if the synchronisation
 * reported an error. If `bits` is not NULL it receives the raw status bits
 * (1: a consumer timed out, 2: a producer timed out, 4: draining copies
 * timed out, 8: a schedule invariant failed, 16: an index check failed).
 *
 * The debug build (libsgemm_gb300_debug.so, the package's build with
 * debug=True) compiles the same kernels with device-side checks of every
 * shared-memory, workspace and C index and of each work item against the
 * schedule; a failed check sets bit 16 and the kernel carries on (no trap),
 * so a test reads it here. It is slower and not meant for timing.
 */
SGEMM_API int sgemm_check_status(cudaStream_t stream, int* bits);

/* Human-readable text for a return code (static storage, never NULL). */
SGEMM_API const char* sgemm_error_string(int code);

/* The CUDA error code behind the last SGEMM_ERR_LAUNCH / SGEMM_ERR_CUDA
 * returned on this thread (0 if none). */
SGEMM_API int sgemm_last_cuda_error(void);

/*
 * sgemm_plan — describe, without launching, the kernel sgemm would use for
 * these arguments: writes a NUL-terminated name such as
 * "ws_128x128x32_s4_Atma_Btma" into buf (at most buflen bytes) and the
 * launch grid into *grid (if not NULL). "+packA" / "+packB" mean that
 * operand is first copied to an aligned buffer by a small copy kernel;
 * "+packAT" that A is first copied transposed by a copy kernel and read
 * through the transposed-A path ("_ATtma_" in the kernel name),
 * "+packATfused" that the GEMM kernel makes that copy itself; a "+sk"
 * suffix means the last wave is split across the SMs (stream-K) and
 * finished inside the GEMM kernel, "+skfix" by a second, small fixup
 * kernel. Returns the same argument errors as sgemm, or
 * SGEMM_OK. A name of "scale" means the alpha == 0 / K == 0 path; "none"
 * means M == 0 or N == 0.
 */
SGEMM_API int sgemm_plan(int64_t M, int64_t N, int64_t K, float alpha, const float* A, int64_t lda,
               const float* B, int64_t ldb, float beta, const float* C, int64_t ldc,
               char* buf, int buflen, int* grid);

/* sgemm_plan for sgemm_ex's arguments. A transposed A shows as "_ATtma_"
 * in the kernel name; "+packBT" means B is first transposed into a
 * row-major buffer by a copy kernel, "+packBTfused" that the GEMM kernel
 * makes that copy itself (when A is read through the transposed-A path). */
SGEMM_API int sgemm_plan_ex(int opa, int opb, int64_t M, int64_t N, int64_t K, float alpha,
                            const float* A, int64_t lda, const float* B, int64_t ldb, float beta,
                            const float* C, int64_t ldc, char* buf, int buflen, int* grid);

/*
 * sgemm_set_config — force a kernel configuration for later calls in this
 * process (for sweeps and tests). `name` is "auto" (default), "128x128",
 * "64x64" or "128x64" for the CTA tile, or one of the family names sgemm_config_names
 * lists, optionally followed by modifiers: ":cpasync" loads both operands
 * with cp.async even when TMA could be used (a transposed A excepted: it is
 * always loaded by TMA), ":dp" never splits the last
 * wave (plain data-parallel schedule), ":at" / ":noat" always / never
 * read a row-major A through a transposed copy (the default decides by
 * size; the 128 x 128 kernel makes the copy itself), ":atcopy" the same
 * copy (and that of a transposed B) made by a copy kernel first, ":xp" the
 * transpose in shared memory
 * instead, ":fixup" the stream-K tail finished by a second kernel, e.g.
 * "128x128:cpasync:dp" or "auto:dp". Returns SGEMM_ERR_INVALID_VALUE for an
 * unknown name. The environment variable SGEMM_FORCE_CONFIG, read on the
 * first call, sets the same thing.
 */
SGEMM_API int sgemm_set_config(const char* name);

/*
 * sgemm_config_names — write the names sgemm_set_config accepts besides
 * "auto", "128x128", "64x64" and "128x64" (every compiled kernel family, comma
 * separated, NUL-terminated) into buf (at most buflen bytes). Returns
 * SGEMM_ERR_INVALID_VALUE if buf is NULL or too small.
 */
SGEMM_API int sgemm_config_names(char* buf, int buflen);

/*
 * sgemm_set_shape_config — per-shape form of sgemm_set_config: later calls
 * whose (M, N, K) equal these use configuration `name` (same syntax as
 * sgemm_set_config) while the global configuration is "auto". `name` equal
 * to "auto", or NULL, removes the rule for that shape. Up to 256 shapes;
 * a new shape beyond that, a negative size or an unknown name returns
 * SGEMM_ERR_INVALID_VALUE. The pages note that the best tile depends on
 * the GPU and on the matrix shape and that libraries pick one per shape
 * ("The road to a fast GEMM", section "Where to go next", autotuning), and
 * the Tinyforge README sweeps tiles per size; this is where such a sweep's
 * choice is installed. The package's autotune module writes it.
 * sgemm_clear_shape_configs removes every rule. Thread-safe; affects calls
 * on every device.
 */
SGEMM_API int sgemm_set_shape_config(int64_t M, int64_t N, int64_t K, const char* name);
SGEMM_API int sgemm_clear_shape_configs(void);

/*
 * sgemm_set_wait_timeout_ns — limit on every bounded wait inside the
 * kernels launched after this call, on an mbarrier or on another CTA's flag
 * (default 2e9 ns). Values below 1000 ns are rejected with
 * SGEMM_ERR_INVALID_VALUE.
 */
SGEMM_API int sgemm_set_wait_timeout_ns(uint64_t ns);

/*
 * sgemm_fp32_peak — the pure-FFMA microbenchmark that measures the device's
 * real FP32 ceiling, as the Tinyforge README's fp32_peak does (its measured
 * 6,884 GFLOPS against a 9,100 GFLOPS datasheet figure). Every thread of a
 * grid of 8 CTAs of 256 threads per SM runs 8 independent FFMA chains; the
 * run is calibrated to last about target_ms (>= 1) and timed with CUDA
 * events on `stream` after one untimed warm-up launch of the same length.
 * Outputs (each may be NULL): *gflops = 2 * FMAs / time, *ms = time of
 * the timed launch, *flops = floating-point operations of the timed launch.
 * Blocking: synchronises `stream`.
 */
SGEMM_API int sgemm_fp32_peak(double target_ms, double* gflops, double* ms, double* flops,
                    cudaStream_t stream);

/* Instruction forms of the ceiling microbenchmark. */
#define SGEMM_PEAK_FFMA 0    /* scalar FFMA chains (what sgemm_fp32_peak runs)        */
#define SGEMM_PEAK_FFMA2 1   /* packed fma.rn.f32x2 chains, the form the SGEMM issues */
#define SGEMM_PEAK_OUTER 2   /* the SGEMM's register outer product, no memory access  */

/*
 * sgemm_fp32_peak_ex — sgemm_fp32_peak in a chosen instruction form. With
 * SGEMM_PEAK_FFMA2 every thread runs 8 independent chains of the packed
 * two-lane FMA (two single-rounding FP32 FMAs per instruction, 4 FLOP), the
 * instruction the SGEMM's inner loop is built from, so the ceiling is
 * measured on what the GEMM actually issues. Same grid, calibration, timing,
 * outputs and blocking as sgemm_fp32_peak. With SGEMM_PEAK_OUTER one CTA of
 * 8 warps per SM (two per scheduler, the 128 x 128 kernel's occupancy) runs
 * the GEMM's inner loop without its loads: each lane's 8 x 8 accumulators
 * take 32 packed FMAs per k-step in the kernel's order, on A and B values
 * held in registers (opaque to the compiler at every k-step); 128 FLOP per
 * lane and k-step. It is the rate that instruction mix reaches when shared
 * memory costs nothing, not a device peak. Another form returns
 * SGEMM_ERR_INVALID_VALUE.
 */
SGEMM_API int sgemm_fp32_peak_ex(int form, double target_ms, double* gflops, double* ms,
                                 double* flops, cudaStream_t stream);

/*
 * sgemm_tf32_mma_peak — the TF32 tensor-core ceiling that sgemm_3xtf32 is
 * measured against: one CTA per SM issues back-to-back
 * tcgen05.mma.kind::tf32 instructions of the shape sgemm_3xtf32 uses
 * (M 128, N = n, K 8; n is 128 or 256) on operands resident in shared
 * memory, accumulating in TMEM; nothing else runs. Calibrated to last about
 * target_ms (>= 1) and timed with CUDA events on `stream` after one untimed
 * warm-up launch of the same length. Outputs (each may be NULL): *tflops =
 * 2 M N K per MMA x MMAs / time, *ms = time of the timed launch, *flops =
 * floating-point operations of the timed launch. Blocking: synchronises
 * `stream`. SGEMM_ERR_INVALID_VALUE for another n or target.
 */
SGEMM_API int sgemm_tf32_mma_peak(int n, double target_ms, double* tflops, double* ms,
                                  double* flops, cudaStream_t stream);

/*
 * sgemm_null_launch — enqueue one kernel that does nothing (one CTA of 32
 * threads) on `stream`. Timed like a call, it gives the launch-latency floor
 * below which no call of this library can go on the device; the small
 * problems (256^3) are measured against it. Returns SGEMM_ERR_LAUNCH if the
 * launch fails (no device, for instance).
 */
SGEMM_API int sgemm_null_launch(cudaStream_t stream);

/*
 * sgemm_selftest_wait_timeout — launch one CTA whose bounded mbarrier wait
 * can never be satisfied (nothing arrives) with a limit of timeout_ns, to
 * show that the time-out path returns instead of hanging. The kernel sets
 * status bit 1 and exits; read it with sgemm_check_status. Returns launch
 * errors like sgemm.
 */
SGEMM_API int sgemm_selftest_wait_timeout(uint64_t timeout_ns, cudaStream_t stream);

/*
 * sgemm_selftest_occupy — launch `ctas` CTAs on `stream`, each holding one
 * SM (so much shared memory that no SGEMM CTA fits beside it) for `ns`
 * nanoseconds and doing nothing else: another kernel holding SMs, for
 * showing that an SGEMM started meanwhile on another stream still finishes
 * while its CTAs start a few at a time (see "Sharing the GPU" at sgemm).
 * Returns SGEMM_ERR_INVALID_VALUE unless 1 <= ctas <= the device's SM count
 * and 0 < ns <= 2e9, else launch errors like sgemm.
 */
SGEMM_API int sgemm_selftest_occupy(int ctas, uint64_t ns, cudaStream_t stream);

/*
 * sgemm_3xtf32 — the same operation, arguments and errors as sgemm, computed
 * on the tcgen05 tensor cores with the three-term TF32 split: each FP32
 * input x = x_hi + x_lo (x_hi = tf32(x), x_lo = tf32(x - x_hi)) and
 * a*b ~ a_hi*b_hi + a_hi*b_lo + a_lo*b_hi with FP32 accumulation in TMEM.
 * The dropped terms are at most about 3 * 2^-22 |a b| per product, which
 * keeps every element within the FP32 bound 4 K 2^-24 (|alpha| sum|a b| +
 * |beta c|) for K >= 3; calls with K < 16 or alpha == 0 run the FFMA path
 * (sgemm). It is reported separately from the strict FFMA path: the tensor
 * cores do not round every accumulation step like FFMA, so results differ
 * from sgemm's in the last bits. The pages measure TF32 only as an inexact
 * mode and describe no split; this entry point is this library's own.
 * Infinite inputs are outside its contract: the lo part of an infinity is
 * NaN, so an output the definition makes +-inf comes out NaN (NaN inputs
 * still give NaN).
 *
 * Large problems (enough 256 x 256 output tiles to give one to every CTA
 * pair the GPU runs at once) run on CTA pairs: the two CTAs of a cluster
 * share one 256 x 256 tile through tcgen05.mma.cta_group::2, each holding
 * half of the tile's rows of A and half of its columns of B. Otherwise,
 * where a tile row of C holds two 128 x 128 tiles (N > 128), the CTAs run in
 * thread-block clusters of two that share each A tile by TMA multicast.
 * Every variant gives the same bits.
 *
 * Each call splits A and the transpose of B into a workspace of
 * 8 * (M + N) * K bytes (K rounded up to 4) taken from the library's
 * stream-ordered pool, so it allocates like sgemm's stream-K tail; if that
 * allocation fails it runs sgemm instead.
 */
SGEMM_API int sgemm_3xtf32(int64_t M, int64_t N, int64_t K, float alpha, const float* A,
                           int64_t lda, const float* B, int64_t ldb, float beta, float* C,
                           int64_t ldc, cudaStream_t stream);

/* sgemm_3xtf32 with sgemm_ex's transposition flags and leading-dimension
 * rules. The split pre-passes read each operand in its stored layout and
 * write the K-major hi/lo copies the MMAs take, so transposition costs no
 * extra pass here. */
SGEMM_API int sgemm_3xtf32_ex(int opa, int opb, int64_t M, int64_t N, int64_t K, float alpha,
                              const float* A, int64_t lda, const float* B, int64_t ldb,
                              float beta, float* C, int64_t ldc, cudaStream_t stream);

/*
 * sgemm_noalloc — the same operation, arguments, results and errors as
 * sgemm, for callers that must not allocate device memory. The pages this
 * library follows have no counterpart: it exists for code that cannot call
 * cudaMalloc or a pool allocator: programs whose device memory is owned by
 * another allocator that must account for every byte, and latency-critical
 * paths that may not take an allocator's locks. sgemm allocates a status word on its first call on a
 * device and a stream-K workspace for some problems; sgemm_noalloc instead
 * uses one fixed 32 MiB scratch array compiled into the library (held by
 * every GPU that loads the library until the process exits).
 *
 * The first call on a device looks up the scratch array's device address
 * and performs the library's per-device kernel set-up: make that first call
 * before any stream capture begins. Every call on a device shares the
 * scratch, which keeps the last call's contents; nothing in it needs
 * clearing between calls. Calls that overlap on the GPU (on streams with no
 * ordering between them) race on the scratch and can produce wrong results,
 * so serialise them. Returns SGEMM_ERR_INVALID_VALUE, with nothing enqueued,
 * if the problem's stream-K workspace would not fit in the scratch (never on
 * a 152-SM GB300, which needs at most 19.5 MB). Time-outs of bounded waits
 * inside its kernels are recorded in the scratch, not in the word that
 * sgemm_check_status reads: sgemm_noalloc_check_status reads and clears
 * them.
 */
SGEMM_API int sgemm_noalloc(int64_t M, int64_t N, int64_t K, float alpha, const float* A,
                            int64_t lda, const float* B, int64_t ldb, float beta, float* C,
                            int64_t ldc, cudaStream_t stream);

/*
 * sgemm_noalloc_check_status — sgemm_check_status for sgemm_noalloc: it
 * synchronises `stream`, then reads and clears the status word kept in the
 * fixed scratch of the current device, where the kernels sgemm_noalloc
 * launches record bounded-wait time-outs. It allocates nothing (the copy
 * goes to a host variable of the call). Returns SGEMM_OK,
 * SGEMM_ERR_DEVICE_TIMEOUT if a kernel launched by sgemm_noalloc since the
 * last check gave up on a wait (its output is then incomplete), or
 * SGEMM_ERR_CUDA if the synchronisation or the copy failed. If `bits` is not
 * NULL it receives the raw status bits, with the meaning sgemm_check_status
 * gives them. Like sgemm_noalloc, a first call on a device looks up the
 * scratch address; the check itself should not overlap a running
 * sgemm_noalloc on another stream.
 */
SGEMM_API int sgemm_noalloc_check_status(cudaStream_t stream, int* bits);

#ifdef __cplusplus
}
#endif

#endif /* SGEMM_GB300_H */
