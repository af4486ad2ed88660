// ptx.cuh — thin inline-PTX wrappers for sm_103a: mbarrier, TMA tile loads,
// element-wise cp.async, GPU-scope flags, timers.
//
// Every wait built on these is bounded by the caller (see sgemm_kernel.cuh):
// nothing here spins.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace sg {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- programmatic dependent launch ----------------------------------------
// A kernel launched with programmatic stream serialisation may begin while
// the kernel before it on the stream is still running. griddep_wait blocks
// the calling thread until that kernel has completed and its memory writes
// are visible (for a kernel launched the ordinary way it returns at once);
// every thread calls it before its first global-memory access.
// griddep_launch_dependents lets the kernel after this one be scheduled once
// every CTA of this grid has issued it (or exited); that kernel still waits
// for this one to complete before it touches memory.

__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- thread-block clusters ---------------------------------------------------
// A cluster's CTAs run at the same time on one GPC and can reach each
// other's shared memory (distributed shared memory).

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

// Every thread of every CTA in the cluster arrives (release) and waits
// (acquire). Not the .aligned form: the threads of a warp may reach it at
// different times.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\n\t"
                 "barrier.cluster.wait.acquire;" ::: "memory");
}

// The shared::cluster address of the same shared-memory offset in CTA
// `rank` of this cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float4 v) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};"
                 :: "r"(addr), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w) : "memory");
}

// Arrive on an mbarrier in another CTA of the cluster, releasing this
// thread's earlier writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];"
                 :: "r"(cluster_addr) : "memory");
}

// ---- mbarrier --------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy (TMA) and to the
// other threads of the CTA (followed by a __syncthreads at the call site).
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{\n\t.reg .b64 st;\n\t"
                 "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}"
                 :: "r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\t"
                 "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
                 :: "r"(bar), "r"(bytes) : "memory");
}

// True once the phase with the given parity has completed. Never blocks for
// long: the hardware may suspend the thread for a bounded, system-defined
// time before returning false.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// try_wait with acquire semantics at cluster scope: once true, the writes
// that other CTAs of the cluster made before their release-arrive on this
// barrier (to this CTA's shared memory) are visible.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// Non-blocking probe: true if the phase with the given parity has completed
// (acquire semantics when true, like try_wait).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// ---- TMA (cp.async.bulk.tensor) --------------------------------------------

__device__ __forceinline__ void tma_prefetch_desc(const void* desc) {
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(desc)) : "memory");
}

// 2-D tile load: box at (x = inner coordinate, y = outer coordinate) into
// shared memory at dst; completion is signalled as transaction bytes on bar.
// The caller guarantees x * 4 bytes is a multiple of 16 (x is a multiple of
// the tile width, itself a multiple of 4 floats).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* desc, uint32_t bar,
                                            int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(desc)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

// ---- element-wise cp.async (4 bytes, zero-fill) ----------------------------

// Copies 4 bytes from src to shared dst; when !valid no byte is read and the
// destination is zero-filled (src-size 0). src must still be a valid address.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const float* src, bool valid) {
    const uint32_t n = valid ? 4u : 0u;
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;"
                 :: "r"(dst), "l"(src), "r"(n) : "memory");
}

// Arrive on bar once every cp.async this thread issued so far has landed.
// .noinc: the arrival is counted in the barrier's expected count.
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(bar) : "memory");
}

// ---- L2 prefetch -------------------------------------------------------------

// Bring the 128-byte line holding `p` into L2 (no register result, no fault
// semantics the callers rely on: every address passed is inside its matrix).
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" :: "l"(p));
}

// ---- flags between the CTAs of one grid (global memory, GPU scope) ----------

// Load with acquire semantics at GPU scope: writes released before the flag
// by another CTA are visible to this thread after it reads the flag.
__device__ __forceinline__ unsigned long long ld_acquire_gpu(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Store with release semantics at GPU scope.
__device__ __forceinline__ void st_release_gpu(unsigned long long* p, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}

// Orders this thread's accesses to global memory through the generic proxy
// (ordinary loads and stores) with its accesses through the async proxy
// (TMA): data another thread stored and released, and this thread acquired,
// is then what a TMA load that follows reads.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Named barrier `id` (1..15) among `count` threads (a multiple of 32) of
// the CTA; barrier 0 is __syncthreads.
__device__ __forceinline__ void named_bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(count) : "memory");
}

// ---- timers ----------------------------------------------------------------

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

}  // namespace sg
