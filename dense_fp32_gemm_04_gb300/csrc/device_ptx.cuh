// Inline-PTX helpers for sm_103a shared by every kernel: mbarriers, TMA tile
// loads, the global timer used by the kernels' bounded waits, programmatic
// dependent launch, and the launch helper. Each wraps one PTX instruction (PTX
// ISA, "Parallel Synchronization and Communication Instructions: mbarrier",
// "Data Movement: cp.async.bulk.tensor", "griddepcontrol"), and the thread-block
// cluster primitives (rank, mapa, distributed shared memory loads,
// barrier.cluster). The tensor-core and CTA-pair (.cta_group::2) helpers are in
// tcgen05_ptx.cuh.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace sgemm_dev {

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before its
// later async-proxy (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One non-blocking-ish probe: true once the phase with parity `parity` has completed.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long global_timer_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait on an mbarrier phase. Returns false when `timeout_ns` elapsed
// or another thread of the CTA raised *abort_flag; never spins forever.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  const volatile int *abort_flag,
                                                  long long timeout_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 8; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (abort_flag != nullptr && *abort_flag) return false;
        if (static_cast<long long>(global_timer_ns() - t0) > timeout_ns) return false;
    }
}

// Programmatic dependent launch (kernels of one library call). pdl_wait: block
// until the grid this one was launched after has completed and its writes are
// visible (returns at once for a grid launched the ordinary way). pdl_trigger:
// let the next grid of the call, launched with the programmatic-serialization
// attribute, become resident early; it still waits in pdl_wait.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled TMA load of one box at element coordinates (x = inner, y = outer)
// into shared memory, completing `bytes` of transaction count on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int x, int y)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

// Thread-block clusters (PTX ISA "Cluster of Cooperative Thread Arrays",
// mapa, ld.shared::cluster, barrier.cluster): used by the TF32 CTA-pair kernel
// and by the FFMA kernel's split-K reduced within a cluster.
__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// CTAs in this CTA's cluster (1 when the kernel was not launched with clusters).
__device__ __forceinline__ uint32_t cluster_size()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_id_x()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_count_x()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// shared::cluster address of the variable at shared::cta address `addr` in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// 32-bit load from the shared memory of a CTA of the cluster.
__device__ __forceinline__ uint32_t ld_shared_cluster_u32(uint32_t cluster_addr)
{
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(cluster_addr) : "memory");
    return v;
}

// Every thread of every CTA of the cluster (warp-aligned): release this thread's
// earlier memory operations, acquire the others'.
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 128-bit load from the shared memory of a CTA of the cluster.
__device__ __forceinline__ float4 ld_shared_cluster_v4(uint32_t cluster_addr)
{
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(cluster_addr)
                 : "memory");
    return v;
}

// Named barrier `id` (1..15; 0 is __syncthreads) over `count` threads (a
// multiple of 32, whole warps): returns whether any participating thread
// passed pred = true.
__device__ __forceinline__ bool named_barrier_or(int id, int count, bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// Record the first error of a launch in the handle's device status word.
__device__ __forceinline__ void report_status(int *status, int code)
{
    if (status != nullptr) atomicCAS(status, 0, code);
}

// Debug builds (compiled with SGEMM_DEBUG_CHECKS=1): index checks in front of
// the kernels' memory accesses. A failed check records
// (SGEMM_ERR_INDEX << 16) | where in the status word and returns false, and the
// caller skips the access; it never traps. In the default build the check is
// `true` and compiles away.
#ifndef SGEMM_DEBUG_CHECKS
#define SGEMM_DEBUG_CHECKS 0
#endif
__device__ __forceinline__ bool index_ok(bool ok, int *status, int where)
{
#if SGEMM_DEBUG_CHECKS
    if (!ok) report_status(status, (8 << 16) | where);
    return ok;
#else
    (void)ok;
    (void)status;
    (void)where;
    return true;
#endif
}

// Launch `kernel`; with `dependent`, as a programmatic dependent of the kernel
// launched before it on `stream` (used only between kernels of one call, so a
// grid never waits on a previous call's kernels beyond their completion).
// cluster_x > 1 launches clusters of that many CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel_cluster(bool dependent, int cluster_x, void (*kernel)(KArgs...), dim3 grid, dim3 block,
                                  size_t smem, cudaStream_t stream, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (dependent) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = static_cast<unsigned>(cluster_x);
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(bool dependent, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, Args &&...args)
{
    return launch_kernel_cluster(dependent, 1, kernel, grid, block, smem, stream, static_cast<Args &&>(args)...);
}

}  // namespace sgemm_dev
