// Inline-PTX helpers for the TF32 tensor-core kernels on sm_103a: TMEM
// allocation, tcgen05.mma / commit / ld, shared-memory and instruction
// descriptors (PTX ISA, "TensorCore 5th Generation Family Instructions"), and
// the CTA-pair (cluster of two) operations the pair kernel uses (PTX ISA,
// "Cluster of Cooperative Thread Arrays", mapa, barrier.cluster, the
// .cta_group::2 forms). Each wraps one PTX instruction.
#pragma once

#include "device_ptx.cuh"

// tcgen05 (5th-generation tensor core) and TMEM helpers, cta_group::1.
namespace sgemm_dev {

// Allocate `ncols` TMEM columns (power of two >= 32); the base address is
// written to shared memory at dst. Whole warp, .sync.aligned.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc] with TF32 inputs and FP32 accumulation.
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 32 TMEM lanes x 16 consecutive 32-bit columns: lane i of the warp receives row
// (taddr lane + i), columns taddr.col .. +15. Complete with tmem_wait_ld.
__device__ __forceinline__ void tmem_ld_16(uint32_t taddr, uint32_t (&v)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
}

// Wait for this thread's tcgen05.ld results; the registers are tied in so no
// use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&v)[16])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]), "+r"(v[7]),
                   "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]), "+r"(v[14]),
                   "+r"(v[15])
                 :
                 : "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile written by TMA with
// the 128-byte swizzle: rows of 128 bytes (32 FP32 of K), 8-row groups 1024
// bytes apart. Fields: start address >> 4 (bits 0-13), leading byte offset >> 4
// (bits 16-29, not used by swizzled K-major layouts), stride byte offset >> 4
// (bits 32-45), descriptor version 1 (bits 46-48), swizzle mode 2 = 128-byte
// (bits 61-63).
__device__ __forceinline__ uint64_t smem_desc_k_sw128(uint32_t smem_byte_addr)
{
    uint64_t d = static_cast<uint64_t>((smem_byte_addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1) << 16;
    d |= static_cast<uint64_t>(1024 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Shared-memory matrix descriptor of an MN-major TF32 operand tile (MN
// contiguous), written by TMA in boxes of 32 MN x 32 K with the 128-byte
// swizzle of 32-byte chunks (the swizzle this operand form takes): a box is 32
// K-rows of 128 bytes; boxes along MN are `lbo` bytes apart (leading byte
// offset). The stride byte offset between K-row groups is 512 bytes: the rows
// are contiguous, so that holds for groups of 4 rows, and a K = 8 MMA stays
// inside one group of 8. Version 1, layout type 1 = 128-byte swizzle with
// 32-byte atoms.
__device__ __forceinline__ uint64_t smem_desc_mn_sw128_32b(uint32_t smem_byte_addr, uint32_t lbo)
{
    uint64_t d = static_cast<uint64_t>((smem_byte_addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>(512 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(1) << 61;
    return d;
}

// Instruction descriptor of tcgen05.mma .kind::tf32: D format F32 (bits 4-5 = 1),
// A and B format TF32 (bits 7-9 and 10-12 = 2), A K-major (bit 15 = 0), B K-major
// (bit 16 = 0) or MN-major (bit 16 = 1, b_mn), N >> 3 in bits 17-22, M >> 4 in
// bits 24-28.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N, bool b_mn = false)
{
    return (1u << 4) | (2u << 7) | (2u << 10) | ((b_mn ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// ---------------------------------------------------------------------------
// CTA pairs (thread-block clusters of two along x; PTX ISA "Cluster of
// Cooperative Thread Arrays", and the .cta_group::2 forms of the tcgen05 and
// TMA instructions). Rank 0 of the pair issues the MMAs for both CTAs.

// cluster_ctarank, cluster_size, mapa_shared, ld_shared_cluster_* and
// cluster_sync are in device_ptx.cuh (the FFMA kernel's cluster split-K uses
// them too).

// Arrive (release, cluster scope) on an mbarrier given by its shared::cluster address.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// mbar_try_wait with cluster-scope acquire: for a barrier that CTAs of the
// cluster other than this one arrive on.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint32_t bar, uint32_t parity, const volatile int *abort_flag,
                                                          long long timeout_ns)
{
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 8; ++i)
            if (mbar_try_wait_cluster(bar, parity)) return true;
        if (abort_flag != nullptr && *abort_flag) return false;
        if (static_cast<long long>(global_timer_ns() - t0) > timeout_ns) return false;
    }
}

// 2-D tiled TMA load into this CTA's shared memory whose completion is counted
// on an mbarrier of either CTA of the pair (`bar_cluster`: shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, uint32_t bar_cluster, int x,
                                                 int y)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
        : "memory");
}

// TMEM allocation shared by the pair: one warp of each CTA executes these
// together; the same column range is allocated in both CTAs' TMEM.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Pair MMA (issued by rank 0): rows 0..M/2-1 of A and D in rank 0, the rest in
// rank 1; columns 0..N/2-1 of B in rank 0, the rest in rank 1; the descriptors'
// shared-memory addresses apply in both CTAs.
__device__ __forceinline__ void mma_tf32_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on the mbarrier at shared::cta offset `bar` in both CTAs of the
// pair when this thread's earlier tcgen05 operations have completed.
__device__ __forceinline__ void mma_commit_pair_both(uint32_t bar)
{
    const uint16_t mask = 3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}

// As mma_commit_pair_both, for this CTA's barrier only.
__device__ __forceinline__ void mma_commit_pair_local(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

}  // namespace sgemm_dev
