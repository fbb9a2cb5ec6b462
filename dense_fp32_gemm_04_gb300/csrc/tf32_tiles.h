// Tile shapes of the flagged TF32 tensor-core kernels (tf32_kernels.cu); the
// planner (planner.cpp) sizes plans and workspaces from the same constants.
#pragma once

namespace sgemm_cfg {

// The flagged TF32 tensor-core mode: one CTA per SM computes 128 x 256 tiles
// (tcgen05.mma M = 128, N = 256) from 32-deep K slabs in a 4-stage ring.
constexpr int kTf32BM = 128, kTf32BN = 256, kTf32BK = 32, kTf32Stages = 4, kTf32Threads = 192;
// Staging areas of the four epilogue warps (32 rows x 36 floats each), after
// the ring and the barrier block.
constexpr int kTf32StagingBytes = 4 * 32 * 36 * 4;
constexpr int tf32_smem_bytes()
{
    return 1024 + kTf32Stages * (kTf32BM + kTf32BN) * kTf32BK * 4 + 256 + kTf32StagingBytes;
}

// TF32 on CTA pairs (tcgen05 .cta_group::2): a pair of CTAs on two SMs computes
// a 256 x 256 tile (M = 256, N = 256 per MMA); each CTA stages 128 rows of A
// and 128 columns of B (32 KiB per stage, 6 stages) and holds its 128 rows of
// the accumulator, so per SM the tensor core reads a third less shared memory
// per FMA than with one CTA per 128 x 256 tile.
constexpr int kTf32PairBM = 256, kTf32PairBN = 256, kTf32PairStages = 6;
// 1 KiB for aligning the ring to the swizzle atoms, the ring, the barrier block,
// the epilogue warps' staging areas.
constexpr int tf32_pair_smem_bytes()
{
    return 1024 + kTf32PairStages * (kTf32PairBM / 2 + kTf32PairBN / 2) * kTf32BK * 4 + 256 + kTf32StagingBytes;
}
static_assert(tf32_pair_smem_bytes() <= 227 * 1024 && tf32_smem_bytes() <= 227 * 1024, "shared memory per CTA");

}  // namespace sgemm_cfg
