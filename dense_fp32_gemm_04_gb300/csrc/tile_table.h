// The tile-config table: every FFMA CTA shape the library instantiates. The
// planner (planner.cpp) picks a row and a split-K factor per problem; the
// kernels (ffma_kernels.cu) instantiate exactly these rows, in this order,
// and static_assert that their shared-memory sizes match.
//
// FFMA rows: a CTA computes a BM x BN tile of C from BM x 32 slabs of A and
// 32 x BN slabs of B staged by TMA through a STAGES-deep shared-memory ring.
// Each consumer warp owns a 32 x 64 warp tile, each lane an 8 x 8 microtile
// (the block / warp / thread tiling of "Optimizing Matrix Multiplication in
// CUDA", warp tiling section; the 8 x 8 microtile of "Shared memory and
// register blocking"). One extra warp issues the TMA copies; on a row with
// epilogue warps, those write each finished tile out of a shared-memory
// staging tile while the compute warps go on.
#pragma once

namespace sgemm_cfg {

struct TileConfig {
    int bm, bn, bk, stages;
    int consumer_warps;  // (bm / 32) * (bn / 64)
    int epilogue_warps;  // > 0: warps of their own write each finished tile out of a shared-memory staging tile
    int threads;         // (consumer_warps + 1 + epilogue_warps) * 32
    int ctas_per_sm;     // residency the launch bounds and shared memory allow
    int smem_bytes;      // dynamic shared memory per CTA
    float rel_cost;      // measured time per FMA relative to row 0 (planner weight)
};

constexpr int kFfmaBK = 32;

constexpr int ffma_smem_bytes(int bm, int bn, int stages, int epilogue_warps)
{
    // 1 KiB for aligning the ring to the 128-byte swizzle atom, the ring, the
    // BM x BN staging tile (with an epilogue warp), then 2 * stages mbarriers (+ 2
    // for the staging tile) and an abort flag.
    return 1024 + stages * (bm * kFfmaBK * 4 + kFfmaBK * bn * 4) + (epilogue_warps > 0 ? bm * bn * 4 + 16 : 0) +
           2 * stages * 8 + 16;
}

constexpr TileConfig make_ffma(int bm, int bn, int stages, int ctas, float cost, int epilogue_warps = 0)
{
    return TileConfig{bm, bn, kFfmaBK, stages, (bm / 32) * (bn / 64), epilogue_warps,
                      ((bm / 32) * (bn / 64) + 1 + epilogue_warps) * 32, ctas,
                      ffma_smem_bytes(bm, bn, stages, epilogue_warps), cost};
}

// Row order is part of the ABI of sgemm_config_info / SGEMM_OPT_FORCE_CONFIG.
constexpr TileConfig kFfmaConfigs[] = {
    // rel_cost: time per FMA relative to row 0, measured on large squares
    // (4096^3 .. 16384^3, one split) by dense_fp32_gemm_04_gb300/tune.py.
    make_ffma(128, 128, 5, 1, 1.000f, 2),  // 0: large squares (tiles written out by 2 epilogue warps)
    make_ffma(128, 64, 4, 2, 1.055f),   // 1: N <= 64, or more tiles for mid sizes
    make_ffma(64, 128, 4, 2, 1.055f),   // 2: M <= 64
    make_ffma(64, 64, 4, 3, 1.430f),    // 3: tiny problems (1.5 consumer warps per scheduler)
};
constexpr int kNumFfmaConfigs = sizeof(kFfmaConfigs) / sizeof(kFfmaConfigs[0]);
static_assert(kFfmaConfigs[0].smem_bytes <= 227 * 1024, "shared memory per CTA");

}  // namespace sgemm_cfg
