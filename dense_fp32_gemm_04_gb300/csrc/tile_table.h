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
    // The same row with A transposed in shared memory (A layout 2): a
    // transposer warp turns each staged K-major A slab into one of xbufs
    // M-major buffers, so the ring is shorter.
    int xstages;
    int xbufs;
    int xthreads;        // threads + 32 (the transposer warp)
    int xsmem_bytes;
};

constexpr int kFfmaBK = 32;

constexpr int ffma_smem_bytes(int bm, int bn, int stages, int epilogue_warps, int xbufs = 0)
{
    // 1 KiB for aligning the ring to the 128-byte swizzle atom, the ring, the
    // M-major A buffers (A transposed in shared memory), the BM x BN staging
    // tile (with an epilogue warp), then 2 * stages mbarriers (+ 2 for the
    // staging tile, + 2 per M-major buffer) and an abort flag.
    return 1024 + stages * (bm * kFfmaBK * 4 + kFfmaBK * bn * 4) + xbufs * bm * kFfmaBK * 4 +
           (epilogue_warps > 0 ? bm * bn * 4 + 16 : 0) + 2 * stages * 8 + 2 * xbufs * 8 + 16;
}

constexpr TileConfig make_ffma(int bm, int bn, int stages, int ctas, float cost, int epilogue_warps, int xstages,
                               int xbufs)
{
    return TileConfig{bm, bn, kFfmaBK, stages, (bm / 32) * (bn / 64), epilogue_warps,
                      ((bm / 32) * (bn / 64) + 1 + epilogue_warps) * 32, ctas,
                      ffma_smem_bytes(bm, bn, stages, epilogue_warps), cost, xstages, xbufs,
                      ((bm / 32) * (bn / 64) + 2 + epilogue_warps) * 32,
                      ffma_smem_bytes(bm, bn, xstages, epilogue_warps, xbufs)};
}

// Row order is part of the ABI of sgemm_config_info / SGEMM_OPT_FORCE_CONFIG.
constexpr TileConfig kFfmaConfigs[] = {
    // rel_cost: time per FMA relative to row 0, measured on large squares
    // (4096^3 .. 16384^3, one split) by dense_fp32_gemm_04_gb300/tune.py.
    // xstages, xbufs: ring stages and M-major A buffers with A transposed in shared memory.
    make_ffma(128, 128, 5, 1, 1.000f, 2, 4, 2),  // 0: large squares (tiles written out by 2 epilogue warps)
    make_ffma(128, 64, 4, 2, 1.055f, 0, 3, 2),   // 1: N <= 64, or more tiles for mid sizes
    make_ffma(64, 128, 4, 2, 1.055f, 0, 3, 2),   // 2: M <= 64
    make_ffma(64, 64, 4, 3, 1.430f, 0, 3, 2),    // 3: tiny problems (1.5 consumer warps per scheduler)
};
constexpr int kNumFfmaConfigs = sizeof(kFfmaConfigs) / sizeof(kFfmaConfigs[0]);

// Shared memory of an SM (228 KiB), of which 1 KiB per resident CTA is reserved.
constexpr bool fits_sm(int smem, int ctas) { return smem <= 227 * 1024 && ctas * (smem + 1024) <= 228 * 1024; }
constexpr bool rows_fit()
{
    for (const TileConfig &c : kFfmaConfigs)
        if (!fits_sm(c.smem_bytes, c.ctas_per_sm) || !fits_sm(c.xsmem_bytes, c.ctas_per_sm)) return false;
    return true;
}
static_assert(rows_fit(), "every row (both ring forms) fits its resident CTAs in an SM's shared memory");

}  // namespace sgemm_cfg
