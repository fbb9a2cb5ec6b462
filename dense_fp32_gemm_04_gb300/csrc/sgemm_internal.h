// Interface between the host side of the library (planner, handle, C ABI in
// sgemm_api.cpp / planner.cpp) and its kernels (*.cu). Not installed.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "tf32_tiles.h"
#include "tile_table.h"

namespace sgemm_impl {

// A pointer the kernels may dereference as float (or int): NULL or 4-byte aligned.
// Checked on the host before any launch; a misaligned one is SGEMM_ERR_INVALID_VALUE.
inline bool elem_aligned(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Device status codes: (sgemm_status << 16) | where.
enum : int {
    kWhereConsumerFull = 1,  // a consumer's wait for a filled stage ran out
    kWhereProducerEmpty = 2, // the producer's wait for a released stage ran out
    kWhereDrain = 3,         // waiting for this CTA's own copies in flight ran out
    kWhereMmaEmpty = 4,      // TF32: the MMA issuer's wait for a filled stage ran out
    kWhereAccum = 5,         // TF32: the epilogue's wait for the accumulator ran out
    // 6: not used (TMEM allocation blocks until it succeeds; it reports nothing)
    kWherePairLayout = 7,    // TF32 pair: the two CTAs' shared-memory layouts differ (no work done)
    kWhereStaging = 8,       // FFMA: a wait on the epilogue's staging tile ran out
    kWhereTransposer = 9,    // FFMA, A transposed in shared memory: the transposer warp's wait for a
                             // filled stage or a free M-major buffer ran out
    kWhereClusterShape = 10, // FFMA split-K within clusters: the launch's cluster shape or the CTAs'
                             // shared-memory layouts do not match the plan (nothing computed)
    // Index checks of debug builds (SGEMM_DEBUG_CHECKS=1), reported as SGEMM_ERR_INDEX:
    kWhereIdxCopy = 20,       // TMA tile coordinate outside the tiles / k-blocks (FFMA)
    kWhereIdxTranspose = 21,  // transposer warp's shared-memory offsets
    kWhereIdxRing = 22,       // compute warp's ring stage / M-major buffer
    kWhereIdxStaging = 23,    // staging tile (or the partial tile staged for a cluster)
    kWhereIdxStoreC = 24,     // store to C outside M x N
    kWhereIdxSplit = 25,      // split-K slice outside the workspace
    kWhereIdxPartial = 26,    // stream-K partial tile outside the workspace
    kWhereIdxEpiRead = 27,    // epilogue warps' staging-tile reads
    kWhereIdxCluster = 28,    // distributed shared memory read (split-K within clusters)
    kWhereIdxSkReduce = 29,   // stream-K reduction's partial-tile reads
    kWhereIdxSplitReduce = 30,// split-K reduction's slice reads
    kWhereIdxTf32Copy = 33,   // TF32 TMA tile coordinate
    kWhereIdxTf32Store = 34   // TF32 store to C or to a partial tile
};

// Everything the FFMA mainloop needs besides the two tensor maps.
struct FfmaParams {
    int M, N, K;
    float alpha, beta;
    float *C;
    long long ldc;
    float *W;          // split-K partials: slice s at W + s * wstride, row stride ldw
    long long ldw;
    long long wstride;
    int splits;
    int tiles_m, tiles_n;
    int units;         // tiles_m * tiles_n * splits, or the whole tiles before a stream-K region
    int kblocks;       // ceil(K / 32)
    int vec_c;         // C may be accessed with 16-byte vectors
    int *status;       // device status word (first error wins)
    long long timeout_ns;
    int inject_skip;   // test only: CTA 0's producer never fills its n-th stage (-1 off)
    // Stream-K span (schedule.cuh; sk_tiles > 0 needs splits == 1): after the
    // `units` whole tiles, the last sk_tiles tiles of the raster are cut evenly
    // over sk_grid CTAs by k-block; partial tiles go, tile-packed, to
    // W + slot * BM * BN and sk_reduce_kernel adds them in k order.
    int sk_tiles;
    int sk_grid;
    // Test only (race detection): > 0 delays the producer by this many ns before
    // every fill, < 0 delays every consumer warp before it releases a slab.
    int skew_ns;
    // > 0: split-K reduced within thread-block clusters of cluster_split CTAs
    // (= splits; one (tile, slice) unit per CTA, cluster rank = slice): the
    // partial tiles meet in distributed shared memory, W is not used.
    int cluster_split;
    long long w_elems;  // floats the workspace holds at W (checked by debug builds; 0 without W)
};

// Everything the TF32 tcgen05 mainloops need besides the two tensor maps
// (A: M rows of K, read K-major; B: K rows of N, read MN-major). Tiles are
// 128 x 256 for the one-CTA kernel and 256 x 256 for the pair kernel.
struct Tf32Params {
    int M, N, K;
    float alpha, beta;
    float *C;
    long long ldc;
    int tiles_m, tiles_n;
    int units;         // whole tiles (before a stream-K span)
    int splits;        // always 1 (schedule.cuh interface)
    int kblocks;       // ceil(K / 32)
    int vec_c;
    int *status;
    long long timeout_ns;
    // Stream-K span, as in FfmaParams (partials at W + slot * BM * BN).
    float *W;
    int sk_tiles;
    int sk_grid;
    long long w_elems;  // floats the workspace holds at W (checked by debug builds)
};

// Plain-launch helpers implemented in the .cu files. All return the CUDA
// error of the launch (cudaSuccess when it was enqueued).
cudaError_t ffma_set_attributes();  // opt in to large dynamic shared memory (current device)
// a_layout (plan.transpose_a): 0 = tmA maps A (M rows of K) and the mainloop reads
// it K-major; 1 = tmA maps A^T (K rows of M, M contiguous); 2 = tmA maps A as for
// 0 and a transposer warp turns each staged slab M-major in shared memory.
// dependent: launched as a programmatic dependent of the call's previous kernel
// (transpose / repack), whose completion its copy issue waits for.
cudaError_t launch_ffma(int config, int a_layout, const CUtensorMap &tmA, const CUtensorMap &tmB,
                        const FfmaParams &p, int grid, cudaStream_t stream, bool dependent);
// w_elems: floats at W (checked by debug builds); status: the device status word.
cudaError_t launch_splitk_reduce(const float *W, long long ldw, long long wstride, int splits,
                                 int M, int N, float alpha, float beta, float *C, long long ldc,
                                 int vec_c, int num_sms, cudaStream_t stream, long long w_elems, int *status);
cudaError_t launch_sk_reduce(const FfmaParams &p, int bm, int bn, int num_sms, cudaStream_t stream);
cudaError_t launch_ladder(int rung, int M, int N, int K, float alpha, const float *A, const float *B, float beta,
                          float *C, cudaStream_t stream);
size_t min2_candidate_bytes(int blocks);
cudaError_t launch_min2(const float *C, long long ldc, int M, int N, void *cand, int blocks, float *vals, int *ij,
                        cudaStream_t stream);
cudaError_t launch_scale(int M, int N, float beta, float *C, long long ldc, int num_sms,
                         cudaStream_t stream);
cudaError_t tf32_set_attributes();
// tmA: box 32 k x 128 rows (128-byte swizzle); tmB: box 32 n x 32 k (128-byte
// swizzle). dependent: launched as a programmatic dependent of the call's
// previous kernel (an operand repack).
cudaError_t launch_tf32(const CUtensorMap &tmA, const CUtensorMap &tmB, const Tf32Params &p, int grid,
                        cudaStream_t stream, bool dependent);
// CTA-pair kernel: p in units of 256 x 256 pair tiles (W slots of 256 x 256);
// same tensor maps; grid = 2 x pairs.
cudaError_t launch_tf32_pair(const CUtensorMap &tmA, const CUtensorMap &tmB, const Tf32Params &p, int grid,
                             cudaStream_t stream, bool dependent);
// CTA pairs of the pair kernel that fit on the current device at once (0: none).
int tf32_pair_max_pairs();
// XT (cols x ldxt) = X^T for X (rows x cols, row stride ldx); ldxt % 4 == 0.
cudaError_t launch_transpose(const float *X, long long ldx, float *XT, long long ldxt, int rows, int cols,
                             cudaStream_t stream);
cudaError_t launch_repack(const float *src, long long lds, float *dst, long long ldd, int rows,
                          int cols, int num_sms, cudaStream_t stream);
// Both operand copies of a call in one launch: A^T (a_transpose) or a repack of A
// into a_dst, and a repack of B into b_dst.
cudaError_t launch_prep(const float *A, long long lda, float *a_dst, long long a_ldd, int a_rows, int a_cols,
                        bool a_transpose, const float *B, long long ldb, float *b_dst, long long b_ldd, int b_rows,
                        int b_cols, int num_sms, cudaStream_t stream);

}  // namespace sgemm_impl
