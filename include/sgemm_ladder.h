/*
 * sgemm_ladder.h — the pages' SGEMM kernel ladder on GB300, for comparison.
 *
 * These are context kernels, not the library's product path (include/sgemm.h):
 * each rung is one technique of the pages' ladder, rewritten for sm_103a so its
 * worth can be measured on this GPU:
 *   1 naive (lane index down the rows of C) and 2 coalesced (along the rows):
 *     "Global Memory Coalescing";
 *   3 shared-memory tiles, one output per thread: "Shared memory and register
 *     blocking" and "SGEMM CUDA kernel (First Half)", Part 3;
 *   4 1D register tiling (64 x 64 block, 8 outputs per thread): "1D Register
 *     Tiling: One Thread, TM Outputs";
 *   5 2D register tiling (128 x 128 block, 8 x 8 per thread): "SGEMM CUDA
 *     kernel (First Half)", Part 4;
 *   6 transposed A in shared memory + 128-bit loads: same page, Parts 5 and 6;
 *   7 warp tiling (64 x 64 warp tiles): "Optimizing Matrix Multiplication in
 *     CUDA", warp tiling;
 *   8 cache blocking: 8 x 8 register microtiles per thread with A and B read
 *     through L1 / L2 and no shared memory, the kernel "Shared memory and
 *     register blocking" measures its 32 x 32 shared-memory tiles against.
 */
#ifndef SGEMM_GB300_LADDER_H
#define SGEMM_GB300_LADDER_H

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;

/*
 * C = alpha * A * B + beta * C with rung `rung` (1..8), PACKED row-major DEVICE
 * matrices (A: M x K, B: K x N, C: M x N, leading dimensions K, N, N), on the
 * current device, asynchronously on `stream`. beta == 0: C is not read.
 * Returns SGEMM_OK, SGEMM_ERR_INVALID_VALUE (unknown rung, negative dimension,
 * NULL operand with work to do, an operand not 4-byte aligned), SGEMM_ERR_NOT_SUPPORTED (rungs 6, 7 and 8 need
 * K % 4 == 0, N % 4 == 0 and 16-byte-aligned A and B, as the page's vectorised
 * kernel does; M > 2^21) or SGEMM_ERR_LAUNCH.
 */
int sgemm_ladder_run(int rung, int M, int N, int K, float alpha, const float *A, const float *B, float beta,
                     float *C, struct CUstream_st *stream);

#ifdef __cplusplus
}
#endif

#endif /* SGEMM_GB300_LADDER_H */
