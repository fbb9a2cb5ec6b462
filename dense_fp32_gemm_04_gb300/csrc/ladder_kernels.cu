// The pages' SGEMM kernel ladder, rewritten for sm_103a as context kernels:
// each rung is the technique one page describes, written from that
// description (the printed listings have indexing defects and are not used).
// They exist to measure what each step is worth on GB300; the library's
// product path is ffma_kernels.cu. All rungs compute C = alpha*A*B + beta*C on
// packed row-major matrices (lda = K, ldb = N, ldc = N), FP32 FMAs in ascending
// k, with C not read when beta == 0, and zero-filled tile edges.
//
//   1 naive        one thread per C element; the lane index runs down the rows
//                  ("Global Memory Coalescing", the naive mapping)
//   2 coalesced    the lane index runs along a row of C ("Global Memory
//                  Coalescing", kernel 2)
//   3 smem tile    32 x 32 tiles of A and B in shared memory, one output per
//                  thread ("Shared memory and register blocking", first kernel;
//                  "SGEMM CUDA kernel (First Half)", Part 3)
//   4 1D regtile   64 x 64 block, BK = 8, each thread a column of TM = 8
//                  outputs ("1D Register Tiling: One Thread, TM Outputs")
//   5 2D regtile   128 x 128 block, BK = 8, 8 x 8 outer-product microtile per
//                  thread ("SGEMM CUDA kernel (First Half)", Part 4)
//   6 AsT + float4 A staged transposed in shared memory, 128-bit loads of B
//                  and of the register fragments (same page, Parts 5 and 6);
//                  needs K % 4 == 0 and N % 4 == 0, like the page's rule
//   7 warp tile    128 x 128 block, BK = 16, four warps of 64 x 64, each lane
//                  8 x 4 outputs in four column sub-tiles ("Optimizing Matrix
//                  Multiplication in CUDA", warp tiling); same shape rule
//   8 cache blocks 128 x 128 block, 8 x 8 register microtile per thread, A and
//                  B read straight from global memory through L1 / L2 and no
//                  shared memory: the block's reuse is left to the caches'
//                  eviction policy ("Shared memory and register blocking", the
//                  cache-blocking kernel it measures the shared-memory tiles
//                  against); same shape rule
#include <cuda_runtime.h>

#include "sgemm_internal.h"

namespace sgemm_impl {
namespace {

__device__ __forceinline__ void write_c(float *C, long long idx, float acc, float alpha, float beta)
{
    C[idx] = (beta != 0.0f) ? fmaf(alpha, acc, beta * C[idx]) : alpha * acc;
}

// ---- rung 1 and 2: one thread per output -----------------------------------
template <bool COALESCED>
__global__ void __launch_bounds__(1024) rung_simple(int M, int N, int K, float alpha, const float *__restrict__ A,
                                                    const float *__restrict__ B, float beta, float *__restrict__ C)
{
    const int row = blockIdx.y * 32 + (COALESCED ? threadIdx.y : threadIdx.x);
    const int col = blockIdx.x * 32 + (COALESCED ? threadIdx.x : threadIdx.y);
    if (row >= M || col >= N) return;
    float acc = 0.0f;
    for (int k = 0; k < K; ++k) acc = fmaf(A[static_cast<long long>(row) * K + k], B[static_cast<long long>(k) * N + col], acc);
    write_c(C, static_cast<long long>(row) * N + col, acc, alpha, beta);
}

// ---- rung 3: shared-memory tiles, one output per thread --------------------
__global__ void __launch_bounds__(1024) rung_smem(int M, int N, int K, float alpha, const float *__restrict__ A,
                                                  const float *__restrict__ B, float beta, float *__restrict__ C)
{
    __shared__ float As[32][32];
    __shared__ float Bs[32][32];
    const int ty = threadIdx.y, tx = threadIdx.x;
    const int row = blockIdx.y * 32 + ty, col = blockIdx.x * 32 + tx;
    float acc = 0.0f;
    for (int k0 = 0; k0 < K; k0 += 32) {
        As[ty][tx] = (row < M && k0 + tx < K) ? A[static_cast<long long>(row) * K + k0 + tx] : 0.0f;
        Bs[ty][tx] = (k0 + ty < K && col < N) ? B[static_cast<long long>(k0 + ty) * N + col] : 0.0f;
        __syncthreads();
#pragma unroll
        for (int k = 0; k < 32; ++k) acc = fmaf(As[ty][k], Bs[k][tx], acc);
        __syncthreads();
    }
    if (row < M && col < N) write_c(C, static_cast<long long>(row) * N + col, acc, alpha, beta);
}

// ---- rung 4: 1D register tiling --------------------------------------------
// 512 threads: thread t owns column t % 64 and rows 8 * (t / 64) .. + 7.
__global__ void __launch_bounds__(512) rung_1d(int M, int N, int K, float alpha, const float *__restrict__ A,
                                               const float *__restrict__ B, float beta, float *__restrict__ C)
{
    constexpr int BM = 64, BN = 64, BK = 8, TM = 8;
    __shared__ float As[BM][BK];
    __shared__ float Bs[BK][BN];
    const int t = threadIdx.x;
    const int tcol = t % BN, trow = t / BN;          // compute mapping
    const int a_r = t / BK, a_c = t % BK;            // A slab 64 x 8: one element per thread
    const int b_r = t / BN, b_c = t % BN;            // B slab 8 x 64: one element per thread
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    float acc[TM] = {};
    for (int k0 = 0; k0 < K; k0 += BK) {
        As[a_r][a_c] = (m0 + a_r < M && k0 + a_c < K) ? A[static_cast<long long>(m0 + a_r) * K + k0 + a_c] : 0.0f;
        Bs[b_r][b_c] = (k0 + b_r < K && n0 + b_c < N) ? B[static_cast<long long>(k0 + b_r) * N + n0 + b_c] : 0.0f;
        __syncthreads();
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            const float b = Bs[k][tcol];  // one B value reused for TM outputs
#pragma unroll
            for (int i = 0; i < TM; ++i) acc[i] = fmaf(As[trow * TM + i][k], b, acc[i]);
        }
        __syncthreads();
    }
    const int col = n0 + tcol;
    if (col >= N) return;
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int row = m0 + trow * TM + i;
        if (row < M) write_c(C, static_cast<long long>(row) * N + col, acc[i], alpha, beta);
    }
}

// ---- rung 5: 2D register tiling --------------------------------------------
// 256 threads; thread (ty, tx) = (t / 16, t % 16) owns rows 8ty.. and columns 8tx..
__global__ void __launch_bounds__(256) rung_2d(int M, int N, int K, float alpha, const float *__restrict__ A,
                                               const float *__restrict__ B, float beta, float *__restrict__ C)
{
    constexpr int BM = 128, BN = 128, BK = 8, TM = 8, TN = 8;
    __shared__ float As[BM][BK];
    __shared__ float Bs[BK][BN];
    const int t = threadIdx.x, ty = t / 16, tx = t % 16;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    float acc[TM][TN] = {};
    for (int k0 = 0; k0 < K; k0 += BK) {
        for (int e = t; e < BM * BK; e += 256) {
            const int r = e / BK, c = e % BK;
            As[r][c] = (m0 + r < M && k0 + c < K) ? A[static_cast<long long>(m0 + r) * K + k0 + c] : 0.0f;
        }
        for (int e = t; e < BK * BN; e += 256) {
            const int r = e / BN, c = e % BN;
            Bs[r][c] = (k0 + r < K && n0 + c < N) ? B[static_cast<long long>(k0 + r) * N + n0 + c] : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            float ra[TM], rb[TN];
#pragma unroll
            for (int i = 0; i < TM; ++i) ra[i] = As[ty * TM + i][k];
#pragma unroll
            for (int j = 0; j < TN; ++j) rb[j] = Bs[k][tx * TN + j];
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(ra[i], rb[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int row = m0 + ty * TM + i;
        if (row >= M) break;
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            const int col = n0 + tx * TN + j;
            if (col < N) write_c(C, static_cast<long long>(row) * N + col, acc[i][j], alpha, beta);
        }
    }
}

// ---- rung 6: transposed A in shared memory + 128-bit loads ------------------
__global__ void __launch_bounds__(256) rung_vec(int M, int N, int K, float alpha, const float *__restrict__ A,
                                                const float *__restrict__ B, float beta, float *__restrict__ C)
{
    constexpr int BM = 128, BN = 128, BK = 8, TM = 8, TN = 8;
    __shared__ __align__(16) float AsT[BK][BM];
    __shared__ __align__(16) float Bs[BK][BN];
    const int t = threadIdx.x, ty = t / 16, tx = t % 16;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    float acc[TM][TN] = {};
    for (int k0 = 0; k0 < K; k0 += BK) {
        {   // A slab 128 x 8: one float4 (4 k) per thread, stored transposed
            const int r = t / 2, c = (t % 2) * 4;
            const float4 v = (m0 + r < M && k0 + c < K)
                                 ? *reinterpret_cast<const float4 *>(A + static_cast<long long>(m0 + r) * K + k0 + c)
                                 : zero;
            AsT[c][r] = v.x;
            AsT[c + 1][r] = v.y;
            AsT[c + 2][r] = v.z;
            AsT[c + 3][r] = v.w;
        }
        {   // B slab 8 x 128: one float4 per thread
            const int r = t / 32, c = (t % 32) * 4;
            *reinterpret_cast<float4 *>(&Bs[r][c]) =
                (k0 + r < K && n0 + c < N)
                    ? *reinterpret_cast<const float4 *>(B + static_cast<long long>(k0 + r) * N + n0 + c)
                    : zero;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            const float4 a0 = *reinterpret_cast<const float4 *>(&AsT[k][ty * TM]);
            const float4 a1 = *reinterpret_cast<const float4 *>(&AsT[k][ty * TM + 4]);
            const float4 b0 = *reinterpret_cast<const float4 *>(&Bs[k][tx * TN]);
            const float4 b1 = *reinterpret_cast<const float4 *>(&Bs[k][tx * TN + 4]);
            const float ra[TM] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float rb[TN] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(ra[i], rb[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int row = m0 + ty * TM + i;
        if (row >= M) break;
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            const int col = n0 + tx * TN + j;
            if (col < N) write_c(C, static_cast<long long>(row) * N + col, acc[i][j], alpha, beta);
        }
    }
}

// ---- rung 7: warp tiling ----------------------------------------------------
// 128 threads = 4 warps in 2 x 2, each a 64 x 64 warp tile walked as four
// 64 x 16 column sub-tiles; lane (lr, lc) = (lane / 4, lane % 4) owns rows
// 8lr .. 8lr+7 of the warp tile and columns 4lc .. 4lc+3 of every sub-tile.
__global__ void __launch_bounds__(128) rung_warp(int M, int N, int K, float alpha, const float *__restrict__ A,
                                                 const float *__restrict__ B, float beta, float *__restrict__ C)
{
    constexpr int BM = 128, BN = 128, BK = 16, TM = 8, TN = 4, NSUB = 4;
    __shared__ __align__(16) float AsT[BK][BM];
    __shared__ __align__(16) float Bs[BK][BN];
    const int t = threadIdx.x, warp = t / 32, lane = t % 32;
    const int wm = warp / 2, wn = warp % 2, lr = lane / 4, lc = lane % 4;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    float acc[NSUB][TM][TN] = {};
    for (int k0 = 0; k0 < K; k0 += BK) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int e = t + q * 128;
            const int ra = e / 4, ca = (e % 4) * 4;
            const float4 v = (m0 + ra < M && k0 + ca < K)
                                 ? *reinterpret_cast<const float4 *>(A + static_cast<long long>(m0 + ra) * K + k0 + ca)
                                 : zero;
            AsT[ca][ra] = v.x;
            AsT[ca + 1][ra] = v.y;
            AsT[ca + 2][ra] = v.z;
            AsT[ca + 3][ra] = v.w;
            const int rb = e / 32, cb = (e % 32) * 4;
            *reinterpret_cast<float4 *>(&Bs[rb][cb]) =
                (k0 + rb < K && n0 + cb < N)
                    ? *reinterpret_cast<const float4 *>(B + static_cast<long long>(k0 + rb) * N + n0 + cb)
                    : zero;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            const float4 a0 = *reinterpret_cast<const float4 *>(&AsT[k][wm * 64 + lr * TM]);
            const float4 a1 = *reinterpret_cast<const float4 *>(&AsT[k][wm * 64 + lr * TM + 4]);
            const float ra[TM] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
            for (int sub = 0; sub < NSUB; ++sub) {
                const float4 b = *reinterpret_cast<const float4 *>(&Bs[k][wn * 64 + sub * 16 + lc * TN]);
                const float rb[TN] = {b.x, b.y, b.z, b.w};
#pragma unroll
                for (int i = 0; i < TM; ++i)
#pragma unroll
                    for (int j = 0; j < TN; ++j) acc[sub][i][j] = fmaf(ra[i], rb[j], acc[sub][i][j]);
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int row = m0 + wm * 64 + lr * TM + i;
        if (row >= M) break;
#pragma unroll
        for (int sub = 0; sub < NSUB; ++sub)
#pragma unroll
            for (int j = 0; j < TN; ++j) {
                const int col = n0 + wn * 64 + sub * 16 + lc * TN + j;
                if (col < N) write_c(C, static_cast<long long>(row) * N + col, acc[sub][i][j], alpha, beta);
            }
    }
}

// ---- rung 8: cache blocking --------------------------------------------------
// 256 threads; thread t owns rows 8 (t / 16) .. + 7 of the block's 128 and columns
// 4 (t % 16) .. + 3 and 64 + 4 (t % 16) .. + 3. Per 4-deep k step it loads 16 bytes
// of each of its 8 A rows and, for each k, 16 bytes of each of its 2 B column groups,
// all from global memory on the read-only path: the 16 lanes that share a row group
// read the same A bytes and the 16 that share a column group the same B bytes, so a
// block's operands are re-read from L1 / L2 rather than staged. Needs K % 4 == 0,
// N % 4 == 0 and 16-byte-aligned A and B.
__global__ void __launch_bounds__(256) rung_cache(int M, int N, int K, float alpha, const float *__restrict__ A,
                                                  const float *__restrict__ B, float beta, float *__restrict__ C)
{
    const int t = threadIdx.x;
    const int row0 = blockIdx.y * 128 + 8 * (t / 16);
    const int col0 = blockIdx.x * 128 + 4 * (t % 16);
    const float4 zero = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;
    for (int k0 = 0; k0 < K; k0 += 4) {
        float4 a[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            a[i] = row0 + i < M ? __ldg(reinterpret_cast<const float4 *>(A + static_cast<long long>(row0 + i) * K + k0))
                                : zero;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const float *brow = B + static_cast<long long>(k0 + kk) * N;
            const float4 b0 = col0 < N ? __ldg(reinterpret_cast<const float4 *>(brow + col0)) : zero;
            const float4 b1 = col0 + 64 < N ? __ldg(reinterpret_cast<const float4 *>(brow + col0 + 64)) : zero;
            const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float av = kk == 0 ? a[i].x : kk == 1 ? a[i].y : kk == 2 ? a[i].z : a[i].w;
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av, bv[j], acc[i][j]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int row = row0 + i;
        if (row >= M) break;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int col = col0 + (j < 4 ? j : 60 + j);
            if (col < N) write_c(C, static_cast<long long>(row) * N + col, acc[i][j], alpha, beta);
        }
    }
}

dim3 grid_for(int M, int N, int bm, int bn) { return dim3((N + bn - 1) / bn, (M + bm - 1) / bm); }

}  // namespace

// Launch rung 1..8 (see the file header). Returns cudaErrorInvalidValue for an
// unknown rung or a shape/alignment the rung does not handle.
cudaError_t launch_ladder(int rung, int M, int N, int K, float alpha, const float *A, const float *B, float beta,
                          float *C, cudaStream_t stream)
{
    const bool vec_ok = K % 4 == 0 && N % 4 == 0 && (reinterpret_cast<uintptr_t>(A) & 15u) == 0 &&
                        (reinterpret_cast<uintptr_t>(B) & 15u) == 0;
    if (rung >= 6 && !vec_ok) return cudaErrorInvalidValue;
    if ((M + 31) / 32 > 65535) return cudaErrorInvalidValue;
    switch (rung) {
    case 1: rung_simple<false><<<grid_for(M, N, 32, 32), dim3(32, 32), 0, stream>>>(M, N, K, alpha, A, B, beta, C); break;
    case 2: rung_simple<true><<<grid_for(M, N, 32, 32), dim3(32, 32), 0, stream>>>(M, N, K, alpha, A, B, beta, C); break;
    case 3: rung_smem<<<grid_for(M, N, 32, 32), dim3(32, 32), 0, stream>>>(M, N, K, alpha, A, B, beta, C); break;
    case 4: rung_1d<<<grid_for(M, N, 64, 64), 512, 0, stream>>>(M, N, K, alpha, A, B, beta, C); break;
    case 5: rung_2d<<<grid_for(M, N, 128, 128), 256, 0, stream>>>(M, N, K, alpha, A, B, beta, C); break;
    case 6: rung_vec<<<grid_for(M, N, 128, 128), 256, 0, stream>>>(M, N, K, alpha, A, B, beta, C); break;
    case 7: rung_warp<<<grid_for(M, N, 128, 128), 128, 0, stream>>>(M, N, K, alpha, A, B, beta, C); break;
    case 8: rung_cache<<<grid_for(M, N, 128, 128), 256, 0, stream>>>(M, N, K, alpha, A, B, beta, C); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace sgemm_impl
