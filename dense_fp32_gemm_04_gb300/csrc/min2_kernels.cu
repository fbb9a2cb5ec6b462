// The two smallest elements of C and their (row, column), computed fully in
// parallel on the GPU after the GEMM ("SGEMM CUDA kernel (First Half)",
// Additionally Required: find two minimums of the product C and their 2D
// indices, with no sequential reduction on the host).
//
// Order: (value, row-major position i * N + j), so equal values rank by
// position and the answer is unique; NaN ranks as +infinity. Pass 1: every
// thread keeps a running top-2 (over C as one flat array of 16-byte groups when
// C is contiguous; otherwise block per row, threads striding over columns, with
// 16-byte loads when C allows), merged across the warp with shuffles and across
// warps in shared memory; each block writes one candidate pair. Pass 2: one block merges all candidate pairs. The result
// does not depend on scheduling.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>

#include "device_ptx.cuh"
#include "sgemm_internal.h"

namespace sgemm_impl {
namespace {

using namespace sgemm_dev;

constexpr int kThreads = 256;

struct Top2 {
    float v0, v1;
    long long p0, p1;  // row-major positions (LLONG_MAX: none)
};

__device__ __forceinline__ bool before(float a, long long pa, float b, long long pb)
{
    return a < b || (a == b && pa < pb);
}

__device__ __forceinline__ void push(Top2 &t, float v, long long p)
{
    if (v > t.v1) return;  // the common case: above the current second (v0 <= v1, never NaN)
    if (v != v) v = __int_as_float(0x7f800000);  // NaN ranks as +inf
    if (before(v, p, t.v0, t.p0)) {
        t.v1 = t.v0;
        t.p1 = t.p0;
        t.v0 = v;
        t.p0 = p;
    } else if (before(v, p, t.v1, t.p1)) {
        t.v1 = v;
        t.p1 = p;
    }
}

__device__ __forceinline__ void merge(Top2 &t, const Top2 &o)
{
    push(t, o.v0, o.p0);
    push(t, o.v1, o.p1);
}

__device__ __forceinline__ Top2 empty_top2()
{
    Top2 t;
    t.v0 = t.v1 = __int_as_float(0x7f800000);
    t.p0 = t.p1 = LLONG_MAX;
    return t;
}

// Warp, then block reduction of each thread's Top2; thread 0 gets the result.
__device__ Top2 block_reduce(Top2 t)
{
    __shared__ Top2 part[kThreads / 32];
    for (int off = 16; off > 0; off >>= 1) {
        Top2 o;
        o.v0 = __shfl_down_sync(0xffffffffu, t.v0, off);
        o.v1 = __shfl_down_sync(0xffffffffu, t.v1, off);
        o.p0 = __shfl_down_sync(0xffffffffu, t.p0, off);
        o.p1 = __shfl_down_sync(0xffffffffu, t.p1, off);
        merge(t, o);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) part[warp] = t;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kThreads / 32; ++w) merge(t, part[w]);
    }
    return t;
}

// Pushes the four values of a 16-byte group at row-major positions pos..pos+3,
// after a fast reject of the whole group: its smallest value (fminf ignores NaN,
// which ranks as +inf) lies above `thr`, a value that two elements already seen
// do not exceed (this thread's second, or a smaller lane's). Four NaNs give NaN,
// which is not above anything, so they are pushed one by one.
__device__ __forceinline__ void push4(Top2 &t, float4 v, long long pos, float thr)
{
    const float m = fminf(fminf(v.x, v.y), fminf(v.z, v.w));
    if (m > thr) return;
    push(t, v.x, pos);
    push(t, v.y, pos + 1);
    push(t, v.z, pos + 2);
    push(t, v.w, pos + 3);
}

// Pass 1 for a contiguous C (ldc == N, 16-byte aligned): C is one array of M N / 4
// 16-byte groups, whose index times 4 is the row-major position; every warp takes
// an even share (8 loads in flight per lane), so no block waits on a long row.
constexpr int kFlatLoads = 8;

__global__ void __launch_bounds__(kThreads) min2_pass1_flat(const float *__restrict__ C, long long groups,
                                                            Top2 *__restrict__ cand)
{
    pdl_wait();     // C is complete (the call's GEMM kernels)
    pdl_trigger();  // the merge may become resident; it waits for this grid to finish
    Top2 t = empty_top2();
    const float4 *c4 = reinterpret_cast<const float4 *>(C);
    const int lane = threadIdx.x & 31;
    // A warp reads a contiguous chunk of 32 x kFlatLoads groups per step (lane l:
    // groups l, l + 32, ...), consecutive warps consecutive chunks: C streams in
    // address order. The loop is warp-uniform (the threshold below is a shuffle).
    constexpr long long kChunk = 32LL * kFlatLoads;
    const long long warps = static_cast<long long>(gridDim.x) * (kThreads / 32);
    for (long long cw = static_cast<long long>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5); cw * kChunk < groups;
         cw += warps) {
        const long long g0 = cw * kChunk + lane;
        float4 v[kFlatLoads];
#pragma unroll
        for (int j = 0; j < kFlatLoads; ++j)
            if (g0 + 32 * j < groups) v[j] = __ldcs(c4 + g0 + 32 * j);
        // The smallest second of the warp's lanes: two elements already seen by that
        // lane do not exceed it, so nothing above it can be among the two minima.
        float thr = t.v1;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) thr = fminf(thr, __shfl_xor_sync(0xffffffffu, thr, off));
#pragma unroll
        for (int j = 0; j < kFlatLoads; ++j)
            if (g0 + 32 * j < groups) push4(t, v[j], 4 * (g0 + 32 * j), thr);
    }
    t = block_reduce(t);
    if (threadIdx.x == 0) cand[blockIdx.x] = t;
}

template <bool VEC>
__global__ void __launch_bounds__(kThreads) min2_pass1(const float *__restrict__ C, long long ldc, int M, int N,
                                                       Top2 *__restrict__ cand)
{
    pdl_wait();     // C is complete (the call's GEMM kernels)
    pdl_trigger();  // the merge may become resident; it waits for this grid to finish
    Top2 t = empty_top2();
    for (int row = blockIdx.x; row < M; row += gridDim.x) {
        const float *crow = C + static_cast<long long>(row) * ldc;
        const long long base = static_cast<long long>(row) * N;
        if (VEC) {
            // 16-byte loads of 4 consecutive columns (C 16-byte aligned, ldc % 4 == 0),
            // four of them in flight per thread before any is compared
            const int n4 = N & ~3;
            constexpr int kStep = 4 * kThreads;
            for (int c0 = 4 * threadIdx.x; c0 < n4; c0 += 4 * kStep) {
                float4 v[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (c0 + j * kStep < n4) v[j] = __ldcs(reinterpret_cast<const float4 *>(crow + c0 + j * kStep));
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int col = c0 + j * kStep;
                    if (col < n4) push4(t, v[j], base + col, t.v1);
                }
            }
            for (int col = n4 + threadIdx.x; col < N; col += kThreads) push(t, crow[col], base + col);
        } else {
            for (int col = threadIdx.x; col < N; col += kThreads) push(t, crow[col], base + col);
        }
    }
    t = block_reduce(t);
    if (threadIdx.x == 0) cand[blockIdx.x] = t;
}

__global__ void __launch_bounds__(kThreads) min2_pass2(const Top2 *__restrict__ cand, int n, int N,
                                                       float *__restrict__ vals, int *__restrict__ ij)
{
    pdl_wait();  // every candidate pair is written
    Top2 t = empty_top2();
    for (int i = threadIdx.x; i < n; i += kThreads) merge(t, cand[i]);
    t = block_reduce(t);
    if (threadIdx.x == 0) {
        vals[0] = t.v0;
        vals[1] = t.v1;
        ij[0] = t.p0 == LLONG_MAX ? -1 : static_cast<int>(t.p0 / N);
        ij[1] = t.p0 == LLONG_MAX ? -1 : static_cast<int>(t.p0 % N);
        ij[2] = t.p1 == LLONG_MAX ? -1 : static_cast<int>(t.p1 / N);
        ij[3] = t.p1 == LLONG_MAX ? -1 : static_cast<int>(t.p1 % N);
    }
}

}  // namespace

size_t min2_candidate_bytes(int blocks) { return sizeof(Top2) * static_cast<size_t>(blocks); }

cudaError_t launch_min2(const float *C, long long ldc, int M, int N, void *cand, int blocks, float *vals, int *ij,
                        cudaStream_t stream)
{
    const bool vec = (reinterpret_cast<uintptr_t>(C) & 15u) == 0 && ldc % 4 == 0;
    const bool flat = vec && ldc == N;
    const long long groups = static_cast<long long>(M) * N / 4;
    // the flat pass: 4 blocks per SM at most (blocks / 2), and enough groups for every thread
    const long long flat_blocks = std::min<long long>(blocks / 2, (groups + kThreads - 1) / kThreads);
    const int g = flat ? static_cast<int>(std::max<long long>(1, flat_blocks)) : (M < blocks ? (M > 0 ? M : 1) : blocks);
    // Both run as programmatic dependents of the kernel before them (the call's GEMM,
    // then pass 1); with nothing launched by the GEMM they simply follow the stream.
    Top2 *c = static_cast<Top2 *>(cand);
    cudaError_t e =
        flat  ? launch_kernel(true, min2_pass1_flat, dim3(g), dim3(kThreads), 0, stream, C, groups, c)
        : vec ? launch_kernel(true, min2_pass1<true>, dim3(g), dim3(kThreads), 0, stream, C, ldc, M, N, c)
              : launch_kernel(true, min2_pass1<false>, dim3(g), dim3(kThreads), 0, stream, C, ldc, M, N, c);
    if (e != cudaSuccess) return e;
    return launch_kernel(true, min2_pass2, dim3(1), dim3(kThreads), 0, stream, static_cast<const Top2 *>(c), g, N,
                         vals, ij);
}

}  // namespace sgemm_impl
