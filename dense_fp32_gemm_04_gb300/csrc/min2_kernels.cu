// The two smallest elements of C and their (row, column), computed fully in
// parallel on the GPU after the GEMM ("SGEMM CUDA kernel (First Half)",
// Additionally Required: find two minimums of the product C and their 2D
// indices, with no sequential reduction on the host).
//
// Order: (value, row-major position i * N + j), so equal values rank by
// position and the answer is unique; NaN ranks as +infinity. Pass 1: every
// block keeps a running top-2 over rows of C (grid-stride over rows, threads
// stride over columns, coalesced, with 16-byte loads when C allows), merges it
// across the warp with shuffles and across warps in shared memory, and writes
// one candidate pair. Pass 2: one block merges all candidate pairs. The result
// does not depend on scheduling.
#include <cuda_runtime.h>

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
                    if (col < n4) {
                        push(t, v[j].x, base + col);
                        push(t, v[j].y, base + col + 1);
                        push(t, v[j].z, base + col + 2);
                        push(t, v[j].w, base + col + 3);
                    }
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
    const int g = M < blocks ? (M > 0 ? M : 1) : blocks;
    const bool vec = (reinterpret_cast<uintptr_t>(C) & 15u) == 0 && ldc % 4 == 0;
    // Both run as programmatic dependents of the kernel before them (the call's GEMM,
    // then pass 1); with nothing launched by the GEMM they simply follow the stream.
    Top2 *c = static_cast<Top2 *>(cand);
    cudaError_t e = vec ? launch_kernel(true, min2_pass1<true>, dim3(g), dim3(kThreads), 0, stream, C, ldc, M, N, c)
                        : launch_kernel(true, min2_pass1<false>, dim3(g), dim3(kThreads), 0, stream, C, ldc, M, N, c);
    if (e != cudaSuccess) return e;
    return launch_kernel(true, min2_pass2, dim3(1), dim3(kThreads), 0, stream, static_cast<const Top2 *>(c), g, N,
                         vals, ij);
}

}  // namespace sgemm_impl
