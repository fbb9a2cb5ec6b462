// FP32 FFMA SGEMM mainloop for sm_103a, plus the operand layout kernels
// (A / B transposition, repack of unaligned operands), the split-K and
// stream-K reductions and the beta-only scaling kernel.
//
// C = alpha * A * B + beta * C, row-major ("SGEMM CUDA kernel (First Half)",
// opening definition). The structure follows the tiling ladder of the pages —
// a CTA owns a BM x BN tile of C and walks K in BK-deep phases ("Shared memory
// and register blocking"; "SGEMM CUDA kernel (First Half)", Part 3), each
// thread accumulates an 8 x 8 register microtile as a sum of outer products
// (same page, Part 4 "Thread Tile"; "Optimizing Matrix Multiplication in
// CUDA", 2D thread tiling), warps own 32 x 64 sub-tiles (same page, warp
// tiling) — rebuilt for Blackwell:
//
//  * Staging: one producer thread issues TMA tile copies (A^T box BM x 32 or,
//    for A as given, A box 32 x BM with the 128-byte swizzle; B box BN x 32)
//    into a STAGES-deep ring guarded by full/empty mbarriers, in place of the
//    pages' load / __syncthreads / compute / __syncthreads phase loop.
//    Out-of-range rows and columns are zero-filled by the copy engine, which
//    is the pages' zero-fill predication ("SGEMM CUDA kernel (First Half)",
//    Part 5 load_ast) done in hardware.
//  * A layout and bank conflicts: the pages transpose A in shared memory so a
//    thread's TM values of A are contiguous (same page, Part 5). Here A
//    reaches the compute warps M-major in one of two ways. Either
//    transpose_kernel writes A^T (K x M, M contiguous) into the handle's
//    workspace once per call and the copy engine stages As[k][m] slabs of it
//    exactly like B, or (when that copy costs more than it saves: N small
//    against M * K) the copy engine stages A as given and a transposer warp
//    rewrites each slab M-major in shared memory (TMA cannot transpose 4-byte
//    elements). A thread owns rows 4r..4r+3 and 16+4r..16+4r+3 of its warp
//    tile and columns 4c..4c+3 and 32+4c..32+4c+3; per k it reads two 128-bit
//    words of A and two of B. The 8 lanes sharing r read the same A word (a
//    broadcast) and the 8 lanes sharing c read 8 consecutive B words, so every
//    128-bit shared load is conflict-free. A third form, kept for comparison
//    and reachable by option, reads A K-major as given: a thread then takes
//    rows r, r+4, ..., r+28 and reads 4 consecutive k of one row per 128-bit
//    load, and the 128-byte swizzle of the A slab puts the four row groups of
//    a warp in four distinct bank quads.
//  * Arithmetic: packed FFMA2 (two FP32 fused multiply-adds per instruction,
//    round-to-nearest-even, sm_100+) halves the issue slots the 64 FMAs of a
//    k-step need. With A^T the packed operand is a pair of A values along M
//    and the B value is broadcast, (a_m, a_m+1) * (b_n, b_n); the FMA pipe
//    sustains about 10 % more of this form than of (a_m, a_m) * (b_n, b_n+1),
//    which the K-major layout has to use because its two A values of a pair
//    would sit in different 128-bit loads. Either way each output is one chain
//    of IEEE FP32 FMAs in ascending k, so all three layouts give identical bits.
//  * Persistent grid: CTAs loop over (tile, split) work units in a grouped
//    order; the producer keeps prefetching across unit boundaries.
//  * Epilogue: the pages write C from the compute threads once their K loop
//    ends. On the 128 x 128 row the compute warps instead store the finished
//    tile into a shared-memory staging tile and go on with the next one, and
//    two epilogue warps write the staged tile out (alpha / beta into C, or raw
//    split-K / stream-K partials) meanwhile; the other rows, whose 2-3 CTAs per
//    SM leave no room for a staging tile, write from the compute warps.
//  * Watchdog: every mbarrier wait is bounded; on expiry the CTA records
//    SGEMM_ERR_TIMEOUT in the status word, waits (bounded) for its own copies
//    in flight and returns — it never traps or spins forever.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>
#include <type_traits>

#include "device_ptx.cuh"
#include "schedule.cuh"
#include "sgemm_internal.h"

namespace sgemm_impl {
namespace {

using namespace sgemm_dev;
using sgemm_cfg::kFfmaBK;

constexpr int kTimeoutCode = 5 << 16;       // SGEMM_ERR_TIMEOUT << 16
constexpr int kNotSupportedCode = 7 << 16;  // SGEMM_ERR_NOT_SUPPORTED << 16

// Where the mainloop's A operand comes from (plan.transpose_a):
//  kAKMajor  A as given, staged K-major (128-byte swizzle), FFMA2 form (a_m, a_m) * (b_n, b_n+1);
//  kAMMajor  A^T written to the workspace by transpose_kernel first, staged M-major like B;
//  kASmemT   A as given, staged K-major, then turned M-major in shared memory by a
//            transposer warp; the compute warps read it like A^T.
enum : int { kAKMajor = 0, kAMMajor = 1, kASmemT = 2 };

template <int BM_, int BN_, int STAGES_, int MINB_, int EPI_ = 0, int XB_ = 0>
struct Tile {
    static constexpr int BM = BM_, BN = BN_, STAGES = STAGES_, MINB = MINB_, BK = kFfmaBK;
    static constexpr int EPI = EPI_;  // > 0: a staging tile and EPI epilogue warps
    static constexpr int XB = XB_;    // > 0: XB M-major A buffers and a transposer warp (kASmemT)
    static constexpr int WM = 32, WN = 64;
    static constexpr int WARPS_M = BM / WM, WARPS_N = BN / WN;
    static constexpr int CONSUMERS = WARPS_M * WARPS_N;
    static constexpr int THREADS = (CONSUMERS + 1 + (XB > 0 ? 1 : 0) + EPI) * 32;
    static constexpr int A_BYTES = BM * BK * 4;
    static constexpr int B_BYTES = BK * BN * 4;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int XBUF_BYTES = XB * A_BYTES;
    static constexpr int STAGING_BYTES = (EPI > 0 ? 1 : 0) * BM * BN * 4;
    static constexpr int SMEM_BYTES = sgemm_cfg::ffma_smem_bytes(BM, BN, STAGES, EPI, XB);
    static_assert(EPI == 0 || (BN == 128 && BM % EPI == 0),
                  "an epilogue warp moves one 16-byte word of a staged row per lane, whole rows per warp");
    static_assert(BM % WM == 0 && BN % WN == 0, "CTA tile must be a multiple of the warp tile");
    static_assert(BM <= 256 && BN <= 256, "a TMA box side is at most 256 elements");
    static_assert(A_BYTES % 1024 == 0, "A stages must keep the 1024-byte swizzle alignment");
    static_assert(XB == 0 || (BM == 64 || BM == 128), "the transposer warp covers 64 or 128 rows per slab");
};

template <class T, int AL>
__device__ __forceinline__ void producer_loop(const CUtensorMap *tmA, const CUtensorMap *tmB,
                                              const FfmaParams &p, uint32_t a_base, uint32_t b_base,
                                              uint32_t bar_base, volatile int *abort_flag)
{
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0, issued_parity = 0;  // per stage: has a copy outstanding, and its phase parity
    int seq = 0;
    bool ok = true;
    pdl_wait();  // the operands written by this call's transpose / repack are complete
    Work w;
    for (int item = 0; ok && work_at(p, item, w); ++item) {
        const int tm = w.tm, tn = w.tn;
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
            const uint32_t full = bar_base + 8 * stage;
            const uint32_t empty = bar_base + 8 * (T::STAGES + stage);
            if (!mbar_wait_bounded(empty, phase ^ 1u, abort_flag, p.timeout_ns)) {
                if (!*abort_flag) {
                    *abort_flag = 1;
                    report_status(p.status, kTimeoutCode | kWhereProducerEmpty);
                }
                ok = false;
                break;
            }
            if (p.skew_ns > 0) __nanosleep(static_cast<unsigned>(p.skew_ns));
            const bool skip = (p.inject_skip >= 0 && blockIdx.x == 0 && seq == p.inject_skip);
            if (!skip) {
                // a box outside the problem would only read fill values: recorded, not skipped
                index_ok(tm < p.tiles_m && tn < p.tiles_n && kb < p.kblocks, p.status, kWhereIdxCopy);
                mbar_arrive_expect_tx(full, T::STAGE_BYTES);
                if (AL == kAMMajor)  // A^T slab: BK rows of k, BM consecutive m
                    tma_load_2d(a_base + stage * T::A_BYTES, tmA, full, tm * T::BM, kb * T::BK);
                else  // A slab: BM rows of m, BK consecutive k (128-byte swizzle)
                    tma_load_2d(a_base + stage * T::A_BYTES, tmA, full, kb * T::BK, tm * T::BM);
                tma_load_2d(b_base + stage * T::B_BYTES, tmB, full, tn * T::BN, kb * T::BK);
                issued |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
            }
            ++seq;
            if (++stage == T::STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    pdl_trigger();  // every copy is issued: the call's reduction may become resident
    // No copy of ours may still be writing this CTA's shared memory when it exits.
    for (int s = 0; s < T::STAGES; ++s) {
        if (issued >> s & 1u) {
            if (!mbar_wait_bounded(bar_base + 8 * s, issued_parity >> s & 1u, nullptr, p.timeout_ns))
                report_status(p.status, kTimeoutCode | kWhereDrain);
        }
    }
}

// Register accumulator of a thread's 8 x 8 outputs as 32 FFMA2 pairs: with A^T,
// acc[ip][j] = rows (2ip, 2ip+1) of column j; with K-major A, acc[i][jp] =
// row i, columns (2jp, 2jp+1).
template <bool AT>
using Acc = std::conditional_t<AT, float2[4][8], float2[8][4]>;

// Local row (within the warp tile) of a thread's output row i = 0..7.
template <bool AT>
__device__ __forceinline__ int out_row(int r, int i)
{
    return AT ? 4 * r + (i & 3) + 16 * (i >> 2) : r + 4 * i;
}

// Outputs of row i, columns 4c..4c+3 (h = 0) or 32+4c..32+4c+3 (h = 1).
__device__ __forceinline__ float4 out4(const float2 (&acc)[4][8], int i, int h)
{
    const int ip = i >> 1;
    if (i & 1) return make_float4(acc[ip][4 * h].y, acc[ip][4 * h + 1].y, acc[ip][4 * h + 2].y, acc[ip][4 * h + 3].y);
    return make_float4(acc[ip][4 * h].x, acc[ip][4 * h + 1].x, acc[ip][4 * h + 2].x, acc[ip][4 * h + 3].x);
}
__device__ __forceinline__ float4 out4(const float2 (&acc)[8][4], int i, int h)
{
    return make_float4(acc[i][2 * h].x, acc[i][2 * h].y, acc[i][2 * h + 1].x, acc[i][2 * h + 1].y);
}

// One BK = 32 slab of A^T and B: 8 chunks of 4 k. Per k a thread loads two
// 128-bit words of A^T (its rows 4r.. and 16+4r..) and two of B (its columns
// 4c.. and 32+4c..), then issues 4 x 8 FFMA2 (a_m, a_m+1) * (b_n, b_n).
template <class T>
__device__ __forceinline__ void compute_slab_mmajor(const float *__restrict__ a_cols,
                                                    const float *__restrict__ b_cols, float2 (&acc)[4][8])
{
#pragma unroll
    for (int kc = 0; kc < 8; ++kc) {
        float4 a[4][2], b[4][2];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            a[kk][0] = *reinterpret_cast<const float4 *>(a_cols + (kc * 4 + kk) * T::BM);
            a[kk][1] = *reinterpret_cast<const float4 *>(a_cols + (kc * 4 + kk) * T::BM + 16);
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            b[kk][0] = *reinterpret_cast<const float4 *>(b_cols + (kc * 4 + kk) * T::BN);
            b[kk][1] = *reinterpret_cast<const float4 *>(b_cols + (kc * 4 + kk) * T::BN + 32);
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const float2 ap[4] = {make_float2(a[kk][0].x, a[kk][0].y), make_float2(a[kk][0].z, a[kk][0].w),
                                  make_float2(a[kk][1].x, a[kk][1].y), make_float2(a[kk][1].z, a[kk][1].w)};
            const float bv[8] = {b[kk][0].x, b[kk][0].y, b[kk][0].z, b[kk][0].w,
                                 b[kk][1].x, b[kk][1].y, b[kk][1].z, b[kk][1].w};
#pragma unroll
            for (int ip = 0; ip < 4; ++ip)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[ip][j] = __ffma2_rn(ap[ip], make_float2(bv[j], bv[j]), acc[ip][j]);
        }
    }
}

// One BK = 32 slab of K-major A and B: 8 chunks of 4 k. Per chunk a thread
// loads its 8 rows of A (one 128-bit load each: 4 consecutive k) and 4 x 2
// 128-bit loads of B, then issues 4 * 8 * 4 = 128 FFMA2 (a_m, a_m) * (b_n, b_n+1).
template <class T>
__device__ __forceinline__ void compute_slab_kmajor(const float *__restrict__ a_rows,
                                             const float *__restrict__ b_cols, int r,
                                             float2 (&acc)[8][4])
{
#pragma unroll
    for (int kc = 0; kc < 8; ++kc) {
        // 128-byte swizzle: 16-byte chunk q of row `row` sits at chunk q ^ (row & 7).
        // This thread's rows have row & 7 == r (even i) or r + 4 (odd i).
        const int off_even = (kc ^ r) << 2;
        const int off_odd = ((kc ^ 4) ^ r) << 2;
        float4 a[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            a[i] = *reinterpret_cast<const float4 *>(a_rows + i * 4 * T::BK + ((i & 1) ? off_odd : off_even));
        float4 b[4][2];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            b[kk][0] = *reinterpret_cast<const float4 *>(b_cols + (kc * 4 + kk) * T::BN);
            b[kk][1] = *reinterpret_cast<const float4 *>(b_cols + (kc * 4 + kk) * T::BN + 32);
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const float2 b0 = make_float2(b[kk][0].x, b[kk][0].y);
            const float2 b1 = make_float2(b[kk][0].z, b[kk][0].w);
            const float2 b2 = make_float2(b[kk][1].x, b[kk][1].y);
            const float2 b3 = make_float2(b[kk][1].z, b[kk][1].w);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float av = kk == 0 ? a[i].x : kk == 1 ? a[i].y : kk == 2 ? a[i].z : a[i].w;
                const float2 a2 = make_float2(av, av);
                acc[i][0] = __ffma2_rn(a2, b0, acc[i][0]);
                acc[i][1] = __ffma2_rn(a2, b1, acc[i][1]);
                acc[i][2] = __ffma2_rn(a2, b2, acc[i][2]);
                acc[i][3] = __ffma2_rn(a2, b3, acc[i][3]);
            }
        }
    }
}

__device__ __forceinline__ float4 axpby4(float alpha, float4 v, float beta, float4 c)
{
    return make_float4(fmaf(alpha, v.x, beta * c.x), fmaf(alpha, v.y, beta * c.y),
                       fmaf(alpha, v.z, beta * c.z), fmaf(alpha, v.w, beta * c.w));
}

// C[row, col..col+3] = alpha * v + beta * C (beta == 0: C not read), with
// per-element predication on the ragged N edge or when C is not 16-byte
// accessible ("Optimizing Matrix Multiplication in CUDA", 1D thread tiling
// epilogue; bounds predicates of "SGEMM CUDA kernel (First Half)", Part 2).
__device__ __forceinline__ void store_c4(const FfmaParams &p, int row, int col, float4 v)
{
    if (!index_ok(row >= 0 && row < p.M && col >= 0 && col < p.N, p.status, kWhereIdxStoreC)) return;
    float *dst = p.C + static_cast<long long>(row) * p.ldc + col;
    if (p.vec_c && col + 3 < p.N) {
        float4 out;
        if (p.beta != 0.0f)
            out = axpby4(p.alpha, v, p.beta, *reinterpret_cast<const float4 *>(dst));
        else
            out = make_float4(p.alpha * v.x, p.alpha * v.y, p.alpha * v.z, p.alpha * v.w);
        *reinterpret_cast<float4 *>(dst) = out;
    } else {
        const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (col + q < p.N) {
                dst[q] = (p.beta != 0.0f) ? fmaf(p.alpha, e[q], p.beta * dst[q]) : p.alpha * e[q];
            }
        }
    }
}

// The batched form of store_c4, C read first (load_c4) and written later
// (store_c4_loaded): used by the epilogue warps and by the A-as-given compute
// warps. The A^T compute warps keep store_c4 (load and store together): every
// batched variant changed the register allocation of that whole kernel and
// slowed its mainloop by more than it saved.
__device__ __forceinline__ float4 load_c4(const FfmaParams &p, int row, int col)
{
    const float *src = p.C + static_cast<long long>(row) * p.ldc + col;
    if (p.vec_c && col + 3 < p.N) return *reinterpret_cast<const float4 *>(src);
    float e[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) e[q] = col + q < p.N ? src[q] : 0.0f;
    return make_float4(e[0], e[1], e[2], e[3]);
}

__device__ __forceinline__ void store_c4_loaded(const FfmaParams &p, int row, int col, float4 v, float4 c)
{
    if (!index_ok(row >= 0 && row < p.M && col >= 0 && col < p.N, p.status, kWhereIdxStoreC)) return;
    float *dst = p.C + static_cast<long long>(row) * p.ldc + col;
    const float4 out = p.beta != 0.0f ? axpby4(p.alpha, v, p.beta, c)
                                      : make_float4(p.alpha * v.x, p.alpha * v.y, p.alpha * v.z, p.alpha * v.w);
    if (p.vec_c && col + 3 < p.N) {
        *reinterpret_cast<float4 *>(dst) = out;
    } else {
        const float e[4] = {out.x, out.y, out.z, out.w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (col + q < p.N) dst[q] = e[q];
    }
}

template <class T, bool AT>
__device__ __forceinline__ void epilogue(const FfmaParams &p, const Acc<AT> &acc, const Work &w, int wm, int wn,
                                         int r, int c)
{
    const int row0 = w.tm * T::BM + wm * T::WM;
    const int col0 = w.tn * T::BN + wn * T::WN + c * 4;
    if (w.dest == kToPartial) {
        // Stream-K partial: the whole partial tile, tile-packed (rows beyond M
        // or columns beyond N hold sums of the copy engine's zero fill).
        float *W = p.W + static_cast<long long>(w.idx) * (T::BM * T::BN);
        const int lr0 = wm * T::WM;
        const int lc0 = wn * T::WN + c * 4;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const long long e = static_cast<long long>(w.idx) * (T::BM * T::BN) +
                                    (lr0 + out_row<AT>(r, i)) * T::BN + lc0 + 32 * h;
                if (index_ok(w.idx >= 0 && e + 4 <= p.w_elems, p.status, kWhereIdxPartial))
                    *reinterpret_cast<float4 *>(W + (lr0 + out_row<AT>(r, i)) * T::BN + lc0 + 32 * h) =
                        out4(acc, i, h);
            }
        }
        return;
    }
    if (w.dest == kToSplit) {
        // Partial sums to this split's slice; the reduction applies alpha/beta.
        float *W = p.W + static_cast<long long>(w.idx) * p.wstride;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int row = row0 + out_row<AT>(r, i);
            if (row >= p.M) break;  // rows increase with i
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int col = col0 + 32 * h;
                const long long e = static_cast<long long>(w.idx) * p.wstride + static_cast<long long>(row) * p.ldw + col;
                if (col < p.N && index_ok(w.idx >= 0 && w.idx < p.splits && col + 4 <= p.ldw && e + 4 <= p.w_elems,
                                          p.status, kWhereIdxSplit)) {
                    *reinterpret_cast<float4 *>(W + static_cast<long long>(row) * p.ldw + col) = out4(acc, i, h);
                }
            }
        }
        return;
    }
    if constexpr (!AT) {
        // A-as-given kernel: the C loads of four rows (8 x 16 bytes) are issued
        // before any of their stores, so the tile's beta term costs two memory
        // latencies rather than one per row (loads cannot move past stores to
        // other rows by themselves: ldc is not known to keep the rows apart).
        // Measured at 4096^2 x 512, beta 0.5: 48.7 -> 43.8 us per round of tiles.
        // (In the A^T kernel every variant of this, including one row at a time
        // and read-only loads, changed the mainloop's register allocation and
        // cost more there than it saved: that epilogue stays one row at a time.)
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float4 cin[4][2];
            if (p.beta != 0.0f) {
#pragma unroll
                for (int ii = 0; ii < 4; ++ii) {
                    const int row = row0 + out_row<AT>(r, 4 * half + ii);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int col = col0 + 32 * h;
                        cin[ii][h] =
                            (row < p.M && col < p.N) ? load_c4(p, row, col) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    }
                }
            }
#pragma unroll
            for (int ii = 0; ii < 4; ++ii) {
                const int i = 4 * half + ii;
                const int row = row0 + out_row<AT>(r, i);
                if (row >= p.M) break;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int col = col0 + 32 * h;
                    if (col < p.N) store_c4_loaded(p, row, col, out4(acc, i, h), cin[ii][h]);
                }
            }
        }
        return;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int row = row0 + out_row<AT>(r, i);
        if (row >= p.M) break;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int col = col0 + 32 * h;
            if (col < p.N) store_c4(p, row, col, out4(acc, i, h));
        }
    }
}

// Staged epilogue (rows with epilogue warps). A consumer warp writes its 32 x 64
// part of the finished accumulator tile into the BM x BN staging tile (the
// layout of a tile-packed partial; each quarter-warp stores 128 contiguous
// bytes, so the 128-bit stores are conflict-free) and goes on with its next
// tile; the epilogue warps move the staging tile to its destination meanwhile.
template <class T, bool AT>
__device__ __forceinline__ void stage_tile(float *stg, const Acc<AT> &acc, int wm, int wn, int r, int c, int *status)
{
    const int lr0 = wm * T::WM;
    const int lc0 = wn * T::WN + c * 4;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int e = (lr0 + out_row<AT>(r, i)) * T::BN + lc0 + 32 * h;
            if (index_ok(e >= 0 && e + 4 <= T::BM * T::BN, status, kWhereIdxStaging))
                *reinterpret_cast<float4 *>(stg + e) = out4(acc, i, h);
        }
    }
}

// 16 bytes of the staging tile, by shared-memory address (an explicit
// shared-space load rather than a generic one; ordered with the memory accesses
// around it).
__device__ __forceinline__ float4 lds128(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void sts32(uint32_t addr, float v)
{
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// One staged K-major A slab (BM rows of 32 k, 128-byte swizzle: 16-byte chunk
// q of row m sits at chunk q ^ (m & 7)) rewritten M-major (32 rows of BM m),
// the layout the compute warps read A^T in. This is the pages' transposition of
// A on its way into shared memory ("SGEMM CUDA kernel (First Half)", Part 5),
// done by one warp after the copy engine has landed the slab, since TMA cannot
// transpose 4-byte elements.
//
// Lane l takes row m = 32 blk + l of each 32-row block: it loads the row's 8
// chunks of 4 k (16 bytes each) and stores each value on its own into M-major
// row k. A quarter-warp's 8 loads of chunk t read rows with 8 different
// (m & 7), so the swizzle puts them in 8 different 16-byte bank groups; a
// warp's 4-byte stores of one k cover 32 consecutive m, one bank each. Both
// sides are conflict-free and no value moves between registers.
template <class T>
__device__ __forceinline__ void transpose_slab(uint32_t src, uint32_t dst, int lane, int *status)
{
    const uint32_t s0 = src + static_cast<uint32_t>(lane * 128);
    const uint32_t d0 = dst + static_cast<uint32_t>(lane * 4);
    const int sw = lane & 7;  // m & 7 of every row this lane takes
#pragma unroll
    for (int blk = 0; blk < T::BM / 32; ++blk) {
        float4 v[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const int off = (32 * blk + lane) * 128 + ((t ^ sw) << 4);
            v[t] = index_ok(off >= 0 && off + 16 <= T::A_BYTES, status, kWhereIdxTranspose)
                       ? lds128(s0 + blk * 32 * 128 + ((t ^ sw) << 4))
                       : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const uint32_t d = d0 + static_cast<uint32_t>((4 * t * T::BM + 32 * blk) * 4);
            const int off = (4 * t * T::BM + 32 * blk + lane) * 4;
            if (!index_ok(off >= 0 && off + 3 * T::BM * 4 + 4 <= T::A_BYTES, status, kWhereIdxTranspose)) continue;
            sts32(d, v[t].x);
            sts32(d + T::BM * 4, v[t].y);
            sts32(d + 2 * T::BM * 4, v[t].z);
            sts32(d + 3 * T::BM * 4, v[t].w);
        }
    }
}

// The transposer warp (kASmemT): walks the CTA's k-slabs in the producer's
// order; for each, waits for the stage to land and for a free M-major buffer,
// transposes the A slab into it, then releases the stage's A (one arrival on
// its empty barrier, beside the compute warps' ones for B) and marks the buffer
// full. Bounded waits: on expiry it records the location and returns.
template <class T>
__device__ __forceinline__ void transposer_loop(const FfmaParams &p, uint32_t a_base, uint32_t x_base,
                                                uint32_t bar_base, uint32_t xbar_base, volatile int *abort_flag,
                                                int lane)
{
    int stage = 0, xs = 0;
    uint32_t phase = 0, xphase = 0;
    Work w;
    for (int item = 0; work_at(p, item, w); ++item) {
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
            const uint32_t full = bar_base + 8 * stage;
            const uint32_t xempty = xbar_base + 8 * (T::XB + xs);
            bool ok = mbar_wait_bounded(full, phase, abort_flag, p.timeout_ns) &&
                      mbar_wait_bounded(xempty, xphase ^ 1u, abort_flag, p.timeout_ns);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                if (lane == 0 && !*abort_flag) {
                    *abort_flag = 1;
                    report_status(p.status, kTimeoutCode | kWhereTransposer);
                }
                return;
            }
            if (p.skew_ns > 0) __nanosleep(static_cast<unsigned>(p.skew_ns));
            transpose_slab<T>(a_base + stage * T::A_BYTES, x_base + xs * T::A_BYTES, lane, p.status);
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar_base + 8 * (T::STAGES + stage));  // the stage's A has been read
                mbar_arrive(xbar_base + 8 * xs);                  // the M-major slab is written
            }
            if (++stage == T::STAGES) {
                stage = 0;
                phase ^= 1u;
            }
            if (++xs == T::XB) {
                xs = 0;
                xphase ^= 1u;
            }
        }
    }
}

// The epilogue warps: for every work item of the CTA, warp e writes rows
// [e BM / EPI, (e + 1) BM / EPI) of the staged tile (lane l: columns 4l..4l+3)
// to its destination: C with alpha / beta (the C loads of 8 rows issued before
// their stores), or raw to a split-K slice or a stream-K partial tile; then hands
// the staging tile back (one arrival per epilogue warp). (Prefetching the tile's
// C rows into L2 during its mainloop, and bulk asynchronous copies out of the
// staging tile, were measured and gained nothing.)
template <class T>
__device__ __forceinline__ void epilogue_warp_loop(const FfmaParams &p, uint32_t stg, uint32_t staged, uint32_t freed,
                                                   volatile int *abort_flag, int e, int lane)
{
    constexpr int ROWS = T::BM / T::EPI;
    const int lc = 4 * lane;
    const int lr_begin = e * ROWS;
    const uint32_t src0 = stg + static_cast<uint32_t>((lr_begin * T::BN + lc) * 4);
    Work w;
    for (int item = 0; work_at(p, item, w); ++item) {
        bool ok = mbar_wait_bounded(staged, static_cast<uint32_t>(item & 1), abort_flag, p.timeout_ns);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
            if (lane == 0 && !*abort_flag) {
                *abort_flag = 1;
                report_status(p.status, kTimeoutCode | kWhereStaging);
            }
            return;
        }
        if (!index_ok(lr_begin + ROWS <= T::BM && lc + 4 <= T::BN, p.status, kWhereIdxEpiRead)) {
            // (nothing of this tile is moved)
        } else if (w.dest == kToPartial) {
            float *W = p.W + static_cast<long long>(w.idx) * (T::BM * T::BN) + lr_begin * T::BN + lc;
            const long long e_last = static_cast<long long>(w.idx) * (T::BM * T::BN) + (lr_begin + ROWS - 1) * T::BN + lc;
            if (index_ok(w.idx >= 0 && e_last + 4 <= p.w_elems, p.status, kWhereIdxPartial)) {
#pragma unroll 8
                for (int lr = 0; lr < ROWS; ++lr)
                    *reinterpret_cast<float4 *>(W + lr * T::BN) = lds128(src0 + lr * T::BN * 4);
            }
        } else if (w.dest == kToSplit) {
            float *W = p.W + static_cast<long long>(w.idx) * p.wstride;
            const int col = w.tn * T::BN + lc;
            if (col < p.N) {
#pragma unroll 8
                for (int lr = 0; lr < ROWS; ++lr) {
                    const int row = w.tm * T::BM + lr_begin + lr;
                    if (row >= p.M) break;
                    const long long e = static_cast<long long>(w.idx) * p.wstride + static_cast<long long>(row) * p.ldw + col;
                    if (index_ok(w.idx >= 0 && w.idx < p.splits && col + 4 <= p.ldw && e + 4 <= p.w_elems, p.status,
                                 kWhereIdxSplit))
                        *reinterpret_cast<float4 *>(W + static_cast<long long>(row) * p.ldw + col) =
                            lds128(src0 + lr * T::BN * 4);
                }
            }
        } else {
            const int col = w.tn * T::BN + lc;
            if (col < p.N) {
                for (int lr0 = 0; lr0 < ROWS; lr0 += 8) {
                    float4 cin[8];
                    if (p.beta != 0.0f) {
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int row = w.tm * T::BM + lr_begin + lr0 + j;
                            cin[j] = row < p.M ? load_c4(p, row, col) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int row = w.tm * T::BM + lr_begin + lr0 + j;
                        if (row < p.M) store_c4_loaded(p, row, col, lds128(src0 + (lr0 + j) * T::BN * 4), cin[j]);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(freed);  // this warp's rows of the staging tile have been read
    }
}

// Split-K reduced within a thread-block cluster (p.cluster_split = S > 0): the
// cluster's S CTAs hold the S K slices of one tile (rank = slice). Each stages
// its raw partial tile in its own shared memory (the staging tile, or the
// drained stage ring on rows without one), then, after a cluster barrier, adds
// 1/S of the tile's elements over all S partials in slice order 0..S-1 through
// distributed shared memory and writes them to C with alpha / beta: the same
// additions, in the same order, as splitk_reduce_kernel does from a workspace,
// so the bits match the split-K path, without the workspace round trip or a
// second launch. A second cluster barrier keeps every CTA (and its shared
// memory) alive until its peers have read it. Run by the compute warps only
// (threads 0 .. CONSUMERS * 32 - 1); the other warps have exited, and exited
// threads do not take part in cluster barriers. `staged_ok` is false after a
// bounded wait ran out: the CTA then still meets both barriers (its peers would
// otherwise read the shared memory of an exited CTA) but writes nothing.
template <class T, bool AT>
__device__ __forceinline__ void cluster_split_epilogue(const FfmaParams &p, const Acc<AT> &acc, float *stg,
                                                       uint32_t layout_word, uint32_t layout, int wm, int wn, int r,
                                                       int c, bool staged_ok)
{
    constexpr int kThreads = T::CONSUMERS * 32;
    // every compute warp is done with the ring (its memory may hold the staged tile)
    named_barrier_or(1, kThreads, false);
    if (staged_ok) stage_tile<T, AT>(stg, acc, wm, wn, r, c, p.status);
    cluster_sync();
    const int S = p.cluster_split;
    // The partials are read at this CTA's own staging offset in every peer: all
    // CTAs of the launch must have laid out their shared memory alike.
    const int t = static_cast<int>(threadIdx.x);
    bool mismatch = false;
    // compared on the offset inside the CTA's shared memory (higher bits of a
    // shared::cta address differ between the CTAs of a cluster)
    constexpr uint32_t kOffsetMask = 0x3FFFFu;
    if (t < S)
        mismatch = ((ld_shared_cluster_u32(mapa_shared(layout_word, static_cast<uint32_t>(t))) ^ layout) & kOffsetMask) != 0;
    mismatch = named_barrier_or(1, kThreads, mismatch);
    if (mismatch && t == 0) report_status(p.status, kNotSupportedCode | kWhereClusterShape);
    if (staged_ok && !mismatch) {
        Work w;
        work_at(p, 0, w);
        const int rank = static_cast<int>(cluster_ctarank());
        constexpr int Q = T::BM * T::BN / 4;  // 16-byte groups of the tile-packed partial
        const int q1 = (rank + 1) * Q / S;
        const uint32_t base = smem_addr(stg);
        for (int q = rank * Q / S + t; q < q1; q += kThreads) {
            float4 v[8];
            if (!index_ok(q >= 0 && q < Q && S <= static_cast<int>(cluster_size()) && S <= 8, p.status, kWhereIdxCluster))
                continue;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (j < S) v[j] = ld_shared_cluster_v4(mapa_shared(base + static_cast<uint32_t>(q) * 16u, j));
            float4 sum = v[0];
#pragma unroll
            for (int j = 1; j < 8; ++j) {
                if (j < S) {
                    sum.x += v[j].x;
                    sum.y += v[j].y;
                    sum.z += v[j].z;
                    sum.w += v[j].w;
                }
            }
            const int lr = (4 * q) / T::BN, lc = (4 * q) % T::BN;
            const int row = w.tm * T::BM + lr, col = w.tn * T::BN + lc;
            if (row < p.M && col < p.N) store_c4(p, row, col, sum);
        }
    }
    cluster_sync();
}

// CL: the split-K-within-clusters form (p.cluster_split > 0), compiled as a
// kernel of its own so that the other forms' code, and their register
// allocation, do not carry its branches.
template <class T, int AL, bool CL = false>
__global__ void __launch_bounds__(T::THREADS, T::MINB)
ffma_sgemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const FfmaParams p)
{
    constexpr bool AT = AL != kAKMajor;  // the compute warps read A M-major
    static_assert((AL == kASmemT) == (T::XB > 0), "M-major A buffers exactly when A is transposed in shared memory");
    constexpr int XW = T::XB > 0 ? 1 : 0;  // transposer warps
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    unsigned char *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const float *sA = reinterpret_cast<const float *>(smem);
    const float *sB = reinterpret_cast<const float *>(smem + T::STAGES * T::A_BYTES);
    const float *sX = reinterpret_cast<const float *>(smem + T::STAGES * T::STAGE_BYTES);  // M-major A (XB)
    float *stg = reinterpret_cast<float *>(smem + T::STAGES * T::STAGE_BYTES + T::XBUF_BYTES);  // staging tile (EPI)
    unsigned char *bar_ptr = smem + T::STAGES * T::STAGE_BYTES + T::XBUF_BYTES + T::STAGING_BYTES;
    const uint32_t bar_base = smem_addr(bar_ptr);
    const uint32_t staged_bar = bar_base + 8 * (2 * T::STAGES);     // EPI: the consumers' arrivals
    const uint32_t freed_bar = bar_base + 8 * (2 * T::STAGES + 1);  // EPI: the epilogue warps' arrivals
    // XB: xfull[x] (the transposer's arrival), then xempty[x] (one arrival per consumer warp)
    const uint32_t xbar_base = bar_base + 8 * (2 * T::STAGES + (T::EPI > 0 ? 2 : 0));
    volatile int *abort_flag =
        reinterpret_cast<volatile int *>(bar_ptr + (2 * T::STAGES + (T::EPI > 0 ? 2 : 0) + 2 * T::XB) * 8);

    // split-K within clusters: the partial tile is staged in the staging tile, or
    // in the drained ring on rows without one; its offset goes into the layout
    // word beside the abort flag, which the cluster's CTAs compare
    float *cs_stage = T::EPI > 0 ? stg : reinterpret_cast<float *>(smem);
    static_assert(T::EPI > 0 || T::BM * T::BN * 4 <= T::STAGES * T::STAGE_BYTES, "a partial tile fits in the ring");
    const uint32_t layout_word = smem_addr(bar_ptr) + (2 * T::STAGES + (T::EPI > 0 ? 2 : 0) + 2 * T::XB) * 8 + 4;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (CL ? (p.cluster_split <= 0 || cluster_size() != static_cast<uint32_t>(p.cluster_split) ||
              p.splits != p.cluster_split || p.units != static_cast<int>(gridDim.x) || p.sk_tiles != 0)
           : p.cluster_split != 0) {
        // not launched as the plan's form (clusters of one unit per CTA, or no
        // clusters): do nothing (before any barrier or copy)
        if (threadIdx.x == 0) report_status(p.status, kNotSupportedCode | kWhereClusterShape);
        return;
    }

    if (threadIdx.x == 0) {
        if constexpr (CL)
            *reinterpret_cast<volatile uint32_t *>(bar_ptr + (2 * T::STAGES + (T::EPI > 0 ? 2 : 0) + 2 * T::XB) * 8 +
                                                   4) = smem_addr(cs_stage);
        for (int s = 0; s < T::STAGES; ++s) {
            mbar_init(bar_base + 8 * s, 1);                                 // full: producer's arrive + bytes
            mbar_init(bar_base + 8 * (T::STAGES + s), T::CONSUMERS + XW);  // empty: consumers (+ transposer)
        }
        if (T::EPI) {
            mbar_init(staged_bar, T::CONSUMERS);
            mbar_init(freed_bar, T::EPI);
        }
        for (int x = 0; x < T::XB; ++x) {
            mbar_init(xbar_base + 8 * x, 1);
            mbar_init(xbar_base + 8 * (T::XB + x), T::CONSUMERS);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == T::CONSUMERS && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    __syncthreads();

    if (warp == T::CONSUMERS) {
        if (lane == 0)
            producer_loop<T, AL>(&tmA, &tmB, p, smem_addr(sA), smem_addr(sB), bar_base, abort_flag);
        return;
    }
    if constexpr (T::XB > 0) {
        if (warp == T::CONSUMERS + 1) {
            transposer_loop<T>(p, smem_addr(sA), smem_addr(sX), bar_base, xbar_base, abort_flag, lane);
            return;
        }
    }
    if constexpr (T::EPI > 0) {
        if (warp > T::CONSUMERS + XW) {
            // (split-K within clusters: the compute warps write C themselves)
            if constexpr (!CL)
                epilogue_warp_loop<T>(p, smem_addr(stg), staged_bar, freed_bar, abort_flag,
                                      warp - T::CONSUMERS - 1 - XW, lane);
            return;
        }
    }

    const int wm = warp % T::WARPS_M;
    const int wn = warp / T::WARPS_M;
    const int r = lane >> 3;  // row group: rows wm*32 + out_row(r, i)
    const int c = lane & 7;   // column group: columns wn*64 + 4c + {0..3} and + 32
    // A slab of the current k-block: ring stage (kAKMajor, kAMMajor) or M-major buffer (kASmemT)
    const float *a_base = AL == kASmemT ? sX + wm * T::WM + 4 * r
                          : AT          ? sA + wm * T::WM + 4 * r
                                        : sA + (wm * T::WM + r) * T::BK;
    const float *b_cols_base = sB + wn * T::WN + c * 4;

    int stage = 0, xs = 0;
    uint32_t phase = 0, xphase = 0;
    for (int item = 0;; ++item) {
        int kb0, kb1;
        {
            Work w;
            if (!work_at(p, item, w)) break;
            kb0 = w.kb0;
            kb1 = w.kb1;
        }
        Acc<AT> acc;
        constexpr int kRows = AT ? 4 : 8;
#pragma unroll
        for (int i = 0; i < kRows; ++i)
#pragma unroll
            for (int j = 0; j < 32 / kRows; ++j) acc[i][j] = make_float2(0.0f, 0.0f);

        [[maybe_unused]] bool failed = false;
        for (int kb = kb0; kb < kb1; ++kb) {
            const uint32_t full = bar_base + 8 * stage;
            bool ok = mbar_wait_bounded(full, phase, abort_flag, p.timeout_ns);
            if constexpr (AL == kASmemT) ok = ok && mbar_wait_bounded(xbar_base + 8 * xs, xphase, abort_flag, p.timeout_ns);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                if (lane == 0 && !*abort_flag) {
                    *abort_flag = 1;
                    report_status(p.status, kTimeoutCode | kWhereConsumerFull);
                }
                if constexpr (CL) {  // still meet the cluster's barriers
                    failed = true;
                    break;
                }
                return;
            }
            index_ok(stage < T::STAGES && (AL != kASmemT || xs < T::XB), p.status, kWhereIdxRing);
            if constexpr (AL == kASmemT)
                compute_slab_mmajor<T>(a_base + xs * (T::A_BYTES / 4), b_cols_base + stage * (T::B_BYTES / 4), acc);
            else if constexpr (AT)
                compute_slab_mmajor<T>(a_base + stage * (T::A_BYTES / 4), b_cols_base + stage * (T::B_BYTES / 4), acc);
            else
                compute_slab_kmajor<T>(a_base + stage * (T::A_BYTES / 4), b_cols_base + stage * (T::B_BYTES / 4), r,
                                       acc);
            if (p.skew_ns < 0) __nanosleep(static_cast<unsigned>(-p.skew_ns));
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar_base + 8 * (T::STAGES + stage));
                if constexpr (AL == kASmemT) mbar_arrive(xbar_base + 8 * (T::XB + xs));
            }
            if (++stage == T::STAGES) {
                stage = 0;
                phase ^= 1u;
            }
            if constexpr (AL == kASmemT) {
                if (++xs == T::XB) {
                    xs = 0;
                    xphase ^= 1u;
                }
            }
        }
        if constexpr (CL) {  // one unit per CTA
            cluster_split_epilogue<T, AT>(p, acc, cs_stage, layout_word, smem_addr(cs_stage), wm, wn, r, c, !failed);
            return;
        }
        if constexpr (T::EPI != 0) {
            // wait until the epilogue warp has read the previous tile out of the staging tile
            bool ok = mbar_wait_bounded(freed_bar, static_cast<uint32_t>(item & 1) ^ 1u, abort_flag, p.timeout_ns);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                if (lane == 0 && !*abort_flag) {
                    *abort_flag = 1;
                    report_status(p.status, kTimeoutCode | kWhereStaging);
                }
                return;
            }
            stage_tile<T, AT>(stg, acc, wm, wn, r, c, p.status);
            __syncwarp();
            if (lane == 0) mbar_arrive(staged_bar);
        } else {
            Work w;  // recomputed here so that only `item` stays live across the mainloop
            work_at(p, item, w);
            epilogue<T, AT>(p, acc, w, wm, wn, r, c);
        }
    }
}

// Table row i in both ring forms: R (A staged for the compute warps) and X (A
// transposed in shared memory by a transposer warp, fewer ring stages).
template <int I>
struct Row {
    static constexpr sgemm_cfg::TileConfig c = sgemm_cfg::kFfmaConfigs[I];
    using R = Tile<c.bm, c.bn, c.stages, c.ctas_per_sm, c.epilogue_warps>;
    using X = Tile<c.bm, c.bn, c.xstages, c.ctas_per_sm, c.epilogue_warps, c.xbufs>;
    static_assert(R::THREADS == c.threads && R::SMEM_BYTES == c.smem_bytes && X::THREADS == c.xthreads &&
                      X::SMEM_BYTES == c.xsmem_bytes,
                  "kernel instantiations must match the tile-config table");
};
static_assert(sgemm_cfg::kNumFfmaConfigs == 4, "one instantiation per table row");

template <int I>
cudaError_t set_attr()
{
    using R = typename Row<I>::R;
    using X = typename Row<I>::X;
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(ffma_sgemm_kernel<R, kAMMajor>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  R::SMEM_BYTES)) != cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(ffma_sgemm_kernel<R, kAKMajor>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  R::SMEM_BYTES)) != cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(ffma_sgemm_kernel<X, kASmemT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  X::SMEM_BYTES)) != cudaSuccess)
        return e;
    return cudaFuncSetAttribute(ffma_sgemm_kernel<X, kASmemT, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                X::SMEM_BYTES);
}

// Split-K within clusters (A transposed in shared memory only) launches its
// own kernel form in clusters of p.cluster_split CTAs along x.
template <int I>
cudaError_t launch(int a_layout, const CUtensorMap &tmA, const CUtensorMap &tmB, const FfmaParams &p, int grid,
                   cudaStream_t stream, bool dependent)
{
    using R = typename Row<I>::R;
    using X = typename Row<I>::X;
    if (p.cluster_split > 0) {
        const int cl = p.cluster_split;
        if (a_layout != kASmemT || cl > 8 || grid % cl != 0) return cudaErrorInvalidValue;
        return launch_kernel_cluster(dependent, cl, ffma_sgemm_kernel<X, kASmemT, true>, dim3(grid),
                                     dim3(X::THREADS), X::SMEM_BYTES, stream, tmA, tmB, p);
    }
    switch (a_layout) {
    case kAMMajor:
        return launch_kernel(dependent, ffma_sgemm_kernel<R, kAMMajor>, dim3(grid), dim3(R::THREADS), R::SMEM_BYTES,
                             stream, tmA, tmB, p);
    case kAKMajor:
        return launch_kernel(dependent, ffma_sgemm_kernel<R, kAKMajor>, dim3(grid), dim3(R::THREADS), R::SMEM_BYTES,
                             stream, tmA, tmB, p);
    case kASmemT:
        return launch_kernel(dependent, ffma_sgemm_kernel<X, kASmemT>, dim3(grid), dim3(X::THREADS), X::SMEM_BYTES,
                             stream, tmA, tmB, p);
    default: return cudaErrorInvalidValue;
    }
}

// ---------------------------------------------------------------------------
// Split-K reduction: C = alpha * sum_{s=0}^{S-1} W_s + beta * C, slices added
// in increasing s so the result depends only on (plan, S). One thread per 4
// consecutive columns of a row.
__global__ void splitk_reduce_kernel(const float *__restrict__ W, long long ldw, long long wstride, int splits,
                                     int M, int N, float alpha, float beta, float *__restrict__ C, long long ldc,
                                     int vec_c, long long w_elems, int *status)
{
    pdl_wait();  // the mainloop's slices are complete and visible
    const int n4 = (N + 3) >> 2;
    const long long total = static_cast<long long>(M) * n4;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int row = static_cast<int>(idx / n4);
        const int col = static_cast<int>(idx - static_cast<long long>(row) * n4) * 4;
        const float *w = W + static_cast<long long>(row) * ldw + col;
        if (!index_ok(col + 4 <= ldw && static_cast<long long>(splits - 1) * wstride + row * ldw + col + 4 <= w_elems,
                      status, kWhereIdxSplitReduce))
            continue;
        float4 s = __ldg(reinterpret_cast<const float4 *>(w));
        for (int q = 1; q < splits; ++q) {
            const float4 t = __ldg(reinterpret_cast<const float4 *>(w + q * wstride));
            s.x += t.x;
            s.y += t.y;
            s.z += t.z;
            s.w += t.w;
        }
        float *dst = C + static_cast<long long>(row) * ldc + col;
        if (vec_c && col + 3 < N) {
            float4 out;
            if (beta != 0.0f)
                out = axpby4(alpha, s, beta, *reinterpret_cast<const float4 *>(dst));
            else
                out = make_float4(alpha * s.x, alpha * s.y, alpha * s.z, alpha * s.w);
            *reinterpret_cast<float4 *>(dst) = out;
        } else {
            const float e[4] = {s.x, s.y, s.z, s.w};
            for (int q = 0; q < 4 && col + q < N; ++q)
                dst[q] = (beta != 0.0f) ? fmaf(alpha, e[q], beta * dst[q]) : alpha * e[q];
        }
    }
}

// Stream-K reduction (schedule.cuh): for every span tile covered by more than
// one CTA, C = alpha * sum_g P_g + beta * C with the partial tiles of the
// covering CTAs added in CTA order, which is k order. Serves the FFMA and the
// TF32 kernels (same raster, same partial-tile layout). Grid: blockIdx.y = span
// tile, blockIdx.x = 256 column quads of it, one per thread; each block works
// out the covering CTAs' partial-tile offsets once, in shared memory.
constexpr int kSkMaxShared = 64;  // covering CTAs whose offsets are kept in shared memory

__global__ void __launch_bounds__(256) sk_reduce_kernel(const FfmaParams p, int bm, int bn)
{
    __shared__ long long off[kSkMaxShared];
    pdl_wait();  // the mainloop's partial tiles are complete and visible
    const long long S = static_cast<long long>(p.sk_tiles) * p.kblocks;
    const long long G = p.sk_grid;
    const int rel = blockIdx.y;
    const long long start = static_cast<long long>(rel) * p.kblocks;
    const long long g0 = ((start + 1) * G - 1) / S;
    const long long g1 = ((start + p.kblocks) * G - 1) / S;
    if (g0 == g1) return;  // inside one CTA's range: written to C by the mainloop (whole block)
    const int nseg = static_cast<int>(g1 - g0 + 1);
    for (int j = threadIdx.x; j < nseg && j < kSkMaxShared; j += blockDim.x) {
        const long long g = g0 + j;
        off[j] = (2 * g + (rel == (g * S / G) / p.kblocks ? 0 : 1)) * bm * bn;  // slot of CTA g
    }
    __syncthreads();
    const int q4 = bn / 4;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= bm * q4) return;
    int tm, tn;
    decode_tile(p.tiles_m, p.tiles_n, p.units + rel, tm, tn);
    if (!p.vec_c) {
        // C not 16-byte accessible: the warp's 128 consecutive elements of the tile
        // (tile-packed order) go one per lane and 32 apart, so that every access to C
        // and to the partials is a coalesced 4-byte one; all partial loads come before
        // the C accesses (same sums, same order as below)
        const int lane = static_cast<int>(threadIdx.x & 31u);
        const int t0 = 4 * (e - lane) + lane;  // t0 + 96 < bm * bn: whole blocks per tile (launch_sk_reduce)
        bool in[4];
        long long cidx[4];
        float s[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int t = t0 + 32 * k;
            const int lr = t / bn, lc = t - lr * bn;
            const int row = tm * bm + lr, col = tn * bn + lc;
            in[k] = row < p.M && col < p.N &&
                    index_ok(off[0] >= 0 && off[0] + t < p.w_elems, p.status, kWhereIdxSkReduce);
            cidx[k] = static_cast<long long>(row) * p.ldc + col;
            s[k] = in[k] ? __ldg(p.W + off[0] + t) : 0.0f;
        }
        for (int j = 1; j < nseg; ++j) {
            long long o;
            if (j < kSkMaxShared) {
                o = off[j];
            } else {
                const long long g = g0 + j;
                o = (2 * g + (rel == (g * S / G) / p.kblocks ? 0 : 1)) * bm * bn;
            }
            if (!index_ok(o >= 0 && o + t0 + 96 < p.w_elems, p.status, kWhereIdxSkReduce)) continue;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (in[k]) s[k] += __ldg(p.W + o + t0 + 32 * k);
        }
        float c[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if (p.beta != 0.0f) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (in[k]) c[k] = p.C[cidx[k]];
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (in[k]) p.C[cidx[k]] = (p.beta != 0.0f) ? fmaf(p.alpha, s[k], p.beta * c[k]) : p.alpha * s[k];
        return;
    }
    const int lr = e / q4, lc = (e - lr * q4) * 4;
    const int row = tm * bm + lr, col = tn * bn + lc;
    if (row >= p.M || col >= p.N) return;
    const float *w = p.W + lr * bn + lc;
    if (!index_ok(off[0] >= 0 && off[0] + lr * bn + lc + 4 <= p.w_elems, p.status, kWhereIdxSkReduce)) return;
    float4 s = *reinterpret_cast<const float4 *>(w + off[0]);
    for (int j = 1; j < nseg; ++j) {
        long long o;
        if (j < kSkMaxShared) {
            o = off[j];
        } else {
            const long long g = g0 + j;
            o = (2 * g + (rel == (g * S / G) / p.kblocks ? 0 : 1)) * bm * bn;
        }
        if (!index_ok(o >= 0 && o + lr * bn + lc + 4 <= p.w_elems, p.status, kWhereIdxSkReduce)) continue;
        const float4 v = *reinterpret_cast<const float4 *>(w + o);
        s.x += v.x;
        s.y += v.y;
        s.z += v.z;
        s.w += v.w;
    }
    store_c4(p, row, col, s);
}

// C = beta * C for K == 0 or alpha == 0 (beta == 0 writes +0 without reading C).
__global__ void scale_kernel(int M, int N, float beta, float *__restrict__ C, long long ldc)
{
    const long long total = static_cast<long long>(M) * N;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long row = idx / N;
        const long long col = idx - row * N;
        float *dst = C + row * ldc + col;
        *dst = (beta != 0.0f) ? beta * *dst : 0.0f;
    }
}

// dst (rows x cols, row stride ldd) = src (row stride lds): gives an operand a
// 16-byte-aligned base and row stride so the TMA path can read it.
constexpr int kRepackThreads = 256, kRepackPerThread = 8;
constexpr int kRepackChunk = kRepackThreads * kRepackPerThread;  // columns per work item

// Work item `it` = (row, chunk of kRepackChunk columns) of a repack: the block's
// threads stride along the chunk (coalesced on both sides; kRepackThreads threads),
// kRepackPerThread loads in flight per thread before any store.
__device__ __forceinline__ void repack_item(const float *__restrict__ src, long long lds, float *__restrict__ dst,
                                            long long ldd, int cols, long long nchunks, long long it)
{
    const long long row = it / nchunks;
    const int c0 = static_cast<int>(it - row * nchunks) * kRepackChunk;
    const int c1 = min(cols, c0 + kRepackChunk);
    const float *s = src + row * lds;
    float *d = dst + row * ldd;
    float v[kRepackPerThread];
#pragma unroll
    for (int j = 0; j < kRepackPerThread; ++j) {
        const int col = c0 + static_cast<int>(threadIdx.x) + j * kRepackThreads;
        if (col < c1) v[j] = __ldg(s + col);
    }
#pragma unroll
    for (int j = 0; j < kRepackPerThread; ++j) {
        const int col = c0 + static_cast<int>(threadIdx.x) + j * kRepackThreads;
        if (col < c1) d[col] = v[j];
    }
}

__global__ void repack_kernel(const float *__restrict__ src, long long lds, float *__restrict__ dst, long long ldd,
                              int rows, int cols)
{
    pdl_trigger();  // the call's mainloop may become resident; it waits for this grid to finish
    const long long nchunks = (cols + kRepackChunk - 1) / kRepackChunk;
    const long long items = static_cast<long long>(rows) * nchunks;
    for (long long it = blockIdx.x; it < items; it += gridDim.x) repack_item(src, lds, dst, ldd, cols, nchunks, it);
}

// The 64 x 64 tile of X at (r0, c0) into XT (cols x ldxt) = X^T through shared
// memory, so both the reads of X rows and the writes of XT rows are coalesced;
// interior tiles move 16 bytes per thread access when X allows it (VEC: X 16-byte
// aligned and ldx % 4 == 0; ldxt is always a multiple of 4). 256 threads; ends
// with a barrier, so the tile can be reused at once.
template <bool VEC>
__device__ __forceinline__ void transpose_tile(const float *__restrict__ X, long long ldx, float *__restrict__ XT,
                                               long long ldxt, int rows, int cols, int r0, int c0,
                                               float (&tile)[64][65])
{
    const int t = threadIdx.x;
    const bool interior = VEC && r0 + 64 <= rows && c0 + 64 <= cols;
    if (interior) {
        const int c = (t % 16) * 4;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int r = t / 16 + 16 * q;
            const float4 v = *reinterpret_cast<const float4 *>(X + static_cast<long long>(r0 + r) * ldx + c0 + c);
            tile[r][c] = v.x;
            tile[r][c + 1] = v.y;
            tile[r][c + 2] = v.z;
            tile[r][c + 3] = v.w;
        }
        __syncthreads();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int n = t / 16 + 16 * q;
            *reinterpret_cast<float4 *>(XT + static_cast<long long>(c0 + n) * ldxt + r0 + c) =
                make_float4(tile[c][n], tile[c + 1][n], tile[c + 2][n], tile[c + 3][n]);
        }
    } else {
        for (int e = t; e < 64 * 64; e += 256) {
            const int r = e / 64, c = e % 64;
            if (r0 + r < rows && c0 + c < cols) tile[r][c] = X[static_cast<long long>(r0 + r) * ldx + c0 + c];
        }
        __syncthreads();
        for (int e = t; e < 64 * 64; e += 256) {
            const int n = e / 64, k = e % 64;
            if (c0 + n < cols && r0 + k < rows) XT[static_cast<long long>(c0 + n) * ldxt + r0 + k] = tile[k][n];
        }
    }
    __syncthreads();  // the tile is reused by the next row block
}

// XT = X^T (see transpose_tile), grid-stride over tile rows, so any row count fits
// the grid's y limit. Gives the FFMA mainloop A^T.
template <bool VEC>
__global__ void __launch_bounds__(256) transpose_kernel(const float *__restrict__ X, long long ldx,
                                                        float *__restrict__ XT, long long ldxt, int rows, int cols)
{
    __shared__ float tile[64][65];
    pdl_trigger();  // the call's mainloop may become resident; it waits for this grid to finish
    const int c0 = blockIdx.x * 64;
    for (long long r0l = blockIdx.y * 64LL; r0l < rows; r0l += gridDim.y * 64LL)
        transpose_tile<VEC>(X, ldx, XT, ldxt, rows, cols, static_cast<int>(r0l), c0, tile);
}

// Both operand copies of a call in one launch (instead of one launch each):
// blocks [0, a_blocks) do job A, the others job B. Job A is A^T (one 64 x 64 tile
// per block, a_transpose) or a repack of A (grid-stride over its items); job B is
// a repack of B. 256 threads.
struct PrepJobs {
    const float *a;
    long long lda;
    float *a_dst;
    long long a_ldd;
    int a_rows, a_cols;
    int a_transpose;  // 1: A^T (tiles of 64 x 64, one per block), 0: repack
    int a_vec;        // A^T: 16-byte accesses inside interior tiles
    int a_blocks;
    const float *b;
    long long ldb;
    float *b_dst;
    long long b_ldd;
    int b_rows, b_cols;
};

__global__ void __launch_bounds__(256) prep_kernel(const PrepJobs j)
{
    __shared__ float tile[64][65];
    pdl_trigger();  // the call's mainloop may become resident; it waits for this grid to finish
    const int bid = static_cast<int>(blockIdx.x);
    if (bid < j.a_blocks) {
        if (j.a_transpose) {
            const int tiles_c = (j.a_cols + 63) / 64;
            const int r0 = (bid / tiles_c) * 64, c0 = (bid % tiles_c) * 64;
            if (j.a_vec)
                transpose_tile<true>(j.a, j.lda, j.a_dst, j.a_ldd, j.a_rows, j.a_cols, r0, c0, tile);
            else
                transpose_tile<false>(j.a, j.lda, j.a_dst, j.a_ldd, j.a_rows, j.a_cols, r0, c0, tile);
        } else {
            const long long nchunks = (j.a_cols + kRepackChunk - 1) / kRepackChunk;
            const long long items = static_cast<long long>(j.a_rows) * nchunks;
            for (long long it = bid; it < items; it += j.a_blocks)
                repack_item(j.a, j.lda, j.a_dst, j.a_ldd, j.a_cols, nchunks, it);
        }
        return;
    }
    const int nb = static_cast<int>(gridDim.x) - j.a_blocks;
    const long long nchunks = (j.b_cols + kRepackChunk - 1) / kRepackChunk;
    const long long items = static_cast<long long>(j.b_rows) * nchunks;
    for (long long it = bid - j.a_blocks; it < items; it += nb)
        repack_item(j.b, j.ldb, j.b_dst, j.b_ldd, j.b_cols, nchunks, it);
}

int elementwise_grid(long long work, int threads, int num_sms)
{
    const long long blocks = (work + threads - 1) / threads;
    const long long cap = static_cast<long long>(num_sms) * 8;
    return static_cast<int>(blocks < 1 ? 1 : (blocks < cap ? blocks : cap));
}

}  // namespace

cudaError_t ffma_set_attributes()
{
    cudaError_t e;
    if ((e = set_attr<0>()) != cudaSuccess) return e;
    if ((e = set_attr<1>()) != cudaSuccess) return e;
    if ((e = set_attr<2>()) != cudaSuccess) return e;
    return set_attr<3>();
}

cudaError_t launch_ffma(int config, int a_layout, const CUtensorMap &tmA, const CUtensorMap &tmB,
                        const FfmaParams &p, int grid, cudaStream_t stream, bool dependent)
{
    switch (config) {
    case 0: return launch<0>(a_layout, tmA, tmB, p, grid, stream, dependent);
    case 1: return launch<1>(a_layout, tmA, tmB, p, grid, stream, dependent);
    case 2: return launch<2>(a_layout, tmA, tmB, p, grid, stream, dependent);
    case 3: return launch<3>(a_layout, tmA, tmB, p, grid, stream, dependent);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_splitk_reduce(const float *W, long long ldw, long long wstride, int splits, int M, int N,
                                 float alpha, float beta, float *C, long long ldc, int vec_c, int num_sms,
                                 cudaStream_t stream, long long w_elems, int *status)
{
    const long long work = static_cast<long long>(M) * ((N + 3) / 4);
    return launch_kernel(true, splitk_reduce_kernel, dim3(elementwise_grid(work, 256, num_sms)), dim3(256), 0, stream,
                         W, ldw, wstride, splits, M, N, alpha, beta, C, ldc, vec_c, w_elems, status);
}

cudaError_t launch_sk_reduce(const FfmaParams &p, int bm, int bn, int num_sms, cudaStream_t stream)
{
    (void)num_sms;
    if ((bm * bn) % 1024 != 0) return cudaErrorInvalidValue;  // whole blocks of 256 column quads per tile
    const dim3 grid(bm * (bn / 4) / 256, p.sk_tiles);  // sk_tiles < SMs * CTAs per SM
    return launch_kernel(true, sk_reduce_kernel, grid, dim3(256), 0, stream, p, bm, bn);
}

cudaError_t launch_scale(int M, int N, float beta, float *C, long long ldc, int num_sms, cudaStream_t stream)
{
    scale_kernel<<<elementwise_grid(static_cast<long long>(M) * N, 256, num_sms), 256, 0, stream>>>(M, N, beta, C,
                                                                                                     ldc);
    return cudaGetLastError();
}

cudaError_t launch_repack(const float *src, long long lds, float *dst, long long ldd, int rows, int cols,
                          int num_sms, cudaStream_t stream)
{
    const long long items = static_cast<long long>(rows) * ((cols + kRepackChunk - 1) / kRepackChunk);
    const long long cap = 8LL * num_sms;
    const int grid = static_cast<int>(items < 1 ? 1 : (items < cap ? items : cap));
    repack_kernel<<<grid, kRepackThreads, 0, stream>>>(src, lds, dst, ldd, rows, cols);
    return cudaGetLastError();
}

cudaError_t launch_prep(const float *A, long long lda, float *a_dst, long long a_ldd, int a_rows, int a_cols,
                        bool a_transpose, const float *B, long long ldb, float *b_dst, long long b_ldd, int b_rows,
                        int b_cols, int num_sms, cudaStream_t stream)
{
    PrepJobs j{};
    j.a = A;
    j.lda = lda;
    j.a_dst = a_dst;
    j.a_ldd = a_ldd;
    j.a_rows = a_rows;
    j.a_cols = a_cols;
    j.a_transpose = a_transpose ? 1 : 0;
    j.a_vec = (reinterpret_cast<uintptr_t>(A) & 15u) == 0 && lda % 4 == 0 && a_ldd % 4 == 0;
    j.b = B;
    j.ldb = ldb;
    j.b_dst = b_dst;
    j.b_ldd = b_ldd;
    j.b_rows = b_rows;
    j.b_cols = b_cols;
    const long long chunk = kRepackChunk;
    const long long b_items = static_cast<long long>(b_rows) * ((b_cols + chunk - 1) / chunk);
    long long a_blocks;
    if (a_transpose) {
        a_blocks = static_cast<long long>((a_rows + 63) / 64) * ((a_cols + 63) / 64);
    } else {
        const long long a_items = static_cast<long long>(a_rows) * ((a_cols + chunk - 1) / chunk);
        a_blocks = std::min<long long>(a_items, 4LL * num_sms);
    }
    const long long b_blocks = std::min<long long>(std::max<long long>(b_items, 1), 4LL * num_sms);
    if (a_blocks < 1 || a_blocks + b_blocks > INT_MAX) return cudaErrorInvalidValue;
    j.a_blocks = static_cast<int>(a_blocks);
    prep_kernel<<<static_cast<unsigned>(a_blocks + b_blocks), 256, 0, stream>>>(j);
    return cudaGetLastError();
}

cudaError_t launch_transpose(const float *X, long long ldx, float *XT, long long ldxt, int rows, int cols,
                             cudaStream_t stream)
{
    const int gy = (rows + 63) / 64;
    const dim3 grid((cols + 63) / 64, gy < 65535 ? gy : 65535);
    if ((reinterpret_cast<uintptr_t>(X) & 15u) == 0 && ldx % 4 == 0 && ldxt % 4 == 0)
        transpose_kernel<true><<<grid, 256, 0, stream>>>(X, ldx, XT, ldxt, rows, cols);
    else
        transpose_kernel<false><<<grid, 256, 0, stream>>>(X, ldx, XT, ldxt, rows, cols);
    return cudaGetLastError();
}

}  // namespace sgemm_impl
