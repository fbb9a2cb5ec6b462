// Flagged TF32 mode (SGEMM_MATH_TF32): C = alpha * A * B + beta * C on the
// 5th-generation tensor cores. A and B are read as TF32 (10 explicit mantissa
// bits), products are accumulated in FP32 in tensor memory (TMEM). It is never
// used unless the caller selects it, and is held to its own, looser bound.
//
// Structure (one CTA per SM, persistent over 128 x 256 output tiles, walking
// the work sequence of schedule.cuh: whole tiles, then the CTA's K slice of
// a stream-K span whose partial tiles sk_reduce_kernel adds in k order):
//   warp 0      TMA producer: A box (32 k x 128 rows, K-major, 128-byte
//               swizzle) and eight B boxes (32 n x 32 k each, MN-major: B as
//               stored, 128-byte swizzle of 32-byte chunks) into a 4-stage ring.
//   warp 1      MMA issuer: one thread issues 4 tcgen05.mma (K = 8 each) per
//               stage into one of two TMEM accumulators (128 lanes x 256
//               columns each), commits the stage back to the producer, and
//               commits a finished accumulator to the epilogue.
//   warps 2..5  epilogue: tcgen05.ld of their 32-lane quarter of the
//               accumulator, alpha/beta, stores to C; then hand the
//               accumulator back so the next tile's MMAs overlap this one's
//               stores.
// A (row-major M x K) is read K-major, B (row-major K x N) MN-major, both as the
// caller stores them (an operand whose base or row stride is not 16-byte
// aligned is first repacked into the handle's workspace).
//
// All waits are bounded; on expiry the CTA records SGEMM_ERR_TIMEOUT, lets its
// copies and MMAs in flight finish (bounded), frees its TMEM and returns.
#include <cuda_runtime.h>

#include <cstdint>

#include "device_ptx.cuh"
#include "tcgen05_ptx.cuh"
#include "schedule.cuh"
#include "sgemm_internal.h"

namespace sgemm_impl {
namespace {

using namespace sgemm_dev;

constexpr int kTimeoutCode = 5 << 16;  // SGEMM_ERR_TIMEOUT << 16
constexpr int BM = sgemm_cfg::kTf32BM, BN = sgemm_cfg::kTf32BN, BK = sgemm_cfg::kTf32BK;
constexpr int STAGES = sgemm_cfg::kTf32Stages;
constexpr int A_BYTES = BM * BK * 4;
constexpr int B_BYTES = BN * BK * 4;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int THREADS = sgemm_cfg::kTf32Threads;
constexpr int MMA_K = 8;                  // K of one tcgen05.mma .kind::tf32
constexpr uint32_t TMEM_COLS = 2 * BN;    // two accumulators
constexpr uint32_t IDESC = idesc_tf32(BM, BN, true);
// B is staged MN-major in boxes of 32 n x 32 k (4 KiB, 128-byte swizzle of 32-byte
// chunks), boxes along n 4 KiB apart.
constexpr int kBoxN = 32;
constexpr int B_BOX_BYTES = kBoxN * BK * 4;
static_assert(sgemm_cfg::tf32_smem_bytes() == 1024 + STAGES * STAGE_BYTES + 256, "smem layout");
static_assert(TMEM_COLS == 512, "two 128 x 256 FP32 accumulators fill TMEM");

struct Bars {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
    int issued[STAGES];
};
static_assert(sizeof(Bars) <= 256, "barrier block");

__device__ __forceinline__ void raise_abort(Bars *b, const Tf32Params &p, int where)
{
    volatile int *f = &b->abort_flag;
    if (!*f) {
        *f = 1;
        report_status(p.status, kTimeoutCode | where);
    }
}

// Epilogue of one accumulator row (a thread's TMEM lane: 256 columns), NB x 16
// columns per step: NB TMEM loads, one wait, then (beta != 0) all of the step's
// C loads before any use. Short K (few k-blocks per tile) makes the epilogue the
// critical path, so there NB = 4 keeps 16 loads in flight per thread; with long
// K it overlaps the next tile's mainloop and NB = 1 keeps its memory traffic
// from crowding the operand copies (measured: NB = 4 everywhere cost 2-4 % at
// 4096^3 and 8192^2 x 4096, and saved 44 % at K = 32).
constexpr int kShortK = 16;  // k-blocks of 32

template <int NB>
__device__ __forceinline__ void load_row_chunks(uint32_t t_col, uint32_t (&v)[NB][16])
{
#pragma unroll
    for (int j = 0; j < NB; ++j) tmem_ld_16(t_col + j * 16, v[j]);
#pragma unroll
    for (int j = 0; j < NB; ++j) tmem_wait_ld(v[j]);
}

// Raw partial row of a stream-K piece (tile-packed workspace row of BN floats).
template <int NB>
__device__ __forceinline__ void store_partial_row(uint32_t t_row, float *wrow)
{
#pragma unroll 1
    for (int ch = 0; ch < BN / 16; ch += NB) {
        uint32_t v[NB][16];
        load_row_chunks<NB>(t_row + ch * 16, v);
#pragma unroll
        for (int q = 0; q < 4 * NB; ++q) {
            const uint32_t *w = &v[q >> 2][4 * (q & 3)];
            *reinterpret_cast<float4 *>(wrow + ch * 16 + 4 * q) =
                make_float4(__uint_as_float(w[0]), __uint_as_float(w[1]), __uint_as_float(w[2]),
                            __uint_as_float(w[3]));
        }
    }
}

// C[row, tn*BN ...] = alpha * acc + beta * C (beta == 0: C not read).
template <int NB>
__device__ __forceinline__ void store_c_row(const Tf32Params &p, uint32_t t_row, int row, int tn)
{
    float *crow = p.C + static_cast<long long>(row) * p.ldc;
#pragma unroll 1
    for (int ch = 0; ch < BN / 16; ch += NB) {
        uint32_t v[NB][16];
        load_row_chunks<NB>(t_row + ch * 16, v);  // every lane: .sync.aligned
        if (row >= p.M) continue;
        const int colb = tn * BN + ch * 16;
        if (p.vec_c && colb + 16 * NB - 1 < p.N) {
            float4 c[4 * NB];
            if (p.beta != 0.0f) {
#pragma unroll
                for (int q = 0; q < 4 * NB; ++q) c[q] = *reinterpret_cast<const float4 *>(crow + colb + 4 * q);
            }
#pragma unroll
            for (int q = 0; q < 4 * NB; ++q) {
                const uint32_t *w = &v[q >> 2][4 * (q & 3)];
                const float4 acc = make_float4(__uint_as_float(w[0]), __uint_as_float(w[1]), __uint_as_float(w[2]),
                                               __uint_as_float(w[3]));
                float4 out;
                if (p.beta != 0.0f)
                    out = make_float4(fmaf(p.alpha, acc.x, p.beta * c[q].x), fmaf(p.alpha, acc.y, p.beta * c[q].y),
                                      fmaf(p.alpha, acc.z, p.beta * c[q].z), fmaf(p.alpha, acc.w, p.beta * c[q].w));
                else
                    out = make_float4(p.alpha * acc.x, p.alpha * acc.y, p.alpha * acc.z, p.alpha * acc.w);
                *reinterpret_cast<float4 *>(crow + colb + 4 * q) = out;
            }
        } else {
            // N edge or C not 16-byte accessible: element by element, every C load of
            // the step issued before any use (one memory latency per step, not one per
            // element)
            float c[16 * NB];
            if (p.beta != 0.0f) {
#pragma unroll
                for (int q = 0; q < 16 * NB; ++q) c[q] = colb + q < p.N ? crow[colb + q] : 0.0f;
            }
#pragma unroll
            for (int q = 0; q < 16 * NB; ++q) {
                const int col = colb + q;
                if (col < p.N) {
                    const float a = __uint_as_float(v[q >> 4][q & 15]);
                    crow[col] = (p.beta != 0.0f) ? fmaf(p.alpha, a, p.beta * c[q]) : p.alpha * a;
                }
            }
        }
    }
}

__global__ void __launch_bounds__(THREADS, 1)
tf32_sgemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const Tf32Params p)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    unsigned char *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t a_base = smem_addr(smem);
    const uint32_t b_base = a_base + STAGES * A_BYTES;
    Bars *bars = reinterpret_cast<Bars *>(smem + STAGES * STAGE_BYTES);
    volatile int *abort_flag = &bars->abort_flag;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_addr(&bars->full[s]), 1);
            mbar_init(smem_addr(&bars->empty[s]), 1);
            bars->issued[s] = 0;
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_addr(&bars->acc_full[b]), 1);
            mbar_init(smem_addr(&bars->acc_empty[b]), 4);
        }
        mbar_init(smem_addr(&bars->mma_done), 1);
        bars->abort_flag = 0;
        fence_barrier_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if (warp == 0) {
        tmem_alloc(smem_addr(&bars->tmem_base), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0 && lane == 0) {
        // ---- TMA producer ----
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        pdl_wait();  // operands repacked by this call's previous kernel are complete
        Work w;
        for (int item = 0; ok && work_at(p, item, w); ++item) {
            const int tm = w.tm, tn = w.tn;
            for (int kb = w.kb0; kb < w.kb1; ++kb) {
                const uint32_t full = smem_addr(&bars->full[stage]);
                if (!mbar_wait_bounded(smem_addr(&bars->empty[stage]), phase ^ 1u, abort_flag, p.timeout_ns)) {
                    raise_abort(bars, p, kWhereProducerEmpty);
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(full, STAGE_BYTES);
                tma_load_2d(a_base + stage * A_BYTES, &tmA, full, kb * BK, tm * BM);
#pragma unroll
                for (int j = 0; j < BN / kBoxN; ++j)
                    tma_load_2d(b_base + stage * B_BYTES + j * B_BOX_BYTES, &tmB, full, tn * BN + j * kBoxN, kb * BK);
                bars->issued[stage] = 2 | static_cast<int>(phase);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        pdl_trigger();  // every copy is issued: the call's reduction may become resident
        for (int s = 0; s < STAGES; ++s) {
            const int rec = bars->issued[s];
            if ((rec & 2) && !mbar_wait_bounded(smem_addr(&bars->full[s]), static_cast<uint32_t>(rec & 1), nullptr,
                                                p.timeout_ns))
                report_status(p.status, kTimeoutCode | kWhereDrain);
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer ----
        int stage = 0;
        uint32_t phase = 0;
        int it = 0;
        bool ok = true;
        Work w;
        for (int item = 0; ok && work_at(p, item, w); ++item, ++it) {
            const int buf = it & 1;
            const uint32_t acc_phase = static_cast<uint32_t>(it >> 1) & 1u;
            if (!mbar_wait_bounded(smem_addr(&bars->acc_empty[buf]), acc_phase ^ 1u, abort_flag, p.timeout_ns)) {
                raise_abort(bars, p, kWhereAccum);
                break;
            }
            tc_fence_after_sync();
            const uint32_t d_tmem = tmem + static_cast<uint32_t>(buf * BN);
            const int kb0 = w.kb0, kb1 = w.kb1;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait_bounded(smem_addr(&bars->full[stage]), phase, abort_flag, p.timeout_ns)) {
                    raise_abort(bars, p, kWhereMmaEmpty);
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t a_s = a_base + stage * A_BYTES;
                const uint32_t b_s = b_base + stage * B_BYTES;
#pragma unroll
                for (int k = 0; k < BK / MMA_K; ++k) {
                    // A: K advances 8 TF32 = 32 bytes inside the 128-byte swizzle atom;
                    // B: one 8-row (8 k) group = 1024 bytes.
                    mma_tf32(d_tmem, smem_desc_k_sw128(a_s + k * MMA_K * 4),
                             smem_desc_mn_sw128_32b(b_s + k * 1024, B_BOX_BYTES), IDESC, (kb != kb0 || k != 0) ? 1u : 0u);
                }
                mma_commit(smem_addr(&bars->empty[stage]));  // stage free once these MMAs are done
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            mma_commit(smem_addr(&bars->acc_full[buf]));
        }
        // Every MMA of ours must be finished before TMEM is released.
        mma_commit(smem_addr(&bars->mma_done));
        if (!mbar_wait_bounded(smem_addr(&bars->mma_done), 0u, nullptr, p.timeout_ns))
            report_status(p.status, kTimeoutCode | kWhereDrain);
    } else if (warp >= 2) {
        // ---- epilogue: warp w reads TMEM lanes 32 * (w % 4) .. + 31 ----
        const int quarter = warp & 3;
        int it = 0;
        Work w;
        for (int item = 0; work_at(p, item, w); ++item, ++it) {
            const int buf = it & 1;
            const uint32_t acc_phase = static_cast<uint32_t>(it >> 1) & 1u;
            bool ok = mbar_wait_bounded(smem_addr(&bars->acc_full[buf]), acc_phase, abort_flag, p.timeout_ns);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                if (lane == 0) raise_abort(bars, p, kWhereAccum);
                break;
            }
            tc_fence_after_sync();
            const int row = w.tm * BM + quarter * 32 + lane;
            const int tn = w.tn;
            const uint32_t t_row = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(buf * BN);
            if (w.dest == kToPartial) {
                // Stream-K piece: the raw partial tile, tile-packed (rows and columns
                // past M and N hold sums of the copy engine's zero fill); the
                // stream-K reduction adds the pieces in k order and applies alpha / beta.
                float *wrow = p.W + static_cast<long long>(w.idx) * (BM * BN) + (quarter * 32 + lane) * BN;
                if (p.kblocks <= kShortK)
                    store_partial_row<4>(t_row, wrow);
                else
                    store_partial_row<1>(t_row, wrow);
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&bars->acc_empty[buf]));
                continue;
            }
            if (p.kblocks <= kShortK)
                store_c_row<4>(p, t_row, row, tn);
            else
                store_c_row<1>(p, t_row, row, tn);
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&bars->acc_empty[buf]));
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 0) {
        __syncwarp();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// CTA-pair kernel (tcgen05 .cta_group::2). A cluster of two CTAs on two SMs
// computes 256 x 256 tiles: rank r stages rows [128 r, 128 r + 128) of the A
// slab (K-major) and columns [128 r, 128 r + 128) of the B slab (MN-major, four
// 32 n x 32 k boxes), both at the same shared-memory offsets in the two CTAs,
// and holds rows
// [128 r, 128 r + 128) of the accumulator in its own TMEM. One thread of rank 0
// issues M = 256, N = 256 MMAs that read both CTAs' stages and write both
// TMEMs. Barriers:
//   full[s]      rank 0 only: both CTAs' copies of stage s complete_tx on it
//                (rank 0 expects the bytes of both).
//   empty[s]     both CTAs: the MMAs that read stage s committed to both.
//   acc_full[b]  both CTAs: accumulator b holds a finished tile.
//   acc_empty[b] rank 0 only: the 4 epilogue warps of each CTA have read
//                accumulator b (8 arrivals, the peer's from the other SM).
// Every wait is bounded; a CTA whose wait runs out records SGEMM_ERR_TIMEOUT
// and stops; the two CTAs leave only through one final cluster barrier, after
// rank 0 saw its MMAs and both CTAs' copies finish (bounded), so no CTA exits
// while the other may still touch its shared memory or TMEM.
constexpr int PBM = sgemm_cfg::kTf32PairBM;
constexpr int PBN = sgemm_cfg::kTf32PairBN;
constexpr int PHALF_M = PBM / 2, PHALF_N = PBN / 2;
constexpr int PSTAGES = sgemm_cfg::kTf32PairStages;
constexpr int PA_BYTES = PHALF_M * BK * 4;
constexpr int PB_BYTES = PHALF_N * BK * 4;
constexpr int PSTAGE_BYTES = PA_BYTES + PB_BYTES;
constexpr uint32_t PIDESC = idesc_tf32(PBM, PBN, true);
constexpr int kLayoutCode = 7 << 16;  // SGEMM_ERR_NOT_SUPPORTED << 16
static_assert(PBN == BN, "the pair kernel's accumulator rows share the one-CTA epilogue (BN columns)");
static_assert(sgemm_cfg::tf32_pair_smem_bytes() == 1024 + PSTAGES * PSTAGE_BYTES + 256, "smem layout");

struct PairBars {
    uint64_t full[PSTAGES];
    uint64_t empty[PSTAGES];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    uint32_t ring_offset;  // this CTA's stage-ring address, compared with the peer's
    int abort_flag;
    int issued[PSTAGES];
};
static_assert(sizeof(PairBars) <= 256, "barrier block");

__device__ __forceinline__ void raise_abort_pair(PairBars *b, const Tf32Params &p, int code)
{
    volatile int *f = &b->abort_flag;
    if (!*f) {
        *f = 1;
        report_status(p.status, code);
    }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
tf32_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const Tf32Params p)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    unsigned char *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t a_base = smem_addr(smem);
    const uint32_t b_base = a_base + PSTAGES * PA_BYTES;
    PairBars *bars = reinterpret_cast<PairBars *>(smem + PSTAGES * PSTAGE_BYTES);
    volatile int *abort_flag = &bars->abort_flag;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int pair = static_cast<int>(cluster_id_x());
    const int pairs = static_cast<int>(cluster_count_x());

    if (threadIdx.x == 0) {
        for (int s = 0; s < PSTAGES; ++s) {
            mbar_init(smem_addr(&bars->full[s]), 1);
            mbar_init(smem_addr(&bars->empty[s]), 1);
            bars->issued[s] = 0;
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_addr(&bars->acc_full[b]), 1);
            mbar_init(smem_addr(&bars->acc_empty[b]), 8);
        }
        mbar_init(smem_addr(&bars->mma_done), 1);
        bars->abort_flag = 0;
        bars->ring_offset = a_base;
        fence_barrier_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if (warp == 0) {
        tmem_alloc_pair(smem_addr(&bars->tmem_base), TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers are initialised before any copy or arrive targets them
    tc_fence_after_sync();
    const uint32_t tmem = bars->tmem_base;
    // The MMAs address both CTAs' stages by rank 0's offsets, which must therefore
    // agree. Compared on the address bits a shared-memory descriptor holds (the
    // offset inside the CTA's shared memory; higher bits of a shared::cta address
    // can differ between the CTAs of a cluster).
    constexpr uint32_t kDescAddrMask = 0x3FFFFu;
    const uint32_t peer_ring = ld_shared_cluster_u32(mapa_shared(smem_addr(&bars->ring_offset), rank ^ 1u));
    const bool same_layout = ((peer_ring ^ a_base) & kDescAddrMask) == 0;
    if (!same_layout && threadIdx.x == 0) raise_abort_pair(bars, p, kLayoutCode | kWherePairLayout);

    if (!same_layout) {
        // both CTAs see the mismatch: no copies, no MMAs
    } else if (warp == 0 && lane == 0) {
        // ---- TMA producer (both CTAs): this CTA's halves of each stage ----
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        pdl_wait();  // operands repacked by this call's previous kernel are complete
        Work w;
        for (int item = 0; ok && work_at_g(p, item, w, pair, pairs); ++item) {
            const int row_a = w.tm * PBM + static_cast<int>(rank) * PHALF_M;
            const int col_b = w.tn * PBN + static_cast<int>(rank) * PHALF_N;
            for (int kb = w.kb0; kb < w.kb1; ++kb) {
                if (!mbar_wait_bounded(smem_addr(&bars->empty[stage]), phase ^ 1u, abort_flag, p.timeout_ns)) {
                    raise_abort_pair(bars, p, kTimeoutCode | kWhereProducerEmpty);
                    ok = false;
                    break;
                }
                const uint32_t full = mapa_shared(smem_addr(&bars->full[stage]), 0);  // rank 0's barrier
                if (rank == 0) mbar_arrive_expect_tx(smem_addr(&bars->full[stage]), 2 * PSTAGE_BYTES);
                tma_load_2d_pair(a_base + stage * PA_BYTES, &tmA, full, kb * BK, row_a);
#pragma unroll
                for (int j = 0; j < PHALF_N / kBoxN; ++j)
                    tma_load_2d_pair(b_base + stage * PB_BYTES + j * B_BOX_BYTES, &tmB, full, col_b + j * kBoxN,
                                     kb * BK);
                bars->issued[stage] = 2 | static_cast<int>(phase);
                if (++stage == PSTAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        pdl_trigger();  // every copy is issued: the call's reduction may become resident
        // Drain. Rank 0: both CTAs' copies of every issued stage have landed (they
        // complete on its full barriers). Both: unless aborted, the MMAs that read
        // them have committed to this CTA's empty barriers.
        for (int s = 0; s < PSTAGES; ++s) {
            const int rec = bars->issued[s];
            if (!(rec & 2)) continue;
            const uint32_t par = static_cast<uint32_t>(rec & 1);
            if (rank == 0 && !mbar_wait_cluster_bounded(smem_addr(&bars->full[s]), par, nullptr, p.timeout_ns)) {
                report_status(p.status, kTimeoutCode | kWhereDrain);
                break;
            }
            if (!*abort_flag && !mbar_wait_bounded(smem_addr(&bars->empty[s]), par, abort_flag, p.timeout_ns)) {
                report_status(p.status, kTimeoutCode | kWhereDrain);
                break;
            }
        }
    } else if (warp == 1 && lane == 0 && rank == 0) {
        // ---- MMA issuer (rank 0 only) ----
        int stage = 0;
        uint32_t phase = 0;
        int it = 0;
        bool ok = true;
        Work w;
        for (int item = 0; ok && work_at_g(p, item, w, pair, pairs); ++item, ++it) {
            const int buf = it & 1;
            const uint32_t acc_phase = static_cast<uint32_t>(it >> 1) & 1u;
            if (!mbar_wait_cluster_bounded(smem_addr(&bars->acc_empty[buf]), acc_phase ^ 1u, abort_flag,
                                           p.timeout_ns)) {
                raise_abort_pair(bars, p, kTimeoutCode | kWhereAccum);
                break;
            }
            tc_fence_after_sync();
            const uint32_t d_tmem = tmem + static_cast<uint32_t>(buf * PBN);
            const int kb0 = w.kb0, kb1 = w.kb1;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait_cluster_bounded(smem_addr(&bars->full[stage]), phase, abort_flag, p.timeout_ns)) {
                    raise_abort_pair(bars, p, kTimeoutCode | kWhereMmaEmpty);
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t a_s = a_base + stage * PA_BYTES;
                const uint32_t b_s = b_base + stage * PB_BYTES;
#pragma unroll
                for (int k = 0; k < BK / MMA_K; ++k)
                    mma_tf32_pair(d_tmem, smem_desc_k_sw128(a_s + k * MMA_K * 4),
                                  smem_desc_mn_sw128_32b(b_s + k * 1024, B_BOX_BYTES), PIDESC,
                                  (kb != kb0 || k != 0) ? 1u : 0u);
                mma_commit_pair_both(smem_addr(&bars->empty[stage]));  // stage free in both CTAs
                if (++stage == PSTAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            mma_commit_pair_both(smem_addr(&bars->acc_full[buf]));
        }
        // Every MMA (they write both CTAs' TMEM) is finished before either CTA frees it.
        mma_commit_pair_local(smem_addr(&bars->mma_done));
        if (!mbar_wait_bounded(smem_addr(&bars->mma_done), 0u, nullptr, p.timeout_ns))
            report_status(p.status, kTimeoutCode | kWhereDrain);
    } else if (warp >= 2) {
        // ---- epilogue (both CTAs): warp w reads TMEM lanes 32 * (w % 4) .. + 31 ----
        const int quarter = warp & 3;
        const int half_row = static_cast<int>(rank) * PHALF_M + quarter * 32 + lane;
        int it = 0;
        Work w;
        for (int item = 0; work_at_g(p, item, w, pair, pairs); ++item, ++it) {
            const int buf = it & 1;
            const uint32_t acc_phase = static_cast<uint32_t>(it >> 1) & 1u;
            bool ok = mbar_wait_cluster_bounded(smem_addr(&bars->acc_full[buf]), acc_phase, abort_flag, p.timeout_ns);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                if (lane == 0) raise_abort_pair(bars, p, kTimeoutCode | kWhereAccum);
                break;
            }
            tc_fence_after_sync();
            const uint32_t t_row = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(buf * PBN);
            if (w.dest == kToPartial) {
                // this CTA's rows of the pair's tile-packed 256 x 256 partial
                float *wrow = p.W + static_cast<long long>(w.idx) * (PBM * PBN) + static_cast<long long>(half_row) * PBN;
                if (p.kblocks <= kShortK)
                    store_partial_row<4>(t_row, wrow);
                else
                    store_partial_row<1>(t_row, wrow);
            } else {
                const int row = w.tm * PBM + half_row;
                if (p.kblocks <= kShortK)
                    store_c_row<4>(p, t_row, row, w.tn);
                else
                    store_c_row<1>(p, t_row, row, w.tn);
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_addr(&bars->acc_empty[buf]), 0));  // rank 0's
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();  // neither CTA leaves while the other may still use its barriers, stages or TMEM
    tc_fence_after_sync();
    if (warp == 0) {
        __syncwarp();
        tmem_dealloc_pair(tmem, TMEM_COLS);
    }
}

}  // namespace

cudaError_t tf32_set_attributes()
{
    cudaError_t e = cudaFuncSetAttribute(tf32_sgemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         sgemm_cfg::tf32_smem_bytes());
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(tf32_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                sgemm_cfg::tf32_pair_smem_bytes());
}

int tf32_pair_max_pairs()
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = sgemm_cfg::tf32_pair_smem_bytes();
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, tf32_pair_kernel, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return clusters;
}

cudaError_t launch_tf32_pair(const CUtensorMap &tmA, const CUtensorMap &tmB, const Tf32Params &p, int grid,
                             cudaStream_t stream, bool dependent)
{
    // grid = 2 x pairs; clusters of two come from the kernel's __cluster_dims__
    return launch_kernel(dependent, tf32_pair_kernel, dim3(grid), dim3(THREADS), sgemm_cfg::tf32_pair_smem_bytes(),
                         stream, tmA, tmB, p);
}

cudaError_t launch_tf32(const CUtensorMap &tmA, const CUtensorMap &tmB, const Tf32Params &p, int grid,
                        cudaStream_t stream, bool dependent)
{
    return launch_kernel(dependent, tf32_sgemm_kernel, dim3(grid), dim3(THREADS), sgemm_cfg::tf32_smem_bytes(),
                         stream, tmA, tmB, p);
}

}  // namespace sgemm_impl
