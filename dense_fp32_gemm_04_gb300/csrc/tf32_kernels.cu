// Flagged TF32 mode (SGEMM_MATH_TF32): C = alpha * A * B + beta * C on the
// 5th-generation tensor cores. A and B are read as TF32 (10 explicit mantissa
// bits), products are accumulated in FP32 in tensor memory (TMEM). It is never
// used unless the caller selects it, and is held to its own, looser bound.
//
// One kernel, two forms (the PAIR template flag), both persistent with one CTA
// per SM, walking the work sequence of schedule.cuh (whole tiles, then the
// worker's K slice of a stream-K span whose partial tiles sk_reduce_kernel adds
// in k order):
//   one CTA     a worker is a CTA computing 128 x 256 tiles with
//               tcgen05.mma.cta_group::1 (M = 128, N = 256, K = 8).
//   CTA pair    a worker is a cluster of two CTAs on two SMs computing 256 x 256
//               tiles with tcgen05.mma.cta_group::2 (M = 256, N = 256): rank r
//               stages rows [128 r, 128 r + 128) of the A slab and columns
//               [128 r, 128 r + 128) of the B slab at the same shared-memory
//               offsets in both CTAs and holds rows [128 r, 128 r + 128) of the
//               accumulator in its own TMEM; rank 0's MMAs read both CTAs'
//               stages and write both TMEMs. Per FMA each SM's shared memory
//               then carries a third less traffic than with one CTA per tile.
// Warps of every CTA:
//   warp 0      TMA producer: the CTA's A box (32 k x 128 rows, K-major,
//               128-byte swizzle) and B boxes (32 n x 32 k each, MN-major: B as
//               stored, 128-byte swizzle of 32-byte chunks) into the stage ring.
//   warp 1      MMA issuer (rank 0 only): one thread issues 4 tcgen05.mma
//               (K = 8 each) per stage into one of two TMEM accumulators (128
//               lanes x 256 columns each), commits the stage back to the
//               producers, and commits a finished accumulator to the epilogues.
//   warps 2..5  epilogue: tcgen05.ld of their 32-lane quarter of the CTA's
//               accumulator, alpha/beta, stores to C; then hand the accumulator
//               back so the next tile's MMAs overlap this one's stores.
// Barriers (in each CTA; for the pair, the MMA issuer's are rank 0's):
//   full[s]      both CTAs' copies of stage s complete_tx on rank 0's (rank 0
//                expects the bytes of both).
//   empty[s]     every CTA: the MMAs that read stage s committed (multicast to
//                both CTAs of a pair).
//   acc_full[b]  every CTA: accumulator b holds a finished tile (multicast).
//   acc_empty[b] rank 0: the epilogue warps of every CTA of the worker have read
//                accumulator b (4 or 8 arrivals, a peer's through its cluster
//                address).
// A (row-major M x K) is read K-major, B (row-major K x N) MN-major, both as the
// caller stores them (an operand whose base or row stride is not 16-byte
// aligned is first repacked into the handle's workspace).
//
// All waits are bounded; on expiry the CTA records SGEMM_ERR_TIMEOUT and stops.
// A CTA leaves only after its copies have landed and the MMAs reading its
// stages have committed (bounded waits), and the two CTAs of a pair only
// through one final cluster barrier, after rank 0 saw its MMAs finish, so no
// CTA exits while the other may still touch its shared memory or TMEM.
#include <cuda_runtime.h>

#include <cstdint>

#include "device_ptx.cuh"
#include "schedule.cuh"
#include "sgemm_internal.h"
#include "tcgen05_ptx.cuh"

namespace sgemm_impl {
namespace {

using namespace sgemm_dev;

constexpr int kTimeoutCode = 5 << 16;  // SGEMM_ERR_TIMEOUT << 16
constexpr int kLayoutCode = 7 << 16;   // SGEMM_ERR_NOT_SUPPORTED << 16
constexpr int BK = sgemm_cfg::kTf32BK;
constexpr int BN = sgemm_cfg::kTf32BN;    // columns of a tile and of a CTA's accumulator (both forms)
constexpr int THREADS = sgemm_cfg::kTf32Threads;
constexpr int MMA_K = 8;                  // K of one tcgen05.mma .kind::tf32
constexpr uint32_t TMEM_COLS = 2 * BN;    // two accumulators
// B is staged MN-major in boxes of 32 n x 32 k (4 KiB, 128-byte swizzle of 32-byte
// chunks), boxes along n 4 KiB apart.
constexpr int kBoxN = 32;
constexpr int B_BOX_BYTES = kBoxN * BK * 4;
static_assert(TMEM_COLS == 512, "two 128 x 256 FP32 accumulators fill TMEM");
static_assert(sgemm_cfg::kTf32PairBN == BN, "both forms keep 256 accumulator columns per CTA");

template <bool PAIR>
struct Tf32Shape {
    static constexpr int CTAS = PAIR ? 2 : 1;  // CTAs per worker
    static constexpr int BM = PAIR ? sgemm_cfg::kTf32PairBM : sgemm_cfg::kTf32BM;  // tile rows
    static constexpr int CTA_M = BM / CTAS;    // rows of A and of the accumulator per CTA
    static constexpr int CTA_N = BN / CTAS;    // columns of B staged per CTA
    static constexpr int STAGES = PAIR ? sgemm_cfg::kTf32PairStages : sgemm_cfg::kTf32Stages;
    static constexpr int A_BYTES = CTA_M * BK * 4;
    static constexpr int B_BYTES = CTA_N * BK * 4;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr uint32_t IDESC = idesc_tf32(BM, BN, true);
    static constexpr int SMEM = PAIR ? sgemm_cfg::tf32_pair_smem_bytes() : sgemm_cfg::tf32_smem_bytes();
    static_assert(CTA_M == 128, "an accumulator holds 128 TMEM lanes");
    static_assert(CTA_N % kBoxN == 0, "whole B boxes");
    static_assert(SMEM == 1024 + STAGES * STAGE_BYTES + 256, "smem layout");
};

template <int STAGES>
struct Tf32Bars {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    uint32_t ring_offset;  // this CTA's stage-ring address, compared with the peer's
    int abort_flag;
    int issued[STAGES];
};
static_assert(sizeof(Tf32Bars<sgemm_cfg::kTf32PairStages>) <= 256, "barrier block");
static_assert(sizeof(Tf32Bars<sgemm_cfg::kTf32Stages>) <= 256, "barrier block");

template <int STAGES>
__device__ __forceinline__ void raise_abort(Tf32Bars<STAGES> *b, const Tf32Params &p, int code)
{
    volatile int *f = &b->abort_flag;
    if (!*f) {
        *f = 1;
        report_status(p.status, code);
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
// Every lane loads (warp-collective TMEM loads); `ok` false skips this lane's stores
// (a failed index check of a debug build).
template <int NB>
__device__ __forceinline__ void store_partial_row(uint32_t t_row, float *wrow, bool ok)
{
#pragma unroll 1
    for (int ch = 0; ch < BN / 16; ch += NB) {
        uint32_t v[NB][16];
        load_row_chunks<NB>(t_row + ch * 16, v);
        if (!ok) continue;
#pragma unroll
        for (int q = 0; q < 4 * NB; ++q) {
            const uint32_t *w = &v[q >> 2][4 * (q & 3)];
            *reinterpret_cast<float4 *>(wrow + ch * 16 + 4 * q) =
                make_float4(__uint_as_float(w[0]), __uint_as_float(w[1]), __uint_as_float(w[2]),
                            __uint_as_float(w[3]));
        }
    }
}

// Shifted frame for a row of C that is not 16-byte aligned. With s the number of
// elements before the row's first 16-byte boundary (C itself is 4-byte aligned),
// the row is written in 4-element chunks at columns s - 4 + 4j: every chunk that
// lies wholly inside [0, lim) is one 16-byte access, the rest (the first chunk,
// the last one when s != 0, chunks past N) go element by element. The step's
// accumulator values come after the previous step's last four (x[0..3]), so
// chunk j of a step holds x[4j + s .. 4j + s + 3]; `pick` makes that runtime
// offset a choice among four registers (i is a constant once the loops unroll).
__device__ __forceinline__ float pick(const float *x, int i, int s)
{
    return s == 0 ? x[i] : s == 1 ? x[i + 1] : s == 2 ? x[i + 2] : x[i + 3];
}

__device__ __forceinline__ bool chunk_whole(int r0, int lim) { return r0 >= 0 && r0 + 3 < lim; }

__device__ __forceinline__ float4 load_chunk(const float *cbase, int r0, int lim)
{
    if (chunk_whole(r0, lim)) return *reinterpret_cast<const float4 *>(cbase + r0);
    float e[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) e[q] = (r0 + q >= 0 && r0 + q < lim) ? cbase[r0 + q] : 0.0f;
    return make_float4(e[0], e[1], e[2], e[3]);
}

__device__ __forceinline__ void store_chunk(const Tf32Params &p, float *cbase, int r0, int lim, const float (&a)[4],
                                            float4 c)
{
    float4 out;
    if (p.beta != 0.0f)
        out = make_float4(fmaf(p.alpha, a[0], p.beta * c.x), fmaf(p.alpha, a[1], p.beta * c.y),
                          fmaf(p.alpha, a[2], p.beta * c.z), fmaf(p.alpha, a[3], p.beta * c.w));
    else
        out = make_float4(p.alpha * a[0], p.alpha * a[1], p.alpha * a[2], p.alpha * a[3]);
    if (chunk_whole(r0, lim)) {
        *reinterpret_cast<float4 *>(cbase + r0) = out;
    } else {
        const float e[4] = {out.x, out.y, out.z, out.w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (r0 + q >= 0 && r0 + q < lim) cbase[r0 + q] = e[q];
    }
}

// The tile's part of row `row` of C (cbase = its first column, lim = the columns
// of the tile inside N) in the shifted frame; same steps and load batching as
// store_c_row.
template <int NB>
__device__ __forceinline__ void store_c_row_shifted(const Tf32Params &p, uint32_t t_row, int row, float *cbase,
                                                    int lim)
{
    const int s = static_cast<int>((4u - ((static_cast<uint32_t>(reinterpret_cast<uintptr_t>(cbase)) >> 2) & 3u)) & 3u);
    float x[16 * NB + 4];
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = 0.0f;
#pragma unroll 1
    for (int ch = 0; ch < BN / 16; ch += NB) {
        uint32_t v[NB][16];
        load_row_chunks<NB>(t_row + ch * 16, v);  // every lane: .sync.aligned
        if (row >= p.M) continue;
#pragma unroll
        for (int i = 0; i < 16 * NB; ++i) x[4 + i] = __uint_as_float(v[i >> 4][i & 15]);
        const int cb = ch * 16 + s - 4;  // column of chunk 0
        float4 c[4 * NB];
        if (p.beta != 0.0f) {
#pragma unroll
            for (int j = 0; j < 4 * NB; ++j) c[j] = load_chunk(cbase, cb + 4 * j, lim);
        }
#pragma unroll
        for (int j = 0; j < 4 * NB; ++j) {
            const float a[4] = {pick(x, 4 * j, s), pick(x, 4 * j + 1, s), pick(x, 4 * j + 2, s),
                                pick(x, 4 * j + 3, s)};
            store_chunk(p, cbase, cb + 4 * j, lim, a, c[j]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) x[i] = x[16 * NB + i];
    }
    if (row >= p.M) return;
    // last chunk: columns BN - 4 + s .. BN - 1 (x[s..3]); the rest of it is the next tile's
    float y[8] = {x[0], x[1], x[2], x[3], 0.0f, 0.0f, 0.0f, 0.0f};
    const int r0 = BN - 4 + s;
    const int lim_last = min(lim, BN);
    const float4 c = p.beta != 0.0f ? load_chunk(cbase, r0, lim_last) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    const float a[4] = {pick(y, 0, s), pick(y, 1, s), pick(y, 2, s), pick(y, 3, s)};
    store_chunk(p, cbase, r0, lim_last, a, c);
}

// C[row, tn*BN ...] = alpha * acc + beta * C (beta == 0: C not read).
template <int NB>
__device__ __forceinline__ void store_c_row(const Tf32Params &p, uint32_t t_row, int row, int tn)
{
    float *crow = p.C + static_cast<long long>(row) * p.ldc;
    if (!p.vec_c) {
        store_c_row_shifted<(NB > 2 ? 2 : NB)>(p, t_row, row, crow + tn * BN, min(BN, p.N - tn * BN));
        return;
    }
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
            // N edge: element by element, every C load of the step issued before any
            // use (one memory latency per step, not one per element)
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

template <bool PAIR>
__global__ void __launch_bounds__(THREADS, 1)
tf32_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const Tf32Params p)
{
    using S = Tf32Shape<PAIR>;
    constexpr int STAGES = S::STAGES;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    unsigned char *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t a_base = smem_addr(smem);
    const uint32_t b_base = a_base + STAGES * S::A_BYTES;
    Tf32Bars<STAGES> *bars = reinterpret_cast<Tf32Bars<STAGES> *>(smem + STAGES * S::STAGE_BYTES);
    volatile int *abort_flag = &bars->abort_flag;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (PAIR && cluster_size() != 2) {
        // not launched as clusters of two: no barrier, copy or tensor-core operation is issued
        if (threadIdx.x == 0) report_status(p.status, kLayoutCode | kWherePairLayout);
        return;
    }
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    const int worker = PAIR ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
    const int workers = PAIR ? static_cast<int>(cluster_count_x()) : static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_addr(&bars->full[s]), 1);
            mbar_init(smem_addr(&bars->empty[s]), 1);
            bars->issued[s] = 0;
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_addr(&bars->acc_full[b]), 1);
            mbar_init(smem_addr(&bars->acc_empty[b]), 4 * S::CTAS);
        }
        mbar_init(smem_addr(&bars->mma_done), 1);
        bars->abort_flag = 0;
        bars->ring_offset = a_base;
        fence_barrier_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if (warp == 0) {
        if constexpr (PAIR) {
            tmem_alloc_pair(smem_addr(&bars->tmem_base), TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_addr(&bars->tmem_base), TMEM_COLS);
            tmem_relinquish();
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();  // both CTAs' barriers are initialised before any copy or arrive targets them
    tc_fence_after_sync();
    const uint32_t tmem = bars->tmem_base;
    bool same_layout = true;
    if constexpr (PAIR) {
        // Rank 0's MMAs address both CTAs' stages by its own offsets, which must
        // therefore agree; compared on the address bits a shared-memory descriptor
        // holds (the offset inside the CTA; higher bits of a shared::cta address
        // differ between the CTAs of a cluster).
        constexpr uint32_t kDescAddrMask = 0x3FFFFu;
        const uint32_t peer_ring = ld_shared_cluster_u32(mapa_shared(smem_addr(&bars->ring_offset), rank ^ 1u));
        same_layout = ((peer_ring ^ a_base) & kDescAddrMask) == 0;
        if (!same_layout && threadIdx.x == 0) raise_abort(bars, p, kLayoutCode | kWherePairLayout);
    }

    if (!same_layout) {
        // both CTAs of the pair see the mismatch: no copies, no MMAs
    } else if (warp == 0 && lane == 0) {
        // ---- TMA producer: this CTA's part of each stage ----
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        pdl_wait();  // operands repacked by this call's previous kernel are complete
        Work w;
        for (int item = 0; ok && work_at_g(p, item, w, worker, workers); ++item) {
            const int row_a = w.tm * S::BM + static_cast<int>(rank) * S::CTA_M;
            const int col_b = w.tn * BN + static_cast<int>(rank) * S::CTA_N;
            for (int kb = w.kb0; kb < w.kb1; ++kb) {
                if (!mbar_wait_bounded(smem_addr(&bars->empty[stage]), phase ^ 1u, abort_flag, p.timeout_ns)) {
                    raise_abort(bars, p, kTimeoutCode | kWhereProducerEmpty);
                    ok = false;
                    break;
                }
                const uint32_t a_dst = a_base + stage * S::A_BYTES;
                const uint32_t b_dst = b_base + stage * S::B_BYTES;
                // a box outside the problem would only read fill values: recorded, not skipped
                index_ok(w.tm < p.tiles_m && w.tn < p.tiles_n && kb < p.kblocks, p.status, kWhereIdxTf32Copy);
                if (rank == 0) mbar_arrive_expect_tx(smem_addr(&bars->full[stage]), S::CTAS * S::STAGE_BYTES);
                if constexpr (PAIR) {
                    const uint32_t full = mapa_shared(smem_addr(&bars->full[stage]), 0);  // rank 0's barrier
                    tma_load_2d_pair(a_dst, &tmA, full, kb * BK, row_a);
#pragma unroll
                    for (int j = 0; j < S::CTA_N / kBoxN; ++j)
                        tma_load_2d_pair(b_dst + j * B_BOX_BYTES, &tmB, full, col_b + j * kBoxN, kb * BK);
                } else {
                    const uint32_t full = smem_addr(&bars->full[stage]);
                    tma_load_2d(a_dst, &tmA, full, kb * BK, row_a);
#pragma unroll
                    for (int j = 0; j < S::CTA_N / kBoxN; ++j)
                        tma_load_2d(b_dst + j * B_BOX_BYTES, &tmB, full, col_b + j * kBoxN, kb * BK);
                }
                bars->issued[stage] = 2 | static_cast<int>(phase);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        pdl_trigger();  // every copy is issued: the call's reduction may become resident
        // Drain. Rank 0: every issued stage's copies (of both CTAs of a pair) have
        // landed, as they complete on its full barriers. Every CTA: unless aborted,
        // the MMAs that read them have committed to this CTA's empty barriers.
        for (int s = 0; s < STAGES; ++s) {
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
        // ---- MMA issuer (rank 0) ----
        int stage = 0;
        uint32_t phase = 0;
        int it = 0;
        bool ok = true;
        Work w;
        for (int item = 0; ok && work_at_g(p, item, w, worker, workers); ++item, ++it) {
            const int buf = it & 1;
            const uint32_t acc_phase = static_cast<uint32_t>(it >> 1) & 1u;
            if (!mbar_wait_cluster_bounded(smem_addr(&bars->acc_empty[buf]), acc_phase ^ 1u, abort_flag,
                                           p.timeout_ns)) {
                raise_abort(bars, p, kTimeoutCode | kWhereAccum);
                break;
            }
            tc_fence_after_sync();
            const uint32_t d_tmem = tmem + static_cast<uint32_t>(buf * BN);
            const int kb0 = w.kb0, kb1 = w.kb1;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait_cluster_bounded(smem_addr(&bars->full[stage]), phase, abort_flag, p.timeout_ns)) {
                    raise_abort(bars, p, kTimeoutCode | kWhereMmaEmpty);
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t a_s = a_base + stage * S::A_BYTES;
                const uint32_t b_s = b_base + stage * S::B_BYTES;
#pragma unroll
                for (int k = 0; k < BK / MMA_K; ++k) {
                    // A: K advances 8 TF32 = 32 bytes inside the 128-byte swizzle atom;
                    // B: one 8-row (8 k) group = 1024 bytes.
                    const uint64_t a_desc = smem_desc_k_sw128(a_s + k * MMA_K * 4);
                    const uint64_t b_desc = smem_desc_mn_sw128_32b(b_s + k * 1024, B_BOX_BYTES);
                    const uint32_t acc = (kb != kb0 || k != 0) ? 1u : 0u;
                    if constexpr (PAIR)
                        mma_tf32_pair(d_tmem, a_desc, b_desc, S::IDESC, acc);
                    else
                        mma_tf32(d_tmem, a_desc, b_desc, S::IDESC, acc);
                }
                // the stage is free (in both CTAs of a pair) once these MMAs are done
                if constexpr (PAIR)
                    mma_commit_pair_both(smem_addr(&bars->empty[stage]));
                else
                    mma_commit(smem_addr(&bars->empty[stage]));
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            if constexpr (PAIR)
                mma_commit_pair_both(smem_addr(&bars->acc_full[buf]));
            else
                mma_commit(smem_addr(&bars->acc_full[buf]));
        }
        // Every MMA (for a pair they write both CTAs' TMEM) is finished before TMEM is freed.
        if constexpr (PAIR)
            mma_commit_pair_local(smem_addr(&bars->mma_done));
        else
            mma_commit(smem_addr(&bars->mma_done));
        if (!mbar_wait_bounded(smem_addr(&bars->mma_done), 0u, nullptr, p.timeout_ns))
            report_status(p.status, kTimeoutCode | kWhereDrain);
    } else if (warp >= 2) {
        // ---- epilogue: warp w reads TMEM lanes 32 * (w % 4) .. + 31 of this CTA ----
        const int quarter = warp & 3;
        const int cta_row = static_cast<int>(rank) * S::CTA_M + quarter * 32 + lane;  // row within the tile
        int it = 0;
        Work w;
        for (int item = 0; work_at_g(p, item, w, worker, workers); ++item, ++it) {
            const int buf = it & 1;
            const uint32_t acc_phase = static_cast<uint32_t>(it >> 1) & 1u;
            bool ok = mbar_wait_cluster_bounded(smem_addr(&bars->acc_full[buf]), acc_phase, abort_flag, p.timeout_ns);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                if (lane == 0) raise_abort(bars, p, kTimeoutCode | kWhereAccum);
                break;
            }
            tc_fence_after_sync();
            const uint32_t t_row = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(buf * BN);
            if (w.dest == kToPartial) {
                // Stream-K piece: this CTA's rows of the raw, tile-packed partial tile
                // (rows and columns past M and N hold sums of the copy engine's zero
                // fill); the stream-K reduction adds the pieces in k order and
                // applies alpha / beta.
                float *wrow = p.W + static_cast<long long>(w.idx) * (S::BM * BN) + static_cast<long long>(cta_row) * BN;
                const bool wok = index_ok(w.idx >= 0 && static_cast<long long>(w.idx) * (S::BM * BN) +
                                                            static_cast<long long>(cta_row + 1) * BN <= p.w_elems,
                                          p.status, kWhereIdxTf32Store);
                if (p.kblocks <= kShortK)
                    store_partial_row<4>(t_row, wrow, wok);
                else
                    store_partial_row<1>(t_row, wrow, wok);
            } else {
                const int row = w.tm * S::BM + cta_row;
                if (p.kblocks <= kShortK)
                    store_c_row<4>(p, t_row, row, w.tn);
                else
                    store_c_row<1>(p, t_row, row, w.tn);
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                if constexpr (PAIR)
                    mbar_arrive_cluster(mapa_shared(smem_addr(&bars->acc_empty[buf]), 0));  // rank 0's
                else
                    mbar_arrive(smem_addr(&bars->acc_empty[buf]));
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();  // neither CTA leaves while the other may still use its barriers, stages or TMEM
    tc_fence_after_sync();
    if (warp == 0) {
        __syncwarp();
        if constexpr (PAIR)
            tmem_dealloc_pair(tmem, TMEM_COLS);
        else
            tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace

cudaError_t tf32_set_attributes()
{
    cudaError_t e = cudaFuncSetAttribute(tf32_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Tf32Shape<false>::SMEM);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(tf32_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Tf32Shape<true>::SMEM);
}

int tf32_pair_max_pairs()
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = Tf32Shape<true>::SMEM;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, tf32_kernel<true>, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return clusters;
}

cudaError_t launch_tf32(const CUtensorMap &tmA, const CUtensorMap &tmB, const Tf32Params &p, int grid,
                        cudaStream_t stream, bool dependent)
{
    return launch_kernel(dependent, tf32_kernel<false>, dim3(grid), dim3(THREADS), Tf32Shape<false>::SMEM, stream,
                         tmA, tmB, p);
}

cudaError_t launch_tf32_pair(const CUtensorMap &tmA, const CUtensorMap &tmB, const Tf32Params &p, int grid,
                             cudaStream_t stream, bool dependent)
{
    // grid = 2 x pairs, launched as clusters of two
    return launch_kernel_cluster(dependent, 2, tf32_kernel<true>, dim3(grid), dim3(THREADS), Tf32Shape<true>::SMEM,
                                 stream, tmA, tmB, p);
}

}  // namespace sgemm_impl
