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
    static_assert(SMEM == 1024 + STAGES * STAGE_BYTES + 256 + sgemm_cfg::kTf32StagingBytes, "smem layout");
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

// Epilogue. A warp holds 32 rows of a CTA's accumulator (its TMEM lane
// quarter); tcgen05.ld hands thread l the columns of row l, so stores made
// straight from those registers touch 32 rows, 16 bytes each, per instruction.
// Instead each 32-column block goes through the warp's staging area in shared
// memory and leaves it coalesced:
//  - 16-byte rows (the partial tiles in W, or C with vec_c): lane l takes
//    16-byte chunk l % 8 of rows 4k + l / 8 (k = 0..7), so 8 lanes cover one
//    row's 128 bytes;
//  - other C: lane l takes column l of each of the 32 rows (4-byte accesses,
//    128 contiguous bytes per instruction, whatever the row's alignment).
// With beta != 0 the next block's C loads are issued before the current block
// is turned and written, so two blocks' loads are in flight.
constexpr int kStgPitch = 36;  // floats between staged rows (see stage_block)
static_assert(sgemm_cfg::kTf32StagingBytes == 4 * 32 * kStgPitch * 4, "four epilogue warps' staging areas");

__device__ __forceinline__ float4 lds128(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ float lds32(uint32_t addr)
{
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t x, uint32_t y, uint32_t z, uint32_t w)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}

// Thread l: TMEM row l, columns [t_col, t_col + 32) into staged row l. With a
// pitch of 36 floats the 8 rows of a quarter-warp's 16-byte stores, and the 8
// chunks of one row that a quarter-warp reads back, fall in 8 different 16-byte
// bank groups.
__device__ __forceinline__ void stage_block(uint32_t t_col, uint32_t stg, int lane)
{
    uint32_t v[2][16];
    tmem_ld_16(t_col, v[0]);  // every lane: .sync.aligned
    tmem_ld_16(t_col + 16, v[1]);
    tmem_wait_ld(v[0]);
    tmem_wait_ld(v[1]);
    const uint32_t row = stg + static_cast<uint32_t>(lane * kStgPitch * 4);
#pragma unroll
    for (int i = 0; i < 8; ++i)
        sts128(row + 16 * i, v[i >> 2][4 * (i & 3)], v[i >> 2][4 * (i & 3) + 1], v[i >> 2][4 * (i & 3) + 2],
               v[i >> 2][4 * (i & 3) + 3]);
    __syncwarp();
}

__device__ __forceinline__ float epi_value(const Tf32Params &p, float acc, float c)
{
    return p.beta != 0.0f ? fmaf(p.alpha, acc, p.beta * c) : p.alpha * acc;
}

// C of block cb for this lane (0 outside the problem): 16-byte form, rows
// 4k + sub, chunk q; or 4-byte form, column `lane` of rows 0..31.
__device__ __forceinline__ void load_c_block(const Tf32Params &p, int grow0, int col0, int cb, int lane,
                                             float (&c)[32])
{
    if (p.vec_c) {
        const int sub = lane >> 3, col = col0 + cb * 32 + 4 * (lane & 7);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int grow = grow0 + 4 * k + sub;
            if (grow < p.M && col + 3 < p.N) {
                const float4 x = *reinterpret_cast<const float4 *>(p.C + static_cast<long long>(grow) * p.ldc + col);
                c[4 * k] = x.x;
                c[4 * k + 1] = x.y;
                c[4 * k + 2] = x.z;
                c[4 * k + 3] = x.w;
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    c[4 * k + e] = (grow < p.M && col + e < p.N) ? p.C[static_cast<long long>(grow) * p.ldc + col + e]
                                                                 : 0.0f;
            }
        }
    } else {
        const int col = col0 + cb * 32 + lane;
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            const int grow = grow0 + r;
            c[r] = (grow < p.M && col < p.N) ? p.C[static_cast<long long>(grow) * p.ldc + col] : 0.0f;
        }
    }
}

// One finished tile, this warp's 32 rows (tile rows row0 .. row0 + 31; TMEM
// lanes of t_row): to C with alpha / beta, or raw into the tile's partial tile
// in W (tile-packed rows of BN floats; rows and columns past M and N hold sums
// of the copy engine's zero fill, and the stream-K reduction adds the pieces in
// k order). `stg`: the warp's staging area.
template <class S>
__device__ __forceinline__ void write_tile(const Tf32Params &p, uint32_t t_row, uint32_t stg, const Work &w, int row0,
                                           int lane)
{
    const int sub = lane >> 3, q = lane & 7;
    if (w.dest == kToPartial) {
        float *wb = p.W + static_cast<long long>(w.idx) * (S::BM * BN) + static_cast<long long>(row0) * BN;
        const bool ok = index_ok(w.idx >= 0 && static_cast<long long>(w.idx) * (S::BM * BN) +
                                                   static_cast<long long>(row0 + 32) * BN <= p.w_elems,
                                 p.status, kWhereIdxTf32Store);
#pragma unroll 1
        for (int cb = 0; cb < BN / 32; ++cb) {
            stage_block(t_row + cb * 32, stg, lane);
            if (ok) {
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int r = 4 * k + sub;
                    *reinterpret_cast<float4 *>(wb + static_cast<long long>(r) * BN + cb * 32 + 4 * q) =
                        lds128(stg + static_cast<uint32_t>((r * kStgPitch + 4 * q) * 4));
                }
            }
            __syncwarp();
        }
        return;
    }
    const int grow0 = w.tm * S::BM + row0, col0 = w.tn * BN;
    const bool use_c = p.beta != 0.0f;
    float cn[32];
    if (use_c) load_c_block(p, grow0, col0, 0, lane, cn);
#pragma unroll 1
    for (int cb = 0; cb < BN / 32; ++cb) {
        float cc[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) cc[i] = use_c ? cn[i] : 0.0f;
        if (use_c && cb + 1 < BN / 32) load_c_block(p, grow0, col0, cb + 1, lane, cn);
        stage_block(t_row + cb * 32, stg, lane);
        if (p.vec_c) {
            const int col = col0 + cb * 32 + 4 * q;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int grow = grow0 + 4 * k + sub;
                const float4 a = lds128(stg + static_cast<uint32_t>(((4 * k + sub) * kStgPitch + 4 * q) * 4));
                const float4 out = make_float4(epi_value(p, a.x, cc[4 * k]), epi_value(p, a.y, cc[4 * k + 1]),
                                               epi_value(p, a.z, cc[4 * k + 2]), epi_value(p, a.w, cc[4 * k + 3]));
                float *dst = p.C + static_cast<long long>(grow) * p.ldc + col;
                if (grow < p.M && col + 3 < p.N) {
                    *reinterpret_cast<float4 *>(dst) = out;
                } else if (grow < p.M) {
                    const float e[4] = {out.x, out.y, out.z, out.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (col + j < p.N) dst[j] = e[j];
                }
            }
        } else {
            const int col = col0 + cb * 32 + lane;
#pragma unroll
            for (int r = 0; r < 32; ++r) {
                const int grow = grow0 + r;
                const float a = lds32(stg + static_cast<uint32_t>((r * kStgPitch + lane) * 4));
                if (grow < p.M && col < p.N) p.C[static_cast<long long>(grow) * p.ldc + col] = epi_value(p, a, cc[r]);
            }
        }
        __syncwarp();
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
    const uint32_t stg_base = a_base + STAGES * S::STAGE_BYTES + 256;  // after the barrier block
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
        const uint32_t stg = stg_base + static_cast<uint32_t>(quarter * 32 * kStgPitch * 4);  // this warp's staging area
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
            write_tile<S>(p, t_row, stg, w, static_cast<int>(rank) * S::CTA_M + quarter * 32, lane);
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
