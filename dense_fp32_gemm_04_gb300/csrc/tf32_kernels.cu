// Flagged TF32 mode (SGEMM_MATH_TF32): C = alpha * A * B + beta * C on the
// 5th-generation tensor cores. A and B are read as TF32 (10 explicit mantissa
// bits), products are accumulated in FP32 in tensor memory (TMEM). It is never
// used unless the caller selects it, and is held to its own, looser bound.
//
// Structure (one CTA per SM, persistent over 128 x 256 output tiles):
//   warp 0      TMA producer: A box (32 k x 128 rows) and B^T box (32 k x 256
//               columns), both with the 128-byte swizzle, into a 4-stage ring.
//   warp 1      MMA issuer: one thread issues 4 tcgen05.mma (K = 8 each) per
//               stage into one of two TMEM accumulators (128 lanes x 256
//               columns each), commits the stage back to the producer, and
//               commits a finished accumulator to the epilogue.
//   warps 2..5  epilogue: tcgen05.ld of their 32-lane quarter of the
//               accumulator, alpha/beta, stores to C; then hand the
//               accumulator back so the next tile's MMAs overlap this one's
//               stores.
// Both operands must be K-major for this instruction form: A (row-major M x K)
// already is; B (row-major K x N) is first transposed into the handle's
// workspace (transpose_kernel, ffma_kernels.cu).
//
// All waits are bounded; on expiry the CTA records SGEMM_ERR_TIMEOUT, lets its
// copies and MMAs in flight finish (bounded), frees its TMEM and returns.
#include <cuda_runtime.h>

#include <cstdint>

#include "device_ptx.cuh"
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
constexpr uint32_t IDESC = idesc_tf32(BM, BN);
constexpr int kGroupM = 8;
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

__device__ __forceinline__ void decode_tile(const Tf32Params &p, int u, int &tm, int &tn)
{
    const int per_group = kGroupM * p.tiles_n;
    const int g = u / per_group;
    const int first_m = g * kGroupM;
    const int gsize = min(p.tiles_m - first_m, kGroupM);
    const int r = u - g * per_group;
    tm = first_m + r % gsize;
    tn = r / gsize;
}

// Work unit u -> tile t (grouped raster), K-block range [kb0, kb1), slice ks
// of ns (ns == 1: the whole tile).
__device__ __forceinline__ void decode_unit(const Tf32Params &p, int u, int &t, int &tm, int &tn, int &ks, int &ns,
                                            int &kb0, int &kb1)
{
    if (p.tail_splits > 1 && u >= p.n_full) {
        const int v = u - p.n_full;
        t = p.n_full + v / p.tail_splits;
        ks = v % p.tail_splits;
        ns = p.tail_splits;
    } else {
        t = u;
        ks = 0;
        ns = 1;
    }
    decode_tile(p, t, tm, tn);
    kb0 = static_cast<int>((static_cast<long long>(ks) * p.kblocks) / ns);
    kb1 = static_cast<int>((static_cast<long long>(ks + 1) * p.kblocks) / ns);
}

__device__ __forceinline__ void raise_abort(Bars *b, const Tf32Params &p, int where)
{
    volatile int *f = &b->abort_flag;
    if (!*f) {
        *f = 1;
        report_status(p.status, kTimeoutCode | where);
    }
}

__global__ void __launch_bounds__(THREADS, 1)
tf32_sgemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmBt,
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
        prefetch_tensormap(&tmBt);
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
        for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
            int t, tm, tn, ks, ns, kb0, kb1;
            decode_unit(p, u, t, tm, tn, ks, ns, kb0, kb1);
            for (int kb = kb0; kb < kb1; ++kb) {
                const uint32_t full = smem_addr(&bars->full[stage]);
                if (!mbar_wait_bounded(smem_addr(&bars->empty[stage]), phase ^ 1u, abort_flag, p.timeout_ns)) {
                    raise_abort(bars, p, kWhereProducerEmpty);
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(full, STAGE_BYTES);
                tma_load_2d(a_base + stage * A_BYTES, &tmA, full, kb * BK, tm * BM);
                tma_load_2d(b_base + stage * B_BYTES, &tmBt, full, kb * BK, tn * BN);
                bars->issued[stage] = 2 | static_cast<int>(phase);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
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
        for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x, ++it) {
            const int buf = it & 1;
            const uint32_t acc_phase = static_cast<uint32_t>(it >> 1) & 1u;
            if (!mbar_wait_bounded(smem_addr(&bars->acc_empty[buf]), acc_phase ^ 1u, abort_flag, p.timeout_ns)) {
                raise_abort(bars, p, kWhereAccum);
                break;
            }
            tc_fence_after_sync();
            const uint32_t d_tmem = tmem + static_cast<uint32_t>(buf * BN);
            int t, tm, tn, ks, ns, kb0, kb1;
            decode_unit(p, u, t, tm, tn, ks, ns, kb0, kb1);
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
                    // K advances 8 TF32 = 32 bytes inside the 128-byte swizzle atom.
                    mma_tf32(d_tmem, smem_desc_k_sw128(a_s + k * MMA_K * 4), smem_desc_k_sw128(b_s + k * MMA_K * 4),
                             IDESC, (kb != kb0 || k != 0) ? 1u : 0u);
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
        for (int u = blockIdx.x; u < p.units; u += gridDim.x, ++it) {
            const int buf = it & 1;
            const uint32_t acc_phase = static_cast<uint32_t>(it >> 1) & 1u;
            bool ok = mbar_wait_bounded(smem_addr(&bars->acc_full[buf]), acc_phase, abort_flag, p.timeout_ns);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                if (lane == 0) raise_abort(bars, p, kWhereAccum);
                break;
            }
            tc_fence_after_sync();
            int t, tm, tn, ks, ns, kb0, kb1;
            decode_unit(p, u, t, tm, tn, ks, ns, kb0, kb1);
            const int row = tm * BM + quarter * 32 + lane;
            const uint32_t t_row = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(buf * BN);
            if (ns > 1) {
                // Tail slice: the raw partial tile, tile-packed (rows and columns past
                // M and N hold sums of the copy engine's zero fill); the tail
                // reduction adds the slices in order and applies alpha / beta.
                float *wrow = p.W + (static_cast<long long>(t - p.n_full) * p.tail_splits + ks) * (BM * BN) +
                              (quarter * 32 + lane) * BN;
#pragma unroll 1
                for (int ch = 0; ch < BN / 16; ++ch) {
                    uint32_t v[16];
                    tmem_ld_16(t_row + ch * 16, v);
                    tmem_wait_ld(v);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        *reinterpret_cast<float4 *>(wrow + ch * 16 + 4 * q) =
                            make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                        __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&bars->acc_empty[buf]));
                continue;
            }
            float *crow = p.C + static_cast<long long>(row) * p.ldc;
#pragma unroll 1
            for (int ch = 0; ch < BN / 16; ++ch) {
                uint32_t v[16];
                tmem_ld_16(t_row + ch * 16, v);
                tmem_wait_ld(v);
                const int col0 = tn * BN + ch * 16;
                if (row < p.M) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int col = col0 + 4 * q;
                        const float4 acc = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                                       __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
                        float *dst = crow + col;
                        if (p.vec_c && col + 3 < p.N) {
                            float4 out;
                            if (p.beta != 0.0f) {
                                const float4 c = *reinterpret_cast<const float4 *>(dst);
                                out = make_float4(fmaf(p.alpha, acc.x, p.beta * c.x), fmaf(p.alpha, acc.y, p.beta * c.y),
                                                  fmaf(p.alpha, acc.z, p.beta * c.z), fmaf(p.alpha, acc.w, p.beta * c.w));
                            } else {
                                out = make_float4(p.alpha * acc.x, p.alpha * acc.y, p.alpha * acc.z, p.alpha * acc.w);
                            }
                            *reinterpret_cast<float4 *>(dst) = out;
                        } else {
                            const float e[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
                            for (int t = 0; t < 4; ++t)
                                if (col + t < p.N)
                                    dst[t] = (p.beta != 0.0f) ? fmaf(p.alpha, e[t], p.beta * dst[t]) : p.alpha * e[t];
                        }
                    }
                }
            }
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

}  // namespace

cudaError_t tf32_set_attributes()
{
    return cudaFuncSetAttribute(tf32_sgemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                sgemm_cfg::tf32_smem_bytes());
}

cudaError_t launch_tf32(const CUtensorMap &tmA, const CUtensorMap &tmBt, const Tf32Params &p, int grid,
                        cudaStream_t stream)
{
    tf32_sgemm_kernel<<<grid, THREADS, sgemm_cfg::tf32_smem_bytes(), stream>>>(tmA, tmBt, p);
    return cudaGetLastError();
}

}  // namespace sgemm_impl
