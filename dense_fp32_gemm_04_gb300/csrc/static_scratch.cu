// Split-K SGEMM whose scratch lives in a file-scope static device array, so a
// call performs no device allocation at all.
//
// Who needs this: code that runs inside another runtime's memory pool and may
// not grow device memory behind its back, and latency-sensitive loops that
// cannot afford the implicit device-wide synchronization of cudaMalloc /
// cudaFree. sgemm_run keeps its split-K partials in a handle-owned workspace
// that grows with cudaMalloc (and creating a handle allocates its status
// word); sgemm_run_splitk_static needs no handle and uses the static array
// below instead.
//
// Limits and sharing rules (also stated in include/sgemm.h):
//  * kStaticScratchBytes (32 MiB) holds the split partials and, for operands
//    that are not 16-byte aligned, their aligned copies. Larger problems are
//    rejected with SGEMM_ERR_NOT_SUPPORTED before anything is launched.
//  * Every GPU that loads this library holds the array until process exit.
//  * All calls on a device share the array, which keeps the last call's
//    contents; calls that overlap on the GPU (different streams, no ordering
//    between them) race on it and must be avoided by the caller. The same holds
//    for the internal watchdog word used when the caller passes no status word.
//  * The first call on a device does a one-time set-up with that device
//    current (symbol address lookup, kernel attributes); make that first call
//    before any stream capture.
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/sgemm.h"
#include "planner.h"
#include "sgemm_internal.h"

namespace {

using sgemm_impl::FfmaParams;
using sgemm_impl::Overrides;
using sgemm_impl::Problem;
using sgemm_impl::Workspace;

constexpr size_t kStaticScratchBytes = SGEMM_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;
constexpr long long kTimeoutNs = 4000000000LL;

// Partials (and aligned operand copies) of sgemm_run_splitk_static.
static __device__ __align__(256) unsigned char g_scratch[kStaticScratchBytes];
// Watchdog word used when the caller passes no status pointer. Nothing reads it
// back: with a NULL status pointer a timeout code is dropped (calls that overlap
// on the GPU race on it like they race on g_scratch).
static __device__ __align__(256) int g_status[64];

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceState {
    bool ready = false;
    unsigned char *scratch = nullptr;  // device address of g_scratch on this device
    int *status = nullptr;             // device address of g_status on this device
    int num_sms = 0;
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];
EncodeTiledFn g_encode = nullptr;

// One-time set-up for device `dev`, which must be current. The host-side names
// g_scratch / g_status are stand-ins, not device addresses: the addresses come
// from cudaGetSymbolAddress on the current device.
int setup_device(int dev, DeviceState **out)
{
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState &s = g_devices[dev];
    if (!s.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return SGEMM_ERR_ARCH;
        }
        if (major != 10 || minor != 3) return SGEMM_ERR_ARCH;
        void *scratch = nullptr, *status = nullptr;
        if (cudaGetSymbolAddress(&scratch, g_scratch) != cudaSuccess ||
            cudaGetSymbolAddress(&status, g_status) != cudaSuccess) {
            cudaGetLastError();
            return SGEMM_ERR_CUDA;
        }
        if (g_encode == nullptr) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult qr;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qr) !=
                    cudaSuccess ||
                qr != cudaDriverEntryPointSuccess || fn == nullptr) {
                cudaGetLastError();
                return SGEMM_ERR_CUDA;
            }
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
        if (sgemm_impl::ffma_set_attributes() != cudaSuccess) {
            cudaGetLastError();
            return SGEMM_ERR_CUDA;
        }
        s.scratch = static_cast<unsigned char *>(scratch);
        s.status = static_cast<int *>(status);
        s.num_sms = sms;
        s.ready = true;
    }
    *out = &s;
    return SGEMM_OK;
}

int encode_2d(CUtensorMap *map, const float *base, int inner, int outer, long long ld, int box_inner, int box_outer,
              CUtensorMapSwizzle swz)
{
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 4u};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_outer)};
    cuuint32_t estr[2] = {1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
               ? SGEMM_OK
               : SGEMM_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int sgemm_run_splitk_static(int M, int N, int K, float alpha, const float *A, int lda, const float *B,
                                       int ldb, float beta, float *C, int ldc, int splits, int *device_status,
                                       struct CUstream_st *stream)
{
    if (splits < 1 || splits > sgemm_impl::kMaxSplits) return SGEMM_ERR_INVALID_VALUE;
    if (!sgemm_impl::elem_aligned(A) || !sgemm_impl::elem_aligned(B) || !sgemm_impl::elem_aligned(C) ||
        !sgemm_impl::elem_aligned(device_status))
        return SGEMM_ERR_INVALID_VALUE;
    const int align = (aligned16(A) ? 1 : 0) | (aligned16(B) ? 2 : 0) | (aligned16(C) ? 4 : 0);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return SGEMM_ERR_CUDA;
    }
    Problem q{M, N, K, lda, ldb, ldc, align, 1, SGEMM_MATH_FP32, alpha, beta};
    if (sgemm_impl::validate(q) != SGEMM_OK) return SGEMM_ERR_INVALID_VALUE;
    if (M > 0 && N > 0) {
        if (C == nullptr) return SGEMM_ERR_INVALID_VALUE;
        if (K > 0 && alpha != 0.0f && (A == nullptr || B == nullptr)) return SGEMM_ERR_INVALID_VALUE;
    }
    DeviceState *s = nullptr;
    int rc = setup_device(dev, &s);
    if (rc != SGEMM_OK) return rc;
    q.num_sms = s->num_sms;

    Overrides ov;
    ov.force_splits = splits;
    ov.force_transpose_a = 2;  // A transposed in shared memory: the scratch array holds split-K partials only
    ov.force_streamk = 0;
    ov.cluster_split = 0;  // partials in the static array, reduced by the reduction kernel
    sgemm_plan_t plan;
    if ((rc = sgemm_impl::make_plan(q, ov, &plan)) != SGEMM_OK) return rc;
    cudaStream_t st = stream;
    const Workspace w = sgemm_impl::workspace_layout(q, plan);
    const bool gemm = plan.kernel != SGEMM_KERNEL_NONE && plan.kernel != SGEMM_KERNEL_SCALE;
    if (gemm && static_cast<unsigned long long>(w.total) > kStaticScratchBytes) return SGEMM_ERR_NOT_SUPPORTED;

    // The watchdog word starts at zero for every call that succeeds, also for the
    // quick returns, so a caller that reuses its word never reads an old code.
    int *status = device_status ? device_status : s->status;
    if ((gemm || device_status) && cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) {
        cudaGetLastError();
        return SGEMM_ERR_CUDA;
    }
    if (plan.kernel == SGEMM_KERNEL_NONE) return SGEMM_OK;
    if (plan.kernel == SGEMM_KERNEL_SCALE)
        return sgemm_impl::launch_scale(M, N, beta, C, ldc, s->num_sms, st) == cudaSuccess ? SGEMM_OK
                                                                                            : SGEMM_ERR_LAUNCH;

    unsigned char *ws = s->scratch;
    const float *a_src = A;
    long long a_ld = lda;
    const float *b_src = B;
    long long b_ld = ldb;
    if (plan.repack_a) {
        float *dst = reinterpret_cast<float *>(ws + w.a_off);
        if (sgemm_impl::launch_repack(A, lda, dst, w.lda, M, K, s->num_sms, st) != cudaSuccess)
            return SGEMM_ERR_LAUNCH;
        a_src = dst;
        a_ld = w.lda;
    }
    if (plan.repack_b) {
        float *dst = reinterpret_cast<float *>(ws + w.b_off);
        if (sgemm_impl::launch_repack(B, ldb, dst, w.ldb, K, N, s->num_sms, st) != cudaSuccess)
            return SGEMM_ERR_LAUNCH;
        b_src = dst;
        b_ld = w.ldb;
    }
    CUtensorMap tmA, tmB;
    if ((rc = encode_2d(&tmA, a_src, K, M, a_ld, sgemm_cfg::kFfmaBK, plan.bm, CU_TENSOR_MAP_SWIZZLE_128B)) != SGEMM_OK)
        return rc;
    if ((rc = encode_2d(&tmB, b_src, N, K, b_ld, plan.bn, sgemm_cfg::kFfmaBK, CU_TENSOR_MAP_SWIZZLE_NONE)) != SGEMM_OK)
        return rc;

    FfmaParams p{};
    p.M = M;
    p.N = N;
    p.K = K;
    p.alpha = alpha;
    p.beta = beta;
    p.C = C;
    p.ldc = ldc;
    p.W = plan.splits > 1 ? reinterpret_cast<float *>(ws + w.w_off) : nullptr;
    p.ldw = w.ldw;
    p.wstride = w.wstride;
    p.splits = plan.splits;
    p.tiles_m = plan.tiles_m;
    p.tiles_n = plan.tiles_n;
    p.units = plan.units;
    p.kblocks = (K + sgemm_cfg::kFfmaBK - 1) / sgemm_cfg::kFfmaBK;
    p.vec_c = plan.vec_c;
    p.status = status;
    p.timeout_ns = kTimeoutNs;
    p.inject_skip = -1;
    p.w_elems = p.W != nullptr ? (w.total - w.w_off) / 4 : 0;
    if (sgemm_impl::launch_ffma(plan.config, plan.transpose_a, tmA, tmB, p, plan.grid, st, false) != cudaSuccess)
        return SGEMM_ERR_LAUNCH;
    if (plan.splits > 1 &&
        sgemm_impl::launch_splitk_reduce(p.W, w.ldw, w.wstride, plan.splits, M, N, alpha, beta, C, ldc, plan.vec_c,
                                         s->num_sms, st, p.w_elems, status) != cudaSuccess)
        return SGEMM_ERR_LAUNCH;
    return SGEMM_OK;
}
