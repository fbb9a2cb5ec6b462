// C ABI of the GB300 SGEMM library: handle lifetime, argument checks, plan
// execution (repack -> mainloop -> split-K reduce), host-buffer entry point
// and status reporting. Declarations and contracts: include/sgemm.h.
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <new>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/sgemm.h"
#include "../../include/sgemm_ladder.h"
#include "planner.h"
#include "sgemm_internal.h"

using namespace sgemm_impl;

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct sgemm_handle_s {
    int device = 0;
    int num_sms = 0;
    int tf32_pairs = -1;  // CTA pairs of the TF32 pair kernel resident at once (-1: none fit)
    int math_mode = SGEMM_MATH_FP32;
    int *d_status = nullptr;
    void *workspace = nullptr;
    size_t ws_bytes = 0;
    float *stage = nullptr;  // sgemm_run_host device copies of A | B | C
    size_t stage_bytes = 0;
    Overrides ov;
    int inject_skip = -1;
    int skew_ns = 0;
    int log = 0;
    long long timeout_ns = 4000000000LL;
    sgemm_plan_t last{};
    EncodeTiledFn encode = nullptr;
    // sgemm_run_host pipeline: copy-in and copy-out streams and their events.
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t ev_start = nullptr, ev_end = nullptr;
    cudaEvent_t ev_in[12] = {}, ev_done[12] = {};  // one pair per pipeline step
    void *min2_cand = nullptr;  // sgemm_run_min2 per-block candidates
};

namespace {

constexpr int kMaxHostPanels = 8;
constexpr int kMaxColBlocks = 4;
constexpr int kMaxHostSteps = kMaxHostPanels - 1 + kMaxColBlocks;
static_assert(kMaxHostSteps <= 12, "events per pipeline step");

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Bind the handle's device for the duration of a call.
struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) != cudaSuccess) {
            ok = false;
            return;
        }
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
    }
    ~DeviceGuard()
    {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

// Grow the handle's workspace to at least `bytes`. Growing synchronizes the
// device and reallocates, which a stream capture forbids: while `stream` is being
// captured, a workspace that is too small is SGEMM_ERR_NOT_SUPPORTED and nothing
// is called (size it first, with sgemm_reserve or an uncaptured call).
int ensure_workspace(sgemm_handle_t h, size_t bytes, cudaStream_t stream)
{
    if (bytes <= h->ws_bytes) return SGEMM_OK;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
        cudaGetLastError();
        return SGEMM_ERR_CUDA;
    }
    if (cap != cudaStreamCaptureStatusNone) return SGEMM_ERR_NOT_SUPPORTED;
    if (h->workspace) {
        // Earlier launches on any stream may still read the old buffer.
        if (cudaDeviceSynchronize() != cudaSuccess) return SGEMM_ERR_CUDA;
        cudaFree(h->workspace);
        h->workspace = nullptr;
        h->ws_bytes = 0;
    }
    // 25 % headroom so that slowly growing problems do not reallocate every call;
    // exactly `bytes` when the headroom does not fit.
    for (size_t size : {bytes + bytes / 4, bytes}) {
        if (cudaMalloc(&h->workspace, size) == cudaSuccess) {
            h->ws_bytes = size;
            return SGEMM_OK;
        }
        cudaGetLastError();
        h->workspace = nullptr;
    }
    return SGEMM_ERR_ALLOC;
}

// 2-D FP32 tensor map over a row-major (outer x inner) matrix with row stride ld.
int make_tmap(sgemm_handle_t h, CUtensorMap *map, const float *base, int inner, int outer, long long ld,
              int box_inner, int box_outer, CUtensorMapSwizzle swz)
{
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 4u};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_outer)};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = h->encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides,
                                 box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? SGEMM_OK : SGEMM_ERR_CUDA;
}

int check_args(sgemm_handle_t h, int M, int N, int K, float alpha, const float *A, int lda, const float *B, int ldb,
               float *C, int ldc)
{
    if (h == nullptr) return SGEMM_ERR_INVALID_VALUE;
    if (!elem_aligned(A) || !elem_aligned(B) || !elem_aligned(C)) return SGEMM_ERR_INVALID_VALUE;
    Problem q{M, N, K, lda, ldb, ldc, 0, 1, SGEMM_MATH_FP32, alpha, 0.0f};
    const int v = validate(q);
    if (v != SGEMM_OK) return v;
    if (M > 0 && N > 0) {
        if (C == nullptr) return SGEMM_ERR_INVALID_VALUE;
        if (K > 0 && alpha != 0.0f && (A == nullptr || B == nullptr)) return SGEMM_ERR_INVALID_VALUE;
    }
    return SGEMM_OK;
}

void log_plan(const sgemm_plan_t &p, int M, int N, int K)
{
    std::fprintf(stderr,
                 "[sgemm] M=%d N=%d K=%d kernel=%d config=%d tile=%dx%dx%d stages=%d splits=%d units=%d grid=%d "
                 "repack=(%d,%d) transpose_a=%d vec_c=%d mode=%d launches=%d ws=%lld sk_tiles=%d cluster_split=%d\n",
                 M, N, K, p.kernel, p.config, p.bm, p.bn, p.bk, p.stages, p.splits, p.units, p.grid, p.repack_a,
                 p.repack_b, p.transpose_a, p.vec_c, p.math_mode, p.launches, p.workspace_bytes, p.sk_tiles,
                 p.cluster_split);
}

// TF32 tensor-core path: [repack A] [repack B] [copy C in] -> tcgen05 mainloop (one
// CTA per 128 x 256 tile, or a CTA pair per 256 x 256 tile) [-> stream-K reduction]
// [-> copy C back].
int run_tf32(sgemm_handle_t h, const sgemm_plan_t &plan, const Workspace &w, int M, int N, int K, float alpha,
             const float *A, int lda, const float *B, int ldb, float beta, float *C, int ldc, cudaStream_t stream)
{
    char *ws = static_cast<char *>(h->workspace);
    const float *a_src = A, *b_src = B;
    long long a_ld = lda, b_ld = ldb;
    if (plan.repack_a && plan.repack_b) {  // both copies in one launch
        float *a_dst = reinterpret_cast<float *>(ws + w.a_off);
        float *b_dst = reinterpret_cast<float *>(ws + w.b_off);
        if (launch_prep(A, lda, a_dst, w.lda, M, K, false, B, ldb, b_dst, w.ldb, K, N, h->num_sms, stream) !=
            cudaSuccess)
            return SGEMM_ERR_LAUNCH;
        a_src = a_dst;
        a_ld = w.lda;
        b_src = b_dst;
        b_ld = w.ldb;
    } else if (plan.repack_a) {
        float *dst = reinterpret_cast<float *>(ws + w.a_off);
        if (launch_repack(A, lda, dst, w.lda, M, K, h->num_sms, stream) != cudaSuccess) return SGEMM_ERR_LAUNCH;
        a_src = dst;
        a_ld = w.lda;
    } else if (plan.repack_b) {
        float *dst = reinterpret_cast<float *>(ws + w.b_off);
        if (launch_repack(B, ldb, dst, w.ldb, K, N, h->num_sms, stream) != cudaSuccess) return SGEMM_ERR_LAUNCH;
        b_src = dst;
        b_ld = w.ldb;
    }
    CUtensorMap tmA, tmB;
    int rc;
    // A box: a CTA's rows of the tile (the pair kernel's CTAs stage 128 rows each);
    // B box: 32 columns x 32 k, read MN-major with the 128-byte swizzle of 32-byte
    // chunks (the kernels issue one per 32 columns).
    const bool pair = plan.config == 1;
    const int box_a = pair ? plan.bm / 2 : plan.bm;
    if ((rc = make_tmap(h, &tmA, a_src, K, M, a_ld, sgemm_cfg::kTf32BK, box_a, CU_TENSOR_MAP_SWIZZLE_128B)) !=
        SGEMM_OK)
        return rc;
    if ((rc = make_tmap(h, &tmB, b_src, N, K, b_ld, 32, sgemm_cfg::kTf32BK, CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B)) !=
        SGEMM_OK)
        return rc;
    // plan.repack_c (C not 16-byte accessible, SGEMM_OPT_FORCE_REPACK_C = 1): computed in an
    // aligned copy, copied back at the end; otherwise the kernel writes C in place
    float *c_dst = C;
    long long c_ld = ldc;
    if (plan.repack_c) {
        c_dst = reinterpret_cast<float *>(ws + w.c_off);
        c_ld = w.ldc;
        if (beta != 0.0f && launch_repack(C, ldc, c_dst, c_ld, M, N, h->num_sms, stream) != cudaSuccess)
            return SGEMM_ERR_LAUNCH;
    }
    Tf32Params p{};
    p.M = M;
    p.N = N;
    p.K = K;
    p.alpha = alpha;
    p.beta = beta;
    p.C = c_dst;
    p.ldc = c_ld;
    p.tiles_m = plan.tiles_m;
    p.tiles_n = plan.tiles_n;
    p.units = plan.units;
    p.kblocks = (K + sgemm_cfg::kTf32BK - 1) / sgemm_cfg::kTf32BK;
    p.vec_c = plan.repack_c ? 1 : plan.vec_c;
    p.status = h->d_status;
    p.timeout_ns = h->timeout_ns;
    p.splits = 1;
    if (plan.sk_tiles > 0) {
        p.W = reinterpret_cast<float *>(ws + w.w_off);
        p.sk_tiles = plan.sk_tiles;
        p.sk_grid = plan.sk_grid;
        p.w_elems = (w.total - w.w_off) / 4;
    }
    const bool dependent = plan.repack_a || plan.repack_b || (plan.repack_c && beta != 0.0f);
    const cudaError_t le = pair ? launch_tf32_pair(tmA, tmB, p, plan.grid, stream, dependent)
                                : launch_tf32(tmA, tmB, p, plan.grid, stream, dependent);
    if (le != cudaSuccess) return SGEMM_ERR_LAUNCH;
    if (plan.sk_tiles > 0) {
        // Same raster and tile-packed partial layout as the FP32 stream-K span.
        FfmaParams r{};
        r.M = M;
        r.N = N;
        r.alpha = alpha;
        r.beta = beta;
        r.C = c_dst;
        r.ldc = c_ld;
        r.W = p.W;
        r.tiles_m = plan.tiles_m;
        r.tiles_n = plan.tiles_n;
        r.units = p.units;
        r.splits = 1;
        r.kblocks = p.kblocks;
        r.vec_c = p.vec_c;
        r.sk_tiles = p.sk_tiles;
        r.sk_grid = p.sk_grid;
        r.status = h->d_status;
        r.w_elems = p.w_elems;
        if (launch_sk_reduce(r, plan.bm, plan.bn, h->num_sms, stream) != cudaSuccess) return SGEMM_ERR_LAUNCH;
    }
    // (an ordinary launch: it waits for the kernels above to complete)
    if (plan.repack_c && launch_repack(c_dst, c_ld, C, ldc, M, N, h->num_sms, stream) != cudaSuccess)
        return SGEMM_ERR_LAUNCH;
    return SGEMM_OK;
}

// Streams and events of the host-buffer pipeline, created on first use.
int ensure_host_pipeline(sgemm_handle_t h)
{
    if (h->h2d != nullptr) return SGEMM_OK;
    bool ok = cudaStreamCreateWithFlags(&h->h2d, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&h->d2h, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&h->ev_start, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&h->ev_end, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; ok && i < kMaxHostSteps; ++i)
        ok = cudaEventCreateWithFlags(&h->ev_in[i], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&h->ev_done[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        return SGEMM_ERR_CUDA;
    }
    return SGEMM_OK;
}

// Pipeline schedule of sgemm_run_host: row panels of A and C (start rows,
// start[panels] = M) and the column blocks of B (col[blocks] = N) in which B is
// copied in and panel 0 is computed.
//
// Copy-in runs at ~200 GB/s on the host link; with B resident a row of C costs
// about three times longer to compute (2NK / ~70 TFLOP/s) than its A and C rows
// take to copy (4 (K + N) bytes at 200 GB/s, at 4096^3), so only the start of the
// pipeline is copy-bound: nothing can be computed before B has arrived. So B is
// copied in column blocks (up to 4, multiples of 128 columns: the first one small,
// 3N/16, so that the first GEMM starts early, then N/4 and two halves of the
// rest), and panel 0 is computed block by block as they arrive. Panel 0 is sized so that computing it
// takes about as long as B takes to arrive: 2 p N K / ~60 TFLOP/s (its GEMMs are
// small) against 4 K N / ~200 GB/s gives p ~ 600 rows whatever N and K; 768 (at
// most M / 4) measured best. Then panels grow, each at most three times its
// predecessor, so its copy-in finishes while the previous panel computes; the
// last panel is half of panel 0, so the copy-out after the last GEMM is short.
// Problems with less than two rounds of 128 x 128 tiles outside the edge panels
// are one panel and one block. All panels but the last have a multiple of 128
// rows. (M = N = K = 4096: panels 768 (blocks of 768, 1024, 1152 and 1152
// columns), 768, 2176, 384.)
struct HostSchedule {
    int panels = 1;
    int start[kMaxHostPanels + 1] = {};
    int blocks = 1;
    int col[kMaxColBlocks + 1] = {};
};

HostSchedule host_schedule(const sgemm_handle_s *h, int M, int N, int K, bool split_b)
{
    HostSchedule sc;
    sc.start[1] = M;
    sc.col[1] = N;
    if (static_cast<double>(M) * N * K < 1.0e9 || M < 1024) return sc;
    const int edge = std::max(128, std::min(768, M / 4 / 128 * 128));
    const int last = std::max(128, edge / 2 / 128 * 128);
    const long long mid_tiles = static_cast<long long>((M - 2 * edge + 127) / 128) * ((N + 127) / 128);
    if (mid_tiles < 2LL * h->num_sms) return sc;
    int P = 0, r = 0, size = edge;
    for (int i = 0;; ++i) {
        const int left = M - r;
        int take = i < 2 ? edge : 3 * size;
        take = std::min(take, left - last) / 128 * 128;  // leave at least `last` rows for the last panel
        if (left <= last || P == kMaxHostPanels - 1 || take <= 0) {
            sc.start[++P] = M;
            break;
        }
        r += take;
        sc.start[++P] = r;
        size = take;
    }
    sc.panels = P;
    if (split_b && N >= 1024) {
        // The first block small (3N/16: the first GEMM waits for less), the second
        // N/4, the rest in two halves; multiples of 128 columns.
        static_assert(kMaxColBlocks >= 4, "four column blocks");
        const int w0 = std::max(128, N * 3 / 16 / 128 * 128);
        const int w1 = std::max(128, N / 4 / 128 * 128);
        const int w2 = ((N - w0 - w1 + 1) / 2 + 127) / 128 * 128;
        sc.col[0] = 0;
        sc.col[1] = w0;
        sc.col[2] = w0 + w1;
        sc.blocks = w0 + w1 + w2 < N ? 4 : 3;
        if (sc.blocks == 4) sc.col[3] = w0 + w1 + w2;
        sc.col[sc.blocks] = N;
    } else if (split_b && N >= 512) {
        const int w = ((N + 1) / 2 + 127) / 128 * 128;
        sc.blocks = (N + w - 1) / w;
        for (int j = 0; j <= sc.blocks; ++j) sc.col[j] = std::min(N, j * w);
    }
    return sc;
}

int run_device(sgemm_handle_t h, int M, int N, int K, float alpha, const float *A, int lda, const float *B, int ldb,
               float beta, float *C, int ldc, cudaStream_t stream)
{
    const int align = (aligned16(A) ? 1 : 0) | (aligned16(B) ? 2 : 0) | (aligned16(C) ? 4 : 0);
    Problem q{M, N, K, lda, ldb, ldc, align, h->num_sms, h->math_mode, alpha, beta};
    q.num_pairs = h->tf32_pairs;
    sgemm_plan_t plan;
    int rc = make_plan(q, h->ov, &plan);
    if (rc != SGEMM_OK) return rc;
    if (plan.kernel == SGEMM_KERNEL_NONE || plan.kernel == SGEMM_KERNEL_SCALE) {
        if (h->log) log_plan(plan, M, N, K);
        h->last = plan;
        if (plan.kernel == SGEMM_KERNEL_NONE) return SGEMM_OK;
        return launch_scale(M, N, beta, C, ldc, h->num_sms, stream) == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
    }

    Workspace w = workspace_layout(q, plan);
    rc = ensure_workspace(h, static_cast<size_t>(w.total), stream);
    if (rc == SGEMM_ERR_ALLOC && plan.transpose_a == 1 && h->ov.force_transpose_a < 0) {
        // No room for A^T (a very large A): transpose A in shared memory instead, same results.
        Overrides ov = h->ov;
        ov.force_transpose_a = 2;
        if ((rc = make_plan(q, ov, &plan)) != SGEMM_OK) return rc;
        w = workspace_layout(q, plan);
        rc = ensure_workspace(h, static_cast<size_t>(w.total), stream);
    }
    if (h->log) log_plan(plan, M, N, K);
    h->last = plan;
    if (rc != SGEMM_OK) return rc;
    char *ws = static_cast<char *>(h->workspace);

    const float *a_src = A;
    long long a_ld = lda;
    const float *b_src = B;
    long long b_ld = ldb;
    if (plan.kernel == SGEMM_KERNEL_TF32) return run_tf32(h, plan, w, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
    const bool copy_a = plan.transpose_a == 1 || plan.repack_a;
    if (copy_a && plan.repack_b) {  // both operand copies in one launch
        float *a_dst = reinterpret_cast<float *>(ws + w.a_off);
        float *b_dst = reinterpret_cast<float *>(ws + w.b_off);
        if (launch_prep(A, lda, a_dst, w.lda, M, K, plan.transpose_a == 1, B, ldb, b_dst, w.ldb, K, N, h->num_sms,
                        stream) != cudaSuccess)
            return SGEMM_ERR_LAUNCH;
        a_src = a_dst;
        a_ld = w.lda;
        b_src = b_dst;
        b_ld = w.ldb;
    } else if (plan.transpose_a == 1) {
        float *dst = reinterpret_cast<float *>(ws + w.a_off);
        if (launch_transpose(A, lda, dst, w.lda, M, K, stream) != cudaSuccess) return SGEMM_ERR_LAUNCH;
        a_src = dst;
        a_ld = w.lda;
    } else if (plan.repack_a) {
        float *dst = reinterpret_cast<float *>(ws + w.a_off);
        if (launch_repack(A, lda, dst, w.lda, M, K, h->num_sms, stream) != cudaSuccess) return SGEMM_ERR_LAUNCH;
        a_src = dst;
        a_ld = w.lda;
    } else if (plan.repack_b) {
        float *dst = reinterpret_cast<float *>(ws + w.b_off);
        if (launch_repack(B, ldb, dst, w.ldb, K, N, h->num_sms, stream) != cudaSuccess) return SGEMM_ERR_LAUNCH;
        b_src = dst;
        b_ld = w.ldb;
    }

    CUtensorMap tmA, tmB;
    if (plan.transpose_a == 1)  // A^T: K rows of M, boxes of 32 k x BM m
        rc = make_tmap(h, &tmA, a_src, M, K, a_ld, plan.bm, sgemm_cfg::kFfmaBK, CU_TENSOR_MAP_SWIZZLE_NONE);
    else  // A (as given, or turned M-major in shared memory): M rows of K, boxes of BM m x 32 k, 128-byte swizzle
        rc = make_tmap(h, &tmA, a_src, K, M, a_ld, sgemm_cfg::kFfmaBK, plan.bm, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != SGEMM_OK) return rc;
    if ((rc = make_tmap(h, &tmB, b_src, N, K, b_ld, plan.bn, sgemm_cfg::kFfmaBK, CU_TENSOR_MAP_SWIZZLE_NONE)) !=
        SGEMM_OK)
        return rc;

    FfmaParams p{};
    p.M = M;
    p.N = N;
    p.K = K;
    p.alpha = alpha;
    p.beta = beta;
    p.C = C;
    p.ldc = ldc;
    p.W = plan.splits > 1 && !plan.cluster_split ? reinterpret_cast<float *>(ws + w.w_off) : nullptr;
    p.ldw = w.ldw;
    p.wstride = w.wstride;
    p.splits = plan.splits;
    p.tiles_m = plan.tiles_m;
    p.tiles_n = plan.tiles_n;
    p.units = plan.units;
    p.kblocks = (K + sgemm_cfg::kFfmaBK - 1) / sgemm_cfg::kFfmaBK;
    p.vec_c = plan.vec_c;
    p.status = h->d_status;
    p.timeout_ns = h->timeout_ns;
    p.inject_skip = h->inject_skip;
    p.skew_ns = h->skew_ns;
    if (plan.sk_tiles > 0) {
        p.W = reinterpret_cast<float *>(ws + w.w_off);
        p.sk_tiles = plan.sk_tiles;
        p.sk_grid = plan.sk_grid;
    }
    p.cluster_split = plan.cluster_split ? plan.splits : 0;
    p.w_elems = p.W != nullptr ? (w.total - w.w_off) / 4 : 0;
    // Right after this call's transpose / repack: launched as its programmatic dependent.
    const bool after_copy = plan.transpose_a == 1 || plan.repack_a || plan.repack_b;
    if (launch_ffma(plan.config, plan.transpose_a, tmA, tmB, p, plan.grid, stream, after_copy) != cudaSuccess)
        return SGEMM_ERR_LAUNCH;
    if (plan.sk_tiles > 0 && launch_sk_reduce(p, plan.bm, plan.bn, h->num_sms, stream) != cudaSuccess)
        return SGEMM_ERR_LAUNCH;
    if (plan.splits > 1 && !plan.cluster_split) {
        if (launch_splitk_reduce(p.W, w.ldw, w.wstride, plan.splits, M, N, alpha, beta, C, ldc, plan.vec_c,
                                 h->num_sms, stream, p.w_elems, h->d_status) != cudaSuccess)
            return SGEMM_ERR_LAUNCH;
    }
    return SGEMM_OK;
}

}  // namespace

extern "C" {

int sgemm_create(sgemm_handle_t *out)
{
    if (out == nullptr) return SGEMM_ERR_INVALID_VALUE;
    *out = nullptr;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SGEMM_ERR_ARCH;
    }
    return sgemm_create_for_device(dev, out);
}

int sgemm_create_for_device(int dev, sgemm_handle_t *out)
{
    if (out == nullptr) return SGEMM_ERR_INVALID_VALUE;
    *out = nullptr;
    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess || dev < 0 || dev >= count) {
        cudaGetLastError();
        return count > 0 ? SGEMM_ERR_INVALID_VALUE : SGEMM_ERR_ARCH;
    }
    DeviceGuard g(dev);
    if (!g.ok) return SGEMM_ERR_CUDA;
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return SGEMM_ERR_ARCH;
    }
    if (major != 10 || minor != 3) return SGEMM_ERR_ARCH;

    sgemm_handle_t h = new (std::nothrow) sgemm_handle_s();
    if (h == nullptr) return SGEMM_ERR_ALLOC;
    h->device = dev;
    h->num_sms = sms;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qr) !=
            cudaSuccess ||
        qr != cudaDriverEntryPointSuccess || fn == nullptr) {
        delete h;
        return SGEMM_ERR_CUDA;
    }
    h->encode = reinterpret_cast<EncodeTiledFn>(fn);
    if (ffma_set_attributes() != cudaSuccess || tf32_set_attributes() != cudaSuccess) {
        cudaGetLastError();
        delete h;
        return SGEMM_ERR_CUDA;
    }
    {
        const int pairs = tf32_pair_max_pairs();
        h->tf32_pairs = pairs > 0 ? std::min(pairs, sms / 2) : -1;
    }
    if (cudaMalloc(&h->d_status, 256) != cudaSuccess || cudaMemset(h->d_status, 0, 256) != cudaSuccess ||
        cudaMalloc(&h->min2_cand, min2_candidate_bytes(8 * sms)) != cudaSuccess) {
        cudaGetLastError();
        if (h->d_status) cudaFree(h->d_status);
        if (h->min2_cand) cudaFree(h->min2_cand);
        delete h;
        return SGEMM_ERR_ALLOC;
    }
    const char *env = std::getenv("SGEMM_LOG");
    h->log = (env != nullptr && env[0] == '1') ? 1 : 0;
    // Tuning overrides for the planner (same ranges as sgemm_set_option).
    if (const char *fc = std::getenv("SGEMM_FORCE_CONFIG")) {
        const long v = std::strtol(fc, nullptr, 10);
        if (v >= -1 && v < sgemm_cfg::kNumFfmaConfigs) h->ov.force_config = static_cast<int>(v);
    }
    if (const char *fs = std::getenv("SGEMM_FORCE_SPLITS")) {
        const long v = std::strtol(fs, nullptr, 10);
        if (v >= 0 && v <= kMaxSplits) h->ov.force_splits = static_cast<int>(v);
    }
    if (const char *ft = std::getenv("SGEMM_FORCE_TRANSPOSE_A")) {
        const long v = std::strtol(ft, nullptr, 10);
        if (v >= -1 && v <= 2) h->ov.force_transpose_a = static_cast<int>(v);
    }
    if (const char *fc2 = std::getenv("SGEMM_CLUSTER_SPLIT")) {
        const long v = std::strtol(fc2, nullptr, 10);
        if (v >= -1 && v <= 1) h->ov.cluster_split = static_cast<int>(v);
    }
    if (const char *fk = std::getenv("SGEMM_FORCE_STREAMK")) {
        const long v = std::strtol(fk, nullptr, 10);
        if (v >= -1 && v <= 1) h->ov.force_streamk = static_cast<int>(v);
    }
    if (const char *fp = std::getenv("SGEMM_FORCE_TF32_KERNEL")) {
        const long v = std::strtol(fp, nullptr, 10);
        if (v >= -1 && v <= 1) h->ov.force_tf32_kernel = static_cast<int>(v);
    }
    *out = h;
    return SGEMM_OK;
}

int sgemm_destroy(sgemm_handle_t h)
{
    if (h == nullptr) return SGEMM_OK;
    DeviceGuard g(h->device);
    cudaDeviceSynchronize();
    if (h->workspace) cudaFree(h->workspace);
    if (h->stage) cudaFree(h->stage);
    if (h->min2_cand) cudaFree(h->min2_cand);
    if (h->h2d) cudaStreamDestroy(h->h2d);
    if (h->d2h) cudaStreamDestroy(h->d2h);
    for (cudaEvent_t e : {h->ev_start, h->ev_end})
        if (e) cudaEventDestroy(e);
    for (int i = 0; i < kMaxHostSteps; ++i) {
        if (h->ev_in[i]) cudaEventDestroy(h->ev_in[i]);
        if (h->ev_done[i]) cudaEventDestroy(h->ev_done[i]);
    }
    if (h->d_status) cudaFree(h->d_status);
    delete h;
    return SGEMM_OK;
}

int sgemm_run(sgemm_handle_t h, int M, int N, int K, float alpha, const float *A, int lda, const float *B, int ldb,
              float beta, float *C, int ldc, struct CUstream_st *stream)
{
    const int v = check_args(h, M, N, K, alpha, A, lda, B, ldb, C, ldc);
    if (v != SGEMM_OK) return v;
    DeviceGuard g(h->device);
    if (!g.ok) return SGEMM_ERR_CUDA;
    return run_device(h, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
}

int sgemm_run_host(sgemm_handle_t h, int M, int N, int K, float alpha, const float *A, int lda, const float *B,
                   int ldb, float beta, float *C, int ldc, struct CUstream_st *stream)
{
    const int v = check_args(h, M, N, K, alpha, A, lda, B, ldb, C, ldc);
    if (v != SGEMM_OK) return v;
    if (M == 0 || N == 0) return SGEMM_OK;
    DeviceGuard g(h->device);
    if (!g.ok) return SGEMM_ERR_CUDA;
    const bool need_ab = K > 0 && alpha != 0.0f;
    // Device copies with row strides rounded up to 4 floats keep every
    // operand on the aligned (TMA, 16-byte) path.
    const long long dlda = (K + 3) / 4 * 4, dldb = (N + 3) / 4 * 4, dldc = (N + 3) / 4 * 4;
    const long long a_elems = need_ab ? static_cast<long long>(M) * (dlda > 0 ? dlda : 4) : 0;
    const long long b_elems = need_ab ? static_cast<long long>(K) * dldb : 0;
    const long long c_elems = static_cast<long long>(M) * dldc;
    const size_t bytes = static_cast<size_t>(a_elems + b_elems + c_elems) * 4u + 512u;
    if (bytes > h->stage_bytes) {
        if (h->stage) {
            if (cudaDeviceSynchronize() != cudaSuccess) return SGEMM_ERR_CUDA;
            cudaFree(h->stage);
            h->stage = nullptr;
            h->stage_bytes = 0;
        }
        if (cudaMalloc(&h->stage, bytes) != cudaSuccess) {
            cudaGetLastError();
            return SGEMM_ERR_ALLOC;
        }
        h->stage_bytes = bytes;
    }
    float *dA = h->stage;
    float *dB = dA + (a_elems + 63) / 64 * 64;
    float *dC = dB + (b_elems + 63) / 64 * 64;
    int rc = ensure_host_pipeline(h);
    if (rc != SGEMM_OK) return rc;

    // Pipeline (host_schedule): on the copy-in stream, B block by block with panel
    // 0's A rows and its C block beside each, then each later panel's A and C rows;
    // every GEMM runs on `stream` once its copies are in (events), and its C rows
    // are copied back on the copy-out stream while later GEMMs compute. Every GEMM
    // is an ordinary device call on the staged copies.
    cudaStream_t s = stream;
    const HostSchedule sc = host_schedule(h, M, N, K, need_ab);
    const bool copy_c_in = beta != 0.0f;
    bool ok = cudaEventRecord(h->ev_start, s) == cudaSuccess && cudaStreamWaitEvent(h->h2d, h->ev_start, 0) == cudaSuccess &&
              cudaStreamWaitEvent(h->d2h, h->ev_start, 0) == cudaSuccess;
    int step = 0;
    for (int p = 0; ok && p < sc.panels; ++p) {
        const int r0 = sc.start[p];
        const int mp = sc.start[p + 1] - r0;
        const float *hA = A + static_cast<long long>(r0) * lda;
        float *hC = C + static_cast<long long>(r0) * ldc;
        float *pA = dA + static_cast<long long>(r0) * dlda;
        float *pC = dC + static_cast<long long>(r0) * dldc;
        // panel 0 in B's column blocks; later panels whole (all of B is in by then)
        const int nblk = p == 0 ? sc.blocks : 1;
        for (int j = 0; ok && j < nblk; ++j) {
            const int c0 = p == 0 ? sc.col[j] : 0;
            const int nc = p == 0 ? sc.col[j + 1] - c0 : N;
            if (p == 0 && need_ab)
                ok = cudaMemcpy2DAsync(dB + c0, dldb * 4, B + c0, static_cast<size_t>(ldb) * 4,
                                       static_cast<size_t>(nc) * 4, K, cudaMemcpyHostToDevice, h->h2d) == cudaSuccess;
            if (ok && j == 0 && need_ab)
                ok = cudaMemcpy2DAsync(pA, dlda * 4, hA, static_cast<size_t>(lda) * 4, static_cast<size_t>(K) * 4, mp,
                                       cudaMemcpyHostToDevice, h->h2d) == cudaSuccess;
            if (ok && copy_c_in)
                ok = cudaMemcpy2DAsync(pC + c0, dldc * 4, hC + c0, static_cast<size_t>(ldc) * 4,
                                       static_cast<size_t>(nc) * 4, mp, cudaMemcpyHostToDevice, h->h2d) == cudaSuccess;
            ok = ok && cudaEventRecord(h->ev_in[step], h->h2d) == cudaSuccess &&
                 cudaStreamWaitEvent(s, h->ev_in[step], 0) == cudaSuccess;
            if (!ok) break;
            rc = run_device(h, mp, nc, K, alpha, need_ab ? pA : nullptr, static_cast<int>(dlda > 0 ? dlda : 1),
                            need_ab ? dB + c0 : nullptr, static_cast<int>(dldb), beta, pC + c0, static_cast<int>(dldc), s);
            if (rc != SGEMM_OK) break;
            const bool c_changed = h->last.kernel != SGEMM_KERNEL_NONE;  // alpha == 0 / K == 0 with beta == 1
            ok = cudaEventRecord(h->ev_done[step], s) == cudaSuccess &&
                 cudaStreamWaitEvent(h->d2h, h->ev_done[step], 0) == cudaSuccess;
            if (ok && c_changed)
                ok = cudaMemcpy2DAsync(hC + c0, static_cast<size_t>(ldc) * 4, pC + c0, dldc * 4,
                                       static_cast<size_t>(nc) * 4, mp, cudaMemcpyDeviceToHost, h->d2h) == cudaSuccess;
            ++step;
        }
        if (rc != SGEMM_OK) break;
    }
    // Join the copy streams back into `stream` and wait: on success and on
    // failure alike no copy into the caller's host buffers is left in flight.
    const bool joined = cudaEventRecord(h->ev_end, h->d2h) == cudaSuccess &&
                        cudaStreamWaitEvent(s, h->ev_end, 0) == cudaSuccess;
    const cudaError_t e1 = cudaStreamSynchronize(h->h2d);
    const cudaError_t e2 = cudaStreamSynchronize(h->d2h);
    const cudaError_t e3 = cudaStreamSynchronize(s);
    if (rc != SGEMM_OK) return rc;
    if (!ok || !joined || e1 != cudaSuccess || e2 != cudaSuccess || e3 != cudaSuccess) {
        cudaGetLastError();
        return SGEMM_ERR_CUDA;
    }
    return SGEMM_OK;
}

int sgemm_run_min2(sgemm_handle_t h, int M, int N, int K, float alpha, const float *A, int lda, const float *B,
                   int ldb, float beta, float *C, int ldc, float *min_vals, int *min_ij, struct CUstream_st *stream)
{
    const int v = check_args(h, M, N, K, alpha, A, lda, B, ldb, C, ldc);
    if (v != SGEMM_OK) return v;
    if (min_vals == nullptr || min_ij == nullptr || !elem_aligned(min_vals) || !elem_aligned(min_ij))
        return SGEMM_ERR_INVALID_VALUE;
    DeviceGuard g(h->device);
    if (!g.ok) return SGEMM_ERR_CUDA;
    int rc = run_device(h, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
    if (rc != SGEMM_OK) return rc;
    const int blocks = 8 * h->num_sms;  // the candidate buffer is sized for this at handle creation
    return launch_min2(C, ldc, M, N, h->min2_cand, blocks, min_vals, min_ij, stream) == cudaSuccess
               ? SGEMM_OK
               : SGEMM_ERR_LAUNCH;
}

int sgemm_ladder_run(int rung, int M, int N, int K, float alpha, const float *A, const float *B, float beta, float *C,
                     struct CUstream_st *stream)
{
    if (rung < 1 || rung > 8 || M < 0 || N < 0 || K < 0) return SGEMM_ERR_INVALID_VALUE;
    if (!elem_aligned(A) || !elem_aligned(B) || !elem_aligned(C)) return SGEMM_ERR_INVALID_VALUE;
    if (M == 0 || N == 0) return SGEMM_OK;
    if (C == nullptr || (K > 0 && (A == nullptr || B == nullptr))) return SGEMM_ERR_INVALID_VALUE;
    if (M > (1 << 21)) return SGEMM_ERR_NOT_SUPPORTED;
    if (rung >= 6 && (K % 4 != 0 || N % 4 != 0 || !aligned16(A) || !aligned16(B))) return SGEMM_ERR_NOT_SUPPORTED;
    const cudaError_t e = launch_ladder(rung, M, N, K, alpha, A, B, beta, C, stream);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return SGEMM_ERR_LAUNCH;
    }
    return SGEMM_OK;
}

int sgemm_set_math_mode(sgemm_handle_t h, int mode)
{
    if (h == nullptr || (mode != SGEMM_MATH_FP32 && mode != SGEMM_MATH_TF32)) return SGEMM_ERR_INVALID_VALUE;
    h->math_mode = mode;
    return SGEMM_OK;
}

int sgemm_get_math_mode(sgemm_handle_t h, int *mode)
{
    if (h == nullptr || mode == nullptr) return SGEMM_ERR_INVALID_VALUE;
    *mode = h->math_mode;
    return SGEMM_OK;
}

int sgemm_set_option(sgemm_handle_t h, int option, long long value)
{
    if (h == nullptr) return SGEMM_ERR_INVALID_VALUE;
    switch (option) {
    case SGEMM_OPT_FORCE_CONFIG:
        if (value < -1 || value >= sgemm_cfg::kNumFfmaConfigs) return SGEMM_ERR_INVALID_VALUE;
        h->ov.force_config = static_cast<int>(value);
        return SGEMM_OK;
    case SGEMM_OPT_FORCE_SPLITS:
        if (value < 0 || value > kMaxSplits) return SGEMM_ERR_INVALID_VALUE;
        h->ov.force_splits = static_cast<int>(value);
        return SGEMM_OK;
    case SGEMM_OPT_WAIT_TIMEOUT_NS:
        if (value < 1000000LL || value > 60000000000LL) return SGEMM_ERR_INVALID_VALUE;
        h->timeout_ns = value;
        return SGEMM_OK;
    case SGEMM_OPT_INJECT_SKIP:
        if (value < -1 || value > (1LL << 30)) return SGEMM_ERR_INVALID_VALUE;
        h->inject_skip = static_cast<int>(value);
        return SGEMM_OK;
    case SGEMM_OPT_LOG:
        h->log = value ? 1 : 0;
        return SGEMM_OK;
    case SGEMM_OPT_SKEW_NS:
        if (value < -100000 || value > 100000) return SGEMM_ERR_INVALID_VALUE;
        h->skew_ns = static_cast<int>(value);
        return SGEMM_OK;
    case SGEMM_OPT_FORCE_TRANSPOSE_A:
        if (value < -1 || value > 2) return SGEMM_ERR_INVALID_VALUE;
        h->ov.force_transpose_a = static_cast<int>(value);
        return SGEMM_OK;
    case SGEMM_OPT_FORCE_STREAMK:
        if (value < -1 || value > 1) return SGEMM_ERR_INVALID_VALUE;
        h->ov.force_streamk = static_cast<int>(value);
        return SGEMM_OK;
    case SGEMM_OPT_FORCE_TF32_KERNEL:
        if (value < -1 || value > 1) return SGEMM_ERR_INVALID_VALUE;
        h->ov.force_tf32_kernel = static_cast<int>(value);
        return SGEMM_OK;
    case SGEMM_OPT_CLUSTER_SPLIT:
        if (value < -1 || value > 1) return SGEMM_ERR_INVALID_VALUE;
        h->ov.cluster_split = static_cast<int>(value);
        return SGEMM_OK;
    case SGEMM_OPT_FORCE_REPACK_C:
        if (value < -1 || value > 1) return SGEMM_ERR_INVALID_VALUE;
        h->ov.force_repack_c = static_cast<int>(value);
        return SGEMM_OK;
    default:
        return SGEMM_ERR_INVALID_VALUE;
    }
}

int sgemm_check_device_status(sgemm_handle_t h, struct CUstream_st *stream, int *device_status)
{
    if (h == nullptr) return SGEMM_ERR_INVALID_VALUE;
    DeviceGuard g(h->device);
    if (!g.ok) return SGEMM_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return SGEMM_ERR_CUDA;
    int code = 0;
    if (cudaMemcpy(&code, h->d_status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return SGEMM_ERR_CUDA;
    if (code != 0 && cudaMemset(h->d_status, 0, sizeof(int)) != cudaSuccess) return SGEMM_ERR_CUDA;
    if (device_status) *device_status = code;
    return code == 0 ? SGEMM_OK : (code >> 16);
}

int sgemm_plan(int M, int N, int K, int lda, int ldb, int ldc, int align_flags, int num_sms, int math_mode,
               sgemm_plan_t *out)
{
    if (out == nullptr) return SGEMM_ERR_INVALID_VALUE;
    Problem q{M, N, K, lda, ldb, ldc, align_flags, num_sms, math_mode, 1.0f, 1.0f};
    return make_plan(q, Overrides{}, out);
}

int sgemm_reserve(sgemm_handle_t h, long long workspace_bytes)
{
    if (h == nullptr || workspace_bytes < 0) return SGEMM_ERR_INVALID_VALUE;
    DeviceGuard g(h->device);
    if (!g.ok) return SGEMM_ERR_CUDA;
    return ensure_workspace(h, static_cast<size_t>(workspace_bytes), nullptr);
}

int sgemm_last_plan(sgemm_handle_t h, sgemm_plan_t *out)
{
    if (h == nullptr || out == nullptr) return SGEMM_ERR_INVALID_VALUE;
    *out = h->last;
    return SGEMM_OK;
}

int sgemm_config_count(void) { return sgemm_cfg::kNumFfmaConfigs; }

int sgemm_config_info(int index, sgemm_plan_t *out)
{
    if (out == nullptr || index < 0 || index >= sgemm_cfg::kNumFfmaConfigs) return SGEMM_ERR_INVALID_VALUE;
    config_as_plan(index, out);
    return SGEMM_OK;
}

const char *sgemm_status_string(int status)
{
    switch (status) {
    case SGEMM_OK: return "SGEMM_OK: success";
    case SGEMM_ERR_INVALID_VALUE: return "SGEMM_ERR_INVALID_VALUE: invalid dimension, leading dimension, pointer, handle or option";
    case SGEMM_ERR_ARCH: return "SGEMM_ERR_ARCH: the current device is not an sm_103 (GB300) GPU";
    case SGEMM_ERR_ALLOC: return "SGEMM_ERR_ALLOC: device allocation failed";
    case SGEMM_ERR_LAUNCH: return "SGEMM_ERR_LAUNCH: kernel launch failed";
    case SGEMM_ERR_TIMEOUT: return "SGEMM_ERR_TIMEOUT: a bounded in-kernel wait ran out";
    case SGEMM_ERR_CUDA: return "SGEMM_ERR_CUDA: a CUDA runtime or driver call failed";
    case SGEMM_ERR_NOT_SUPPORTED: return "SGEMM_ERR_NOT_SUPPORTED: valid request that is not implemented";
    case SGEMM_ERR_INDEX: return "SGEMM_ERR_INDEX: a device-side index check of a debug build failed (access skipped)";
    default: return "unknown sgemm status";
    }
}

}  // extern "C"
