/*
 * sgemm.h — single-precision GEMM for NVIDIA GB300 (sm_103a), C ABI.
 *
 * The operation (all calls below compute it):
 *
 *     C = alpha * A * B + beta * C
 *
 *   A is M x K, B is K x N, C is M x N, FP32, all three row-major:
 *   element (i, k) of A is A[i*lda + k], (k, j) of B is B[k*ldb + j],
 *   (i, j) of C is C[i*ldc + j]. All offsets are computed in 64 bits.
 *
 *   Source of the definition: "SGEMM CUDA kernel (First Half)", opening
 *   definition (S = single precision, GEMM: C = alpha AB + beta C, A is M x K,
 *   B is K x N) and its Part 1 (row-major offsets row * ncols + col);
 *   "Optimizing Matrix Multiplication in CUDA", the kernels' argument order
 *   (M, N, K, alpha, A, B, beta, C) in the global-memory coalescing section.
 *   Leading dimensions (row strides >= the column count) are this library's
 *   extension; the pages use packed matrices.
 *
 * Conventions where the pages are silent (BLAS practice):
 *   - M == 0 or N == 0: nothing is touched, SGEMM_OK.
 *   - K == 0 or alpha == 0: A and B are not read; C = beta * C
 *     (beta == 1: C untouched; beta == 0: C set to +0 without being read).
 *   - beta == 0: C is never read, so NaN/Inf already in C does not propagate.
 *   - C must not overlap A or B.
 *   - Misaligned pointers or leading dimensions are not an error: the library
 *     switches to a path that does not need 16-byte alignment.
 *
 * Numerics: the default mode (SGEMM_MATH_FP32) performs only IEEE FP32 fused
 * multiply-adds (round to nearest even); each output is within
 * (K + 2) * 2^-24 * (|alpha| sum_k |a_ik||b_kj| + |beta||c_ij|) of the exact
 * result, and is bitwise reproducible for a fixed (shape, alignment, plan).
 * SGEMM_MATH_TF32 rounds A and B to TF32 on the tensor cores: the same bound
 * holds with 2^-10 in place of 2^-24.
 *
 * Errors: every call returns an sgemm_status value. Launches are asynchronous
 * on the given stream; a kernel watchdog (bounded waits inside the kernels)
 * records SGEMM_ERR_TIMEOUT in the handle's device status word, which
 * sgemm_check_device_status() reads.
 */
#ifndef SGEMM_GB300_H
#define SGEMM_GB300_H

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* same type as cudaStream_t; NULL means the legacy default stream */

typedef struct sgemm_handle_s *sgemm_handle_t;

typedef enum sgemm_status {
    SGEMM_OK = 0,
    SGEMM_ERR_INVALID_VALUE = 1, /* bad dimension, leading dimension, pointer, handle or option */
    SGEMM_ERR_ARCH = 2,          /* current device is not sm_103 (GB300) */
    SGEMM_ERR_ALLOC = 3,         /* device or pinned allocation failed */
    SGEMM_ERR_LAUNCH = 4,        /* a kernel launch failed (cudaGetLastError) */
    SGEMM_ERR_TIMEOUT = 5,       /* a kernel's bounded wait ran out (see sgemm_check_device_status) */
    SGEMM_ERR_CUDA = 6,          /* another CUDA runtime/driver call failed */
    SGEMM_ERR_NOT_SUPPORTED = 7, /* the request is valid but not implemented */
    SGEMM_ERR_INDEX = 8          /* debug builds only (SGEMM_DEBUG_CHECKS): a device-side index
                                    check failed and its access was skipped (see
                                    sgemm_check_device_status for the location codes) */
} sgemm_status_t;

typedef enum sgemm_math_mode {
    SGEMM_MATH_FP32 = 0, /* default: FP32 FFMA on the CUDA cores, exact-FP32 semantics */
    SGEMM_MATH_TF32 = 1  /* opt-in: tcgen05 tensor cores with TF32 inputs, FP32 accumulate */
} sgemm_math_mode_t;

/* Kernels a plan can use (sgemm_plan_t.kernel). */
typedef enum sgemm_kernel_kind {
    SGEMM_KERNEL_NONE = 0,  /* quick return, nothing launched */
    SGEMM_KERNEL_SCALE = 1, /* C = beta * C only (K == 0 or alpha == 0) */
    SGEMM_KERNEL_FFMA = 2,  /* FP32 FFMA mainloop */
    SGEMM_KERNEL_TF32 = 3   /* tcgen05 TF32 mainloop */
} sgemm_kernel_kind_t;

/* What sgemm_run does for one problem (filled by sgemm_plan / sgemm_last_plan). */
typedef struct sgemm_plan_s {
    int kernel;              /* sgemm_kernel_kind_t */
    int config;              /* FFMA: row of the tile-config table; TF32: 0 = one CTA per 128 x 256
                                tile, 1 = CTA pair per 256 x 256 tile (grid counts CTAs, sk_grid
                                pairs); -1 if none */
    int bm, bn, bk, stages;  /* CTA tile and pipeline depth */
    int threads;             /* threads per CTA */
    int ctas_per_sm;         /* resident CTAs per SM the grid is sized for */
    int splits;              /* split-K factor S (1 = fused epilogue) */
    int tiles_m, tiles_n;    /* output tiles */
    int units;               /* work units: tiles_m * tiles_n * splits; with stream-K the whole
                                tiles before the stream-K span */
    int grid;                /* CTAs launched (persistent: min(units, SMs * ctas_per_sm)) */
    int repack_a, repack_b;  /* operand first copied to a 16-byte-aligned workspace copy */
    int vec_c;               /* 1: C (base and ldc) 16-byte accessible, read/written with 16-byte
                                accesses; 0: 4-byte accesses (FP32 path), or in TF32 mode 16-byte
                                accesses from each row's first 16-byte boundary on */
    int math_mode;           /* sgemm_math_mode_t */
    int launches;            /* kernels one sgemm_run launches for this plan */
    long long workspace_bytes; /* device workspace the handle holds for it */
    int transpose_a;         /* FP32 mainloop's A layout: 1 = A is first transposed into the
                                workspace (K x M, M contiguous) and the mainloop reads A^T;
                                2 = A is staged as given and a transposer warp turns each slab
                                M-major in shared memory (no copy; stages/threads then describe
                                that form: a shorter ring, one more warp); 0 = A is read as given */
    int sk_tiles;            /* stream-K (both modes): the last sk_tiles tiles (after `units`
                                whole tiles) form one span of k-blocks cut evenly over the grid's
                                CTAs; tiles shared by two or more CTAs are reduced in k order
                                (0 = none) */
    int sk_grid;             /* workers sharing the stream-K span (the first sk_grid CTAs, or CTA
                                pairs for the TF32 pair kernel) */
    int repack_c;            /* TF32 mode, C not 16-byte accessible and SGEMM_OPT_FORCE_REPACK_C
                                = 1: C is computed in an aligned workspace copy (filled from C
                                when beta != 0) and copied back (0: C written in place) */
    int cluster_split;       /* FP32 split-K (2 <= splits <= 8): 1 = the `splits` CTAs of a tile
                                form one thread-block cluster and add their partial tiles in
                                distributed shared memory (one CTA per (tile, slice), grid =
                                units, no workspace and no reduction launch); 0 = partials go
                                through the workspace to a reduction kernel */
} sgemm_plan_t;

/* Tuning and test options for sgemm_set_option. */
typedef enum sgemm_option {
    SGEMM_OPT_FORCE_CONFIG = 1,   /* table row to use (-1 = automatic, the default) */
    SGEMM_OPT_FORCE_SPLITS = 2,   /* split-K factor (0 = automatic, the default) */
    SGEMM_OPT_WAIT_TIMEOUT_NS = 3,/* watchdog limit of every in-kernel wait (default 4e9 ns) */
    SGEMM_OPT_INJECT_SKIP = 4,    /* TEST ONLY: CTA 0 never issues the copy of its n-th k-slab
                                     (-1 = off, the default); the consumers' wait then runs out
                                     and the run reports SGEMM_ERR_TIMEOUT without faulting */
    SGEMM_OPT_LOG = 5,            /* 1: print the chosen plan of each call to stderr */
    SGEMM_OPT_SKEW_NS = 6,        /* TEST ONLY (race detection): > 0 delays the FP32 kernel's copy
                                     issue by this many ns per k-slab, < 0 delays every compute warp
                                     before it releases a slab; |value| <= 100000, 0 = off */
    SGEMM_OPT_FORCE_TRANSPOSE_A = 7,/* FP32 path: -1 = automatic (the default), 0 = read A as given,
                                     1 = always transpose A first in global memory, 2 = always
                                     transpose A in shared memory (same results every way) */
    SGEMM_OPT_FORCE_STREAMK = 8,  /* -1 = automatic (the default), 0 = never, 1 = whenever the last
                                     round of tiles is partial (ignored with forced splits) */
    SGEMM_OPT_FORCE_TF32_KERNEL = 9, /* TF32 mode: -1 = automatic (the default), 0 = one CTA per
                                     128 x 256 tile, 1 = a CTA pair (cluster of two, tcgen05
                                     .cta_group::2) per 256 x 256 tile; 1 fails with
                                     SGEMM_ERR_NOT_SUPPORTED where no pair fits */
    SGEMM_OPT_FORCE_REPACK_C = 10,/* TF32 mode, C not 16-byte accessible: -1 = automatic (the
                                     default) and 0 = write C in place (16-byte accesses inside
                                     each row, element by element at its ends); 1 = compute into
                                     an aligned workspace copy of C and copy it back */
    SGEMM_OPT_CLUSTER_SPLIT = 11  /* FP32 split-K: -1 = automatic (the default), 0 = partials
                                     always through the workspace and a reduction kernel, 1 =
                                     always within thread-block clusters when 2..8 splits (same
                                     results either way) */
} sgemm_option_t;

/*
 * Create a handle bound to the current CUDA device.
 * out: receives the handle (set to NULL on failure).
 * Returns SGEMM_ERR_ARCH unless the device is compute capability 10.3,
 * SGEMM_ERR_ALLOC if its small device status word cannot be allocated.
 * The handle owns a lazily grown device workspace (the transposed copy of A,
 * aligned operand copies, split-K and stream-K partials) and, for
 * sgemm_run_host, device staging buffers.
 * A handle must not be used by two host threads or two streams at once.
 * Environment: SGEMM_LOG=1 logs every plan; SGEMM_FORCE_CONFIG=<row> and
 * SGEMM_FORCE_SPLITS=<S>, SGEMM_FORCE_TRANSPOSE_A=<-1|0|1|2>,
 * SGEMM_FORCE_STREAMK=<-1|0|1>, SGEMM_FORCE_TF32_KERNEL=<-1|0|1> and
 * SGEMM_CLUSTER_SPLIT=<-1|0|1> preset the
 * planner overrides of sgemm_set_option.
 */
int sgemm_create(sgemm_handle_t *out);

/* Same as sgemm_create for CUDA device ordinal `device` (the calling thread's
 * current device is left unchanged). SGEMM_ERR_INVALID_VALUE for an ordinal
 * that does not exist. */
int sgemm_create_for_device(int device, sgemm_handle_t *out);

/* Free the handle and everything it owns. NULL is accepted. Waits for the
 * device to finish work that may still use the workspace. */
int sgemm_destroy(sgemm_handle_t h);

/*
 * C = alpha * A * B + beta * C on the device, asynchronously on `stream`.
 * A, B, C: caller-owned DEVICE pointers (the library never frees them).
 * Requirements: M, N, K >= 0; lda >= max(1, K); ldb >= max(1, N);
 * ldc >= max(1, N); A and B non-NULL when M, N > 0 and K > 0 and alpha != 0;
 * C non-NULL when M, N > 0; A, B and C 4-byte aligned (a float's alignment;
 * 16-byte alignment only selects the faster path). Any violation returns
 * SGEMM_ERR_INVALID_VALUE and touches nothing. SGEMM_ERR_ALLOC if the workspace cannot grow.
 */
int sgemm_run(sgemm_handle_t h, int M, int N, int K,
              float alpha, const float *A, int lda,
              const float *B, int ldb,
              float beta, float *C, int ldc,
              struct CUstream_st *stream);

/*
 * Same operation with HOST operands: copies A, B (and C when beta != 0) to
 * handle-owned device buffers, computes C there and copies it back, then
 * synchronizes `stream` before returning. Large problems are pipelined over
 * row panels of A and C (the first panel also over column blocks of B, in
 * which B is copied in), each panel or block one device GEMM on `stream`
 * while the next one's copy-in and the previous one's copy-out run on the
 * handle's own copy streams; the panels depend only on M, N, K and the SM
 * count, so results are reproducible and satisfy the sgemm_run bound. Pinned
 * (page-locked) host memory gives asynchronous, full-bandwidth copies;
 * pageable memory also works. Same argument rules as sgemm_run (pointers are
 * host pointers).
 */
int sgemm_run_host(sgemm_handle_t h, int M, int N, int K,
                   float alpha, const float *A, int lda,
                   const float *B, int ldb,
                   float beta, float *C, int ldc,
                   struct CUstream_st *stream);

/*
 * Split-K SGEMM that allocates no device memory. The pages have no
 * counterpart to this call; it exists for callers that cannot call cudaMalloc:
 * code running inside another runtime's memory pool, which must not grow
 * device memory behind that pool's back, and latency-sensitive loops that
 * cannot afford the device-wide synchronization cudaMalloc / cudaFree imply.
 *
 * Computes the same C = alpha * A * B + beta * C as sgemm_run (same argument
 * rules, DEVICE pointers, asynchronous on `stream`), always with the split-K
 * kernels: `splits` in 1..16 K slices (clamped to ceil(K / 32)) whose partial
 * sums go to a static scratch array, then a reduction in slice order. No
 * handle is needed.
 *
 * Scratch: a file-scope static device array of SGEMM_STATIC_SCRATCH_BYTES
 * (32 MiB), held by every GPU that loads this library until process exit.
 * It must fit splits * M * roundup(N, 4) floats of partials, plus aligned
 * copies of A (M * roundup(K, 4)) and/or B (K * roundup(N, 4)) when an operand
 * is not 16-byte aligned or its leading dimension is not a multiple of 4;
 * otherwise the call returns SGEMM_ERR_NOT_SUPPORTED and launches nothing.
 * All calls on a device share the array and it keeps the last call's
 * contents: calls that overlap on the GPU (e.g. on two unordered streams)
 * race on it, and, when they pass no status word, on the internal one too.
 *
 * device_status: optional caller-owned DEVICE int (4-byte aligned, checked
 * with the operands before anything else). Every call that returns SGEMM_OK
 * sets it to 0 on `stream` before its kernels (quick returns included); a
 * bounded wait that runs out in a kernel then writes
 * (SGEMM_ERR_TIMEOUT << 16) | location into it, and C may be partly written.
 * Read it after synchronizing `stream`. A call that returns an error enqueues
 * nothing and leaves the word as it was. With NULL the kernels write into an
 * internal static word that no call reads back, so a timeout code is lost:
 * callers that need to know pass their own word.
 *
 * The first call on a device performs a one-time set-up with that device
 * current (looks up the array's device address, sets kernel attributes);
 * make that first call before any stream capture.
 */
#define SGEMM_STATIC_SCRATCH_BYTES (32u << 20)
int sgemm_run_splitk_static(int M, int N, int K,
                            float alpha, const float *A, int lda,
                            const float *B, int ldb,
                            float beta, float *C, int ldc,
                            int splits, int *device_status,
                            struct CUstream_st *stream);

/*
 * sgemm_run, then the two smallest elements of the resulting C and their
 * positions ("SGEMM CUDA kernel (First Half)", Additionally Required: the two
 * minimums of the product C and their 2D indices, found in parallel).
 * Elements are ordered by (value, row-major position i * N + j): equal values
 * rank by position, so the answer is unique; NaN ranks as +infinity.
 * min_vals: DEVICE array of 2 floats (smallest first). min_ij: DEVICE array of
 * 4 ints {row0, col0, row1, col1}. Missing entries (M * N < 2) are +inf with
 * row = col = -1. Asynchronous on `stream` like sgemm_run; same argument rules,
 * plus min_vals and min_ij must be non-NULL.
 */
int sgemm_run_min2(sgemm_handle_t h, int M, int N, int K,
                   float alpha, const float *A, int lda,
                   const float *B, int ldb,
                   float beta, float *C, int ldc,
                   float *min_vals, int *min_ij,
                   struct CUstream_st *stream);

/* Select SGEMM_MATH_FP32 (default) or SGEMM_MATH_TF32 for later runs. */
int sgemm_set_math_mode(sgemm_handle_t h, int mode);
int sgemm_get_math_mode(sgemm_handle_t h, int *mode);

/* Set a tuning/test option (sgemm_option_t). Unknown options or values:
 * SGEMM_ERR_INVALID_VALUE. */
int sgemm_set_option(sgemm_handle_t h, int option, long long value);

/*
 * Synchronize `stream`, then read and clear the handle's device status word.
 * device_status (may be NULL) receives 0 when no kernel reported a problem,
 * else a code whose upper 16 bits are an sgemm_status value (SGEMM_ERR_TIMEOUT,
 * or SGEMM_ERR_NOT_SUPPORTED for a TF32 CTA pair whose shared-memory layouts
 * disagree) and whose lower bits say where: 1 a compute warp's wait for a filled
 * stage, 2 the copy warp's wait for a free stage, 3 the wait for a CTA's own
 * copies and MMAs in flight at its end, 4 the TF32 MMA issuer's wait for a
 * filled stage, 5 a wait on a TF32 accumulator, 7 the TF32 pair layout check,
 * 8 a wait on the FP32 epilogue's staging tile, 9 the FP32 transposer
 * warp's wait for a filled stage or a free M-major A buffer, 10 (with
 * SGEMM_ERR_NOT_SUPPORTED) a split-K cluster launched in another shape than
 * planned or with CTAs whose shared memory is laid out differently, in which
 * case nothing is computed (6 is not used). Debug builds of the library
 * (compiled with SGEMM_DEBUG_CHECKS=1, `python -m dense_fp32_gemm_04_gb300._build
 * --debug`, loaded when SGEMM_GB300_DEBUG_CHECKS=1) check the indices of their
 * accesses and report a failed check as SGEMM_ERR_INDEX with the location: 20 a
 * TMA tile coordinate outside the problem's tiles or k-blocks, 21 the
 * transposer warp's shared-memory offsets, 22 a compute warp's ring stage or
 * M-major buffer, 23 the staging tile, 24 a store to C outside M x N, 25 a
 * split-K slice outside the workspace, 26 a stream-K partial tile outside the
 * workspace, 27 the epilogue warps' staging reads, 28 a distributed shared
 * memory read of split-K within clusters, 29 the stream-K reduction's partial
 * reads, 30 the split-K reduction's slice reads, 33 a TF32 TMA coordinate, 34 a
 * TF32 store to C or to a partial tile. Returns that
 * sgemm_status value, or SGEMM_ERR_CUDA if synchronizing failed (e.g. a sticky
 * device error).
 */
int sgemm_check_device_status(sgemm_handle_t h, struct CUstream_st *stream, int *device_status);

/*
 * Host-only planning: what sgemm_run would launch for this problem on a GPU
 * with `num_sms` SMs. align_flags: bit 0 = A is 16-byte aligned, bit 1 = B,
 * bit 2 = C. Validates like sgemm_run (pointers are not checked here).
 * Needs no GPU.
 */
int sgemm_plan(int M, int N, int K, int lda, int ldb, int ldc, int align_flags,
               int num_sms, int math_mode, sgemm_plan_t *out);

/* The plan used by the handle's most recent sgemm_run / sgemm_run_host. */
int sgemm_last_plan(sgemm_handle_t h, sgemm_plan_t *out);

/*
 * Grow the handle's device workspace to at least workspace_bytes now (e.g. the
 * workspace_bytes of sgemm_plan for the problems to come). Growing synchronizes
 * the device. SGEMM_ERR_ALLOC if the memory cannot be had.
 *
 * CUDA graphs: sgemm_run and sgemm_run_min2 may be captured into a CUDA graph
 * (stream capture) once the workspace holds their plan's workspace_bytes (this
 * call, or an earlier uncaptured run of a problem at least as large): they then
 * only launch kernels and encode tensor maps on the host. A captured call whose
 * workspace would have to grow returns SGEMM_ERR_NOT_SUPPORTED and calls
 * nothing on the stream. sgemm_run_host synchronizes and cannot be captured.
 * Graph replays reuse the workspace: replays of graphs holding calls of one
 * handle must not overlap.
 */
int sgemm_reserve(sgemm_handle_t h, long long workspace_bytes);

/* Number of rows in the tile-config table, and row `index` (as a plan whose
 * problem-dependent fields are zero). Needs no GPU. */
int sgemm_config_count(void);
int sgemm_config_info(int index, sgemm_plan_t *out);

/* Static description of a status code. Never NULL. */
const char *sgemm_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* SGEMM_GB300_H */
