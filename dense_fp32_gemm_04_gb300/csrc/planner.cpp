// Host-only planning: argument validation, quick returns, alignment gates,
// tile-config and split-K choice, workspace sizing. No CUDA calls here, so
// sgemm_plan() works on a machine without a GPU.
#include "planner.h"

#include <algorithm>
#include <climits>
#include <cmath>

namespace sgemm_impl {

namespace {

long long round_up(long long x, long long m) { return (x + m - 1) / m * m; }
long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

// One work unit of kb_unit k-blocks on a CTA: the k-blocks plus the pipeline
// fill and the epilogue, ~1.5 k-blocks. With epilogue warps the write-out of a
// tile overlaps the next unit (~0.5 k-blocks left), but a unit then takes at
// least as long as the epilogue warps need to write a tile out (measured at
// 4096^2 x 32: the fitted 4 us raw or with beta = 0, 8 us reading C, pick
// the faster row at 256^3 .. 1024^3 and the ragged shapes), and the kernel
// ends with one such write-out (epilogue_tail).
double epilogue_drain(const sgemm_cfg::TileConfig &c, bool reads_c)
{
    return c.epilogue_warps > 0 ? (reads_c ? 8.0e-6 : 4.0e-6) : 0.0;
}

double unit_time(const sgemm_cfg::TileConfig &c, double kb_unit, double t_kb, bool reads_c)
{
    if (c.epilogue_warps == 0) return (kb_unit + 1.5) * t_kb;
    return std::max((kb_unit + 0.5) * t_kb, epilogue_drain(c, reads_c));
}

// Modelled time (seconds) of one FFMA configuration with S splits. Per CTA a
// 32-deep k-block of a BM x BN tile costs BM*BN*32 FMAs at the SM's FP32 rate
// shared by the CTAs resident on it; a persistent CTA runs ceil(units/slots)
// units one after another; split-K adds the partial write + reduce traffic.
double model_time(const sgemm_cfg::TileConfig &c, int M, int N, int K, int S, int num_sms, bool beta_read)
{
    const double fma_per_sm = 128.0 * 1.9e9 * 0.88;  // FMA/s per SM, at the measured achieved fraction
    const double hbm = 5.5e12;                        // B/s achieved by the elementwise kernels
    const long long kb = ceil_div(K, sgemm_cfg::kFfmaBK);
    const long long tiles = ceil_div(M, c.bm) * ceil_div(N, c.bn);
    const long long units = tiles * S;
    const long long slots = static_cast<long long>(num_sms) * c.ctas_per_sm;
    const long long per_cta = ceil_div(units, slots);
    const double kb_per_unit = static_cast<double>(ceil_div(kb, S));
    const double t_kb = static_cast<double>(c.bm) * c.bn * sgemm_cfg::kFfmaBK * c.ctas_per_sm / fma_per_sm * c.rel_cost;
    const bool reads_c = beta_read && S == 1;  // split slices are written raw
    double t = static_cast<double>(per_cta) * unit_time(c, kb_per_unit, t_kb, reads_c) +
               epilogue_drain(c, reads_c) + 2.0e-6;
    if (S > 1) {
        const double bytes = (2.0 * S + (beta_read ? 2.0 : 1.0)) * 4.0 * M * static_cast<double>(N);
        t += bytes / hbm + 2.5e-6;
    }
    return t;
}

// Stream-K: the first (R - 1) rounds of `slots` whole tiles run data-parallel;
// the `rem` tiles of the last, partial round become one span of rem * kb
// k-blocks cut evenly over the slots CTAs (each CTA then has at most two partial
// tiles, reduced afterwards). Modelled time, or infinity when the last round is
// full (nothing to balance).
double model_time_sk(const sgemm_cfg::TileConfig &c, int M, int N, int K, int num_sms, bool beta_read)
{
    const double fma_per_sm = 128.0 * 1.9e9 * 0.88;
    const double hbm = 5.5e12;
    const long long kb = ceil_div(K, sgemm_cfg::kFfmaBK);
    const long long tiles = ceil_div(M, c.bm) * ceil_div(N, c.bn);
    const long long slots = static_cast<long long>(num_sms) * c.ctas_per_sm;
    const long long rounds = ceil_div(tiles, slots);
    const long long rem = tiles - (rounds - 1) * slots;
    if (rem >= slots) return INFINITY;
    const long long span = rem * kb;
    const long long G = std::min(slots, span);
    const double t_kb = static_cast<double>(c.bm) * c.bn * sgemm_cfg::kFfmaBK * c.ctas_per_sm / fma_per_sm * c.rel_cost;
    // whole tiles, then the span pieces (up to two partial tiles, written raw)
    double t = static_cast<double>(rounds - 1) * unit_time(c, static_cast<double>(kb), t_kb, beta_read) +
               std::max((static_cast<double>(ceil_div(span, G)) + (c.epilogue_warps > 0 ? 2.0 : 3.0)) * t_kb,
                        2.0 * epilogue_drain(c, false)) +
               epilogue_drain(c, false) + 2.0e-6;
    // Partial tiles (written, then read by the reduction) mostly stay in L2: counted
    // at twice the HBM rate; C at the HBM rate.
    const double tile_bytes = 4.0 * c.bm * c.bn;
    const double part_bytes = 2.0 * static_cast<double>(G + rem) * tile_bytes;
    const double c_bytes = (beta_read ? 2.0 : 1.0) * static_cast<double>(rem) * tile_bytes;
    return t + part_bytes / (2.0 * hbm) + c_bytes / hbm + 2.5e-6;
}

// Transposing A first pays when its copy (read + write of A, one more launch)
// costs less than the ~10 % the A^T mainloop saves (measured 9-10 % at
// 2048^3 .. 8192^3; kAtGain keeps a margin). The launch costs ~1.5 us: the
// mainloop is a programmatic dependent of the transposition, so its own launch
// overlaps it (1024^3: A^T 45.2 against 47.1 us as given).
bool transpose_pays(const Problem &q, double t_main)
{
    constexpr double kAtGain = 0.07;
    const double hbm = 5.5e12;
    const double t_copy = 8.0 * static_cast<double>(q.M) * q.K / hbm + 1.5e-6;
    return t_copy < kAtGain * t_main;
}

// TF32 mode, one kernel (one CTA per 128 x 256 tile on `slots` SMs, or one CTA
// pair per 256 x 256 tile on `slots` pairs): modelled time of the persistent
// grid, and the stream-K slicing of its last partial round. The span's rem tiles
// go to rem * St workers in equal K slices, so that every worker's range is
// slice s of one tile (k-blocks [s kb / St, (s + 1) kb / St)) and each writes
// one partial tile; St <= 8 with at least one 32-deep block per slice, taken
// when the modelled time saved exceeds the partial-tile reduction by 1 % of the
// call. (A span spread over all workers, as on the FP32 path, gives two partials
// per worker: the TF32 epilogue writes those slower than it saves, 4096^3 219 ->
// 237 us with one CTA per tile.) Rates: FLOP/s per worker as measured for each
// kernel; C at ~5.5 TB/s, the partial tiles (written, then read back within
// microseconds, mostly from L2) at twice that.
struct Tf32Model {
    double time;
    int slices;  // St, 0 = no stream-K
};

Tf32Model model_tf32(int M, int N, int K, int bm, int bn, long long slots, double flops_per_worker, bool beta_read)
{
    const double hbm = 5.5e12;
    const long long kb = ceil_div(K, sgemm_cfg::kTf32BK);
    const long long tiles = ceil_div(M, bm) * ceil_div(N, bn);
    const long long rounds = ceil_div(tiles, slots);
    const long long rem = tiles - (rounds - 1) * slots;
    const double tile_elems = static_cast<double>(bm) * bn;
    const double t_kb = tile_elems * sgemm_cfg::kTf32BK * 2.0 / flops_per_worker;
    const double t_last = (static_cast<double>(kb) + 1.5) * t_kb;
    const double base = static_cast<double>(rounds) * t_last + 2.0e-6;
    if (rem >= slots) return {base, 0};
    double best_gain = 0.01 * base;
    int best = 0;
    for (int st = 2; st <= 8 && st <= kb && rem * st <= slots; ++st) {
        const double t_span_round = (static_cast<double>(ceil_div(kb, st)) + 1.5) * t_kb;
        const double part_bytes = 2.0 * st * 4.0 * static_cast<double>(rem) * tile_elems;
        const double c_bytes = (beta_read ? 2.0 : 1.0) * 4.0 * static_cast<double>(rem) * tile_elems;
        const double gain = t_last - t_span_round - part_bytes / (2.0 * hbm) - c_bytes / hbm - 2.5e-6;
        if (gain > best_gain) {
            best_gain = gain;
            best = st;
        }
    }
    return {best > 0 ? base - best_gain : base, best};
}

// Measured mainloop rates (GB300, 6144^3 and 8192^3 without stream-K): one CTA
// per tile ~660 TFLOP/s on 152 SMs; a CTA pair does 1.33-1.34x the work of two
// SMs of the one-CTA kernel (a third less shared-memory traffic per FMA).
constexpr double kTf32FlopsPerSm = 650e12 / 152.0;
constexpr double kTf32PairGain = 1.33;

}  // namespace

int validate(const Problem &q)
{
    if (q.M < 0 || q.N < 0 || q.K < 0) return SGEMM_ERR_INVALID_VALUE;
    if (q.lda < std::max(1, q.K) || q.ldb < std::max(1, q.N) || q.ldc < std::max(1, q.N))
        return SGEMM_ERR_INVALID_VALUE;
    if (q.num_sms <= 0) return SGEMM_ERR_INVALID_VALUE;
    if (q.math_mode != SGEMM_MATH_FP32 && q.math_mode != SGEMM_MATH_TF32) return SGEMM_ERR_INVALID_VALUE;
    return SGEMM_OK;
}

void config_as_plan(int index, sgemm_plan_t *out)
{
    *out = sgemm_plan_t{};
    const sgemm_cfg::TileConfig &c = sgemm_cfg::kFfmaConfigs[index];
    out->kernel = SGEMM_KERNEL_FFMA;
    out->config = index;
    out->bm = c.bm;
    out->bn = c.bn;
    out->bk = c.bk;
    out->stages = c.stages;
    out->threads = c.threads;
    out->ctas_per_sm = c.ctas_per_sm;
    out->splits = 1;
}

int choose_ffma(int M, int N, int K, int num_sms, bool beta_read, int force_config, int force_splits,
                int *config, int *splits)
{
    const int kb = static_cast<int>(ceil_div(K, sgemm_cfg::kFfmaBK));
    const int max_s = std::max(1, std::min(kb, kMaxSplits));
    if (force_config >= sgemm_cfg::kNumFfmaConfigs) return SGEMM_ERR_INVALID_VALUE;
    if (force_splits < 0) return SGEMM_ERR_INVALID_VALUE;
    double best = INFINITY;
    int best_c = 0, best_s = 1;
    for (int ci = 0; ci < sgemm_cfg::kNumFfmaConfigs; ++ci) {
        if (force_config >= 0 && ci != force_config) continue;
        const int s_lo = force_splits > 0 ? std::min(force_splits, max_s) : 1;
        const int s_hi = force_splits > 0 ? s_lo : max_s;
        for (int s = s_lo; s <= s_hi; ++s) {
            const double t = model_time(sgemm_cfg::kFfmaConfigs[ci], M, N, K, s, num_sms, beta_read);
            // Prefer earlier rows and fewer splits unless clearly faster (2 %).
            if (t < best * 0.98) {
                best = t;
                best_c = ci;
                best_s = s;
            }
        }
    }
    *config = best_c;
    *splits = best_s;
    return SGEMM_OK;
}

int make_plan(const Problem &q, const Overrides &ov, sgemm_plan_t *out)
{
    const int v = validate(q);
    if (v != SGEMM_OK) return v;
    *out = sgemm_plan_t{};
    out->config = -1;
    out->math_mode = q.math_mode;
    out->splits = 1;
    if (q.M == 0 || q.N == 0) {
        out->kernel = SGEMM_KERNEL_NONE;
        return SGEMM_OK;
    }
    if (q.K == 0 || q.alpha == 0.0f) {
        if (q.beta == 1.0f) {
            out->kernel = SGEMM_KERNEL_NONE;
        } else {
            out->kernel = SGEMM_KERNEL_SCALE;
            out->launches = 1;
        }
        return SGEMM_OK;
    }
    const bool a_ok = (q.align_flags & 1) && q.lda % 4 == 0;
    const bool b_ok = (q.align_flags & 2) && q.ldb % 4 == 0;
    out->repack_a = a_ok ? 0 : 1;
    out->repack_b = b_ok ? 0 : 1;
    out->vec_c = ((q.align_flags & 4) && q.ldc % 4 == 0) ? 1 : 0;
    if (q.math_mode == SGEMM_MATH_TF32) {
        // A is read K-major and B MN-major as stored (repacked only when not 16-byte aligned).
        const long long pairs = q.num_pairs > 0 ? q.num_pairs : (q.num_pairs == 0 ? q.num_sms / 2 : 0);
        const bool beta_read = q.beta != 0.0f;
        const Tf32Model one = model_tf32(q.M, q.N, q.K, sgemm_cfg::kTf32BM, sgemm_cfg::kTf32BN, q.num_sms,
                                         kTf32FlopsPerSm, beta_read);
        Tf32Model two{INFINITY, 0};
        if (pairs > 0)
            two = model_tf32(q.M, q.N, q.K, sgemm_cfg::kTf32PairBM, sgemm_cfg::kTf32PairBN, pairs,
                             2.0 * kTf32FlopsPerSm * kTf32PairGain, beta_read);
        bool use_pair = two.time < one.time;
        if (ov.force_tf32_kernel == 0) use_pair = false;
        if (ov.force_tf32_kernel == 1) {
            if (pairs <= 0) return SGEMM_ERR_NOT_SUPPORTED;
            use_pair = true;
        }
        const Tf32Model &m = use_pair ? two : one;
        const long long slots = use_pair ? pairs : q.num_sms;  // workers
        const int cluster = use_pair ? 2 : 1;                  // CTAs per worker
        out->kernel = SGEMM_KERNEL_TF32;
        out->config = use_pair ? 1 : 0;
        out->bm = use_pair ? sgemm_cfg::kTf32PairBM : sgemm_cfg::kTf32BM;
        out->bn = use_pair ? sgemm_cfg::kTf32PairBN : sgemm_cfg::kTf32BN;
        out->bk = sgemm_cfg::kTf32BK;
        out->stages = use_pair ? sgemm_cfg::kTf32PairStages : sgemm_cfg::kTf32Stages;
        out->threads = sgemm_cfg::kTf32Threads;
        out->ctas_per_sm = 1;
        out->splits = 1;
        out->tiles_m = static_cast<int>(ceil_div(q.M, out->bm));
        out->tiles_n = static_cast<int>(ceil_div(q.N, out->bn));
        const long long units = static_cast<long long>(out->tiles_m) * out->tiles_n;
        if (units > INT_MAX / 2) return SGEMM_ERR_NOT_SUPPORTED;
        out->units = static_cast<int>(units);
        out->grid = static_cast<int>(cluster * std::min<long long>(units, slots));
        if (ov.force_splits == 0 && ov.force_streamk != 0) {
            const long long n_full = (ceil_div(units, slots) - 1) * slots;
            const long long rem = units - n_full;
            const long long kb = ceil_div(q.K, sgemm_cfg::kTf32BK);
            long long st = m.slices;
            if (st < 2 && ov.force_streamk == 1 && rem < slots) st = std::min(kb, slots / rem);  // forced: fill idle workers
            st = std::min(st, slots / rem);  // one slice per worker: rem * st workers at most `slots`
            if (st >= 2 && rem < slots) {
                out->units = static_cast<int>(n_full);
                out->sk_tiles = static_cast<int>(rem);
                out->sk_grid = static_cast<int>(rem * st);
                out->grid = static_cast<int>(cluster * (n_full > 0 ? slots : std::min(slots, rem * st)));
            }
        }
        // C not 16-byte accessible: written in place (16-byte accesses inside each row,
        // the row ends element by element) unless forced through an aligned copy; the
        // copy measured slower at every size (ragged 2047 x 3001 x 1531: 87 vs 95 us).
        if (!out->vec_c && ov.force_repack_c == 1) out->repack_c = 1;
        out->workspace_bytes = workspace_layout(q, *out).total;
        // (both operand copies go in one launch)
        out->launches = (out->repack_a || out->repack_b ? 1 : 0) + 1 + (out->sk_tiles > 0 ? 1 : 0) +
                        (out->repack_c ? (q.beta != 0.0f ? 2 : 1) : 0);
        return SGEMM_OK;
    }

    int cfg = 0, S = 1;
    const int rc = choose_ffma(q.M, q.N, q.K, q.num_sms, q.beta != 0.0f, ov.force_config, ov.force_splits, &cfg, &S);
    if (rc != SGEMM_OK) return rc;
    const bool beta_read = q.beta != 0.0f;
    double t_plan = model_time(sgemm_cfg::kFfmaConfigs[cfg], q.M, q.N, q.K, S, q.num_sms, beta_read);
    const sgemm_cfg::TileConfig &c = sgemm_cfg::kFfmaConfigs[cfg];
    config_as_plan(cfg, out);
    out->math_mode = q.math_mode;
    out->repack_a = a_ok ? 0 : 1;
    out->repack_b = b_ok ? 0 : 1;
    out->vec_c = ((q.align_flags & 4) && q.ldc % 4 == 0) ? 1 : 0;
    out->splits = S;
    out->tiles_m = static_cast<int>(ceil_div(q.M, c.bm));
    out->tiles_n = static_cast<int>(ceil_div(q.N, c.bn));
    const long long units = static_cast<long long>(out->tiles_m) * out->tiles_n * S;
    if (units > INT_MAX) return SGEMM_ERR_NOT_SUPPORTED;
    out->units = static_cast<int>(units);
    out->grid = static_cast<int>(std::min<long long>(units, static_cast<long long>(q.num_sms) * c.ctas_per_sm));
    if (ov.force_splits == 0 && ov.force_streamk != 0) {
        // Stream-K on the chosen row when it beats the split-K plan (or is forced).
        const double t_sk = model_time_sk(c, q.M, q.N, q.K, q.num_sms, beta_read);
        const double t_dp = model_time(c, q.M, q.N, q.K, S, q.num_sms, beta_read);
        if (t_sk < INFINITY && (ov.force_streamk == 1 || t_sk < 0.99 * t_dp)) {
            const long long slots = static_cast<long long>(q.num_sms) * c.ctas_per_sm;
            const long long tiles = static_cast<long long>(out->tiles_m) * out->tiles_n;
            const long long n_full = (ceil_div(tiles, slots) - 1) * slots;
            const long long span = (tiles - n_full) * ceil_div(q.K, sgemm_cfg::kFfmaBK);
            out->splits = S = 1;
            out->units = static_cast<int>(n_full);
            out->sk_tiles = static_cast<int>(tiles - n_full);
            // every slot runs the whole tiles; the span needs at most one CTA per k-block
            out->grid = static_cast<int>(n_full > 0 ? slots : std::min(slots, span));
            out->sk_grid = static_cast<int>(std::min(slots, span));
            t_plan = t_sk;
        }
    }

    // Split-K reduced within clusters (no workspace, no reduction launch), on the
    // plan chosen above: forced onto any plan with 2..kMaxClusterSplits splits,
    // or automatically when all its CTAs fit in one wave and the clusters are of
    // CTAs that share SMs or are at most 4 wide. Measured on GB300 (back-to-back
    // calls): 256^3 13.5 -> 11.2 us, 300 x 200 x 100 13.7 -> 11.2 us, 512^3 equal;
    // 8-CTA clusters of the one-CTA-per-SM row and grids of several waves ran
    // slower (512^3 row 0 with 8 splits 19 -> 27 us; 768^3 rows 1-2 with 8 splits
    // 27 -> 33 us).
    // (the cluster form reads A transposed in shared memory: not with another A layout forced)
    const long long slots_c = static_cast<long long>(q.num_sms) * c.ctas_per_sm;
    const bool cl_fits = out->sk_tiles == 0 && S >= 2 && S <= kMaxClusterSplits &&
                         (ov.force_transpose_a < 0 || ov.force_transpose_a == 2);
    const bool cl = ov.cluster_split == 1 ? cl_fits
                    : ov.cluster_split < 0
                        ? cl_fits && out->units <= slots_c && (c.ctas_per_sm > 1 || S <= 4)
                        : false;
    if (cl) {
        // one (tile, slice) unit per CTA, clusters of S CTAs
        out->cluster_split = 1;
        out->grid = out->units;
    }

    // A layout. The mainloop's FFMA2 form with A pairs along M runs ~10 % faster
    // than the one A as given allows; it needs A M-major, either transposed in
    // global memory first (one read and one write of A) or turned M-major slab by
    // slab in shared memory by a transposer warp (no copy; a shorter ring).
    if (ov.force_transpose_a >= 0) {
        out->transpose_a = ov.force_transpose_a;
    } else {
        out->transpose_a = !cl && transpose_pays(q, t_plan) ? 1 : 2;
    }
    if (out->transpose_a == 1) out->repack_a = 0;  // the transposed copy is aligned whatever A was
    if (out->transpose_a == 2) {
        out->stages = c.xstages;
        out->threads = c.xthreads;
    }

    const Workspace w = workspace_layout(q, *out);
    out->workspace_bytes = w.total;
    // (both operand copies, A^T or A repacked and B repacked, go in one launch)
    out->launches = 1 + (out->transpose_a == 1 || out->repack_a || out->repack_b ? 1 : 0) +
                    ((S > 1 && !out->cluster_split) || out->sk_tiles > 0 ? 1 : 0);
    return SGEMM_OK;
}

Workspace workspace_layout(const Problem &q, const sgemm_plan_t &p)
{
    Workspace w{};
    long long off = 0;
    if (p.transpose_a == 1) {
        w.lda = round_up(q.M, 4);
        w.a_off = off;
        off += round_up(static_cast<long long>(q.K) * w.lda * 4, 256);
    } else if (p.repack_a) {
        w.lda = round_up(q.K, 4);
        w.a_off = off;
        off += round_up(static_cast<long long>(q.M) * w.lda * 4, 256);
    }
    if (p.repack_b) {
        w.ldb = round_up(q.N, 4);
        w.b_off = off;
        off += round_up(static_cast<long long>(q.K) * w.ldb * 4, 256);
    }
    if (p.repack_c) {
        w.ldc = round_up(q.N, 4);
        w.c_off = off;
        off += round_up(static_cast<long long>(q.M) * w.ldc * 4, 256);
    }
    if (p.sk_tiles > 0) {
        // two partial tiles per worker (CTA, or CTA pair) of the stream-K span
        w.w_off = off;
        off += round_up(2LL * p.sk_grid * p.bm * p.bn * 4, 256);
    } else if (p.splits > 1 && !p.cluster_split) {
        w.ldw = round_up(q.N, 4);
        w.wstride = static_cast<long long>(q.M) * w.ldw;
        w.w_off = off;
        off += round_up(static_cast<long long>(p.splits) * w.wstride * 4, 256);
    }
    w.total = off;
    return w;
}

}  // namespace sgemm_impl
