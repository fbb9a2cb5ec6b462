// Host-only planner interface (validation, tile-config / split-K choice,
// workspace layout). Used by the C ABI; needs no CUDA runtime.
#pragma once

#include "../../include/sgemm.h"
#include "tf32_tiles.h"
#include "tile_table.h"

namespace sgemm_impl {

constexpr int kMaxSplits = 16;
constexpr int kMaxClusterSplits = 8;  // portable cluster size

struct Problem {
    int M, N, K;
    int lda, ldb, ldc;
    int align_flags;  // bit 0: A 16-byte aligned, bit 1: B, bit 2: C
    int num_sms;
    int math_mode;
    float alpha, beta;
    int num_pairs = 0;  // TF32 CTA pairs resident at once (0: num_sms / 2; < 0: none)
};

struct Overrides {
    int force_config = -1;  // table row, -1 automatic
    int force_splits = 0;   // 0 automatic
    int force_transpose_a = -1;  // FFMA kernel, A layout: -1 automatic, 0 as given, 1 transposed in
                                 // global memory first, 2 transposed in shared memory
    int force_streamk = -1;      // -1 automatic, 0 never, 1 whenever the last round is partial
    int force_tf32_kernel = -1;  // -1 automatic, 0 one CTA per tile, 1 CTA pairs
    int force_repack_c = -1;     // TF32, C not 16-byte accessible: -1 automatic, 0 in place, 1 aligned copy
    int cluster_split = -1;      // FFMA split-K reduced within clusters: -1 automatic, 0 never,
                                 // 1 whenever the plan has 2..kMaxClusterSplits splits (and no stream-K)
};

// Offsets (bytes) into the handle's workspace and the strides used there.
struct Workspace {
    long long a_off = 0, lda = 0;       // repacked A (M x lda, plan.repack_a) or A^T (K x lda, plan.transpose_a)
    long long b_off = 0, ldb = 0;       // repacked B (K x ldb), when plan.repack_b
    long long w_off = 0, ldw = 0, wstride = 0;  // split-K or stream-K partials
    long long c_off = 0, ldc = 0;       // aligned copy of C (M x ldc), when plan.repack_c
    long long total = 0;
};

int validate(const Problem &q);
int make_plan(const Problem &q, const Overrides &ov, sgemm_plan_t *out);
Workspace workspace_layout(const Problem &q, const sgemm_plan_t &p);
void config_as_plan(int index, sgemm_plan_t *out);
int choose_ffma(int M, int N, int K, int num_sms, bool beta_read, int force_config, int force_splits,
                int *config, int *splits);


}  // namespace sgemm_impl
