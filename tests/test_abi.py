"""The C ABI library loads, exports every function include/sgemm.h declares, and plans on the host."""

import ctypes
import os
import re

import pytest

import dense_fp32_gemm_04_gb300 as sg

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")


def declared_functions():
    text = "".join(open(os.path.join(INCLUDE, f)).read() for f in sorted(os.listdir(INCLUDE)) if f.endswith(".h"))
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?(?:int|char|void)\s*\*?\s*(sgemm_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_core_calls():
    names = declared_functions()
    for n in ("sgemm_create", "sgemm_run", "sgemm_destroy", "sgemm_set_math_mode", "sgemm_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    # and the binding covers them all
    assert set(declared_functions()) <= set(sg._SIGNATURES)


def test_status_strings(lib):
    for st in range(8):
        s = sg.status_string(st)
        assert s and "unknown" not in s
    assert "unknown" in sg.status_string(99)


def test_null_handle_is_rejected(lib):
    assert lib.sgemm_run(None, 4, 4, 4, 1.0, None, 4, None, 4, 0.0, None, 4, None) == sg.SGEMM_ERR_INVALID_VALUE
    assert lib.sgemm_set_option(None, sg.OPT_LOG, 1) == sg.SGEMM_ERR_INVALID_VALUE
    assert lib.sgemm_destroy(None) == sg.SGEMM_OK


def test_create_without_gpu_fails_cleanly(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    st = lib.sgemm_create(ctypes.byref(h))
    assert st in (sg.SGEMM_ERR_ARCH, sg.SGEMM_ERR_INVALID_VALUE) and not h.value


def test_misaligned_pointers_are_refused_on_the_host(lib):
    """An operand pointer that is not 4-byte aligned (a float's alignment) is refused
    with SGEMM_ERR_INVALID_VALUE before any CUDA call. On this GPU-less host the same
    call with aligned pointers passes that check and fails later (no device), which
    shows the check is what refused the misaligned ones. The pointers are never
    dereferenced on the host."""
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: the aligned fake pointers would reach a launch")
    good, bad = 0x100000, 0x100002
    args = lambda a, b, c, st: (4, 4, 4, 1.0, a, 4, b, 4, 0.0, c, 4, 1, st, None)
    for ptrs in ((bad, good, good, None), (good, bad, good, None), (good, good, bad, None), (good, good, good, bad)):
        assert lib.sgemm_run_splitk_static(*args(*ptrs)) == sg.SGEMM_ERR_INVALID_VALUE, ptrs
    assert lib.sgemm_run_splitk_static(*args(good, good, good, None)) == sg.SGEMM_ERR_CUDA
    for ptrs in ((bad, good, good), (good, bad, good), (good, good, bad)):
        assert lib.sgemm_ladder_run(1, 4, 4, 4, 1.0, ptrs[0], ptrs[1], 0.0, ptrs[2], None) == sg.SGEMM_ERR_INVALID_VALUE
    assert lib.sgemm_ladder_run(1, 4, 4, 4, 1.0, good, good, 0.0, good, None) != sg.SGEMM_ERR_INVALID_VALUE


@pytest.mark.parametrize("args", [
    (-1, 4, 4, 4, 4, 4), (4, -1, 4, 4, 4, 4), (4, 4, -1, 4, 4, 4),
    (4, 4, 8, 7, 4, 4),   # lda < K
    (4, 8, 4, 4, 7, 8),   # ldb < N
    (4, 8, 4, 4, 8, 7),   # ldc < N
    (4, 4, 0, 0, 4, 4),   # lda < max(1, K)
])
def test_plan_rejects_bad_dimensions(lib, args):
    M, N, K, lda, ldb, ldc = args
    p = sg.Plan()
    assert lib.sgemm_plan(M, N, K, lda, ldb, ldc, 7, 152, 0, ctypes.byref(p)) == sg.SGEMM_ERR_INVALID_VALUE


def test_plan_quick_returns(lib):
    assert sg.plan(0, 5, 5).kernel == sg.KERNEL_NONE
    assert sg.plan(5, 0, 5).kernel == sg.KERNEL_NONE
    p = sg.plan(5, 5, 0)
    assert p.kernel == sg.KERNEL_NONE  # sgemm_plan assumes beta == 1 for the K == 0 case
    assert p.launches == 0


def test_plan_square_4096(lib):
    p = sg.plan(4096, 4096, 4096, num_sms=152)
    assert p.kernel == sg.KERNEL_FFMA and p.splits == 1
    assert p.repack_a == 0 and p.repack_b == 0 and p.vec_c == 1
    assert p.grid <= 152 * p.ctas_per_sm
    # 1024 tiles on 152 CTAs: 6 whole rounds, then the 112 remaining tiles form
    # one stream-K span of 112 * 128 k-blocks shared evenly by every CTA
    tiles = p.tiles_m * p.tiles_n
    slots = 152 * p.ctas_per_sm
    assert p.sk_tiles == tiles - (tiles // slots) * slots == 112
    assert p.units == tiles - p.sk_tiles == 912 and p.grid == 152
    # A is transposed first (A^T mainloop): transpose + mainloop + stream-K reduction
    assert p.transpose_a == 1 and p.launches == 3
    assert p.workspace_bytes >= 2 * 152 * p.bm * p.bn * 4 + 4096 * 4096 * 4


def test_plan_full_rounds_have_no_tail(lib):
    # 8192^3: 4096 tiles -> 26.9 rounds, the last one 94 % full: not worth splitting
    p = sg.plan(8192, 8192, 8192, num_sms=152)
    assert p.sk_tiles == 0 and p.units == p.tiles_m * p.tiles_n
    assert p.transpose_a == 1 and p.launches == 2


def test_plan_ragged_unaligned_repacks(lib):
    # ld = 1531 / 3001 floats are not multiples of 4: rows are not 16-byte aligned.
    # A is transposed into the workspace (which aligns it too), B goes through the
    # aligned workspace copy, and C is accessed with scalar loads and stores.
    p = sg.plan(2047, 3001, 1531, lda=1531, ldb=3001, ldc=3001)
    assert p.transpose_a == 1 and p.repack_a == 0 and p.repack_b == 1 and p.vec_c == 0
    # A^T and the copy of B in one launch, the mainloop, [the reduction]
    assert p.launches == 2 + (1 if (p.splits > 1 or p.sk_tiles > 0) else 0)
    assert p.workspace_bytes >= 4 * (1531 * 2048 + 1531 * 3004)
    # Without the global transposition (small N) an unaligned A is repacked and then
    # transposed slab by slab in shared memory.
    q = sg.plan(20000, 16, 1531, lda=1531, ldb=16, ldc=16)
    assert q.transpose_a == 2 and q.repack_a == 1 and q.repack_b == 0
    assert q.launches == 2 + (1 if (q.splits > 1 or q.sk_tiles > 0) else 0)


def test_plan_misaligned_pointer_repacks(lib):
    p = sg.plan(512, 512, 512, align_flags=0b110)
    assert p.transpose_a == 2 and p.repack_a == 1 and p.repack_b == 0


def test_plan_skinny_shares_k(lib):
    for M, N in ((16384, 64), (64, 16384)):
        p = sg.plan(M, N, 8192, num_sms=152)
        assert p.kernel == sg.KERNEL_FFMA
        # fewer tiles than CTAs: K is shared, by split-K or by one stream-K span
        tiles = p.tiles_m * p.tiles_n
        if p.sk_tiles:
            assert p.splits == 1 and p.sk_tiles == tiles and p.units == 0 and p.grid == 152 * p.ctas_per_sm
            assert p.workspace_bytes >= 2 * p.grid * p.bm * p.bn * 4
        else:
            assert p.splits > 1 and p.units >= 152, p.as_dict()
            assert p.workspace_bytes >= p.splits * M * N * 4
        # transposing a 16384 x 8192 A in global memory costs more than it saves (it is
        # transposed slab by slab in shared memory instead); a 64 x 8192 A is cheap
        assert p.transpose_a == (1 if M == 64 else 2)
        if p.transpose_a == 2:
            # one more warp (the transposer) and a shorter ring beside the M-major A buffers
            row = sg.configs()[p.config]
            assert p.threads == row.threads + 32 and 2 <= p.stages < row.stages


def test_config_table(lib):
    rows = sg.configs()
    assert len(rows) >= 1
    for r in rows:
        assert r.bm % 32 == 0 and r.bn % 64 == 0 and r.bk == 32
        # warp tiles + the TMA producer warp (+ the 2 epilogue warps of the 128 x 128 row)
        assert r.threads == ((r.bm // 32) * (r.bn // 64) + 1 + (2 if (r.bm, r.bn) == (128, 128) else 0)) * 32



def test_plan_invariants_random_shapes(lib):
    """Host planner invariants over many seeded random problems and SM counts."""
    import numpy as np

    rng = np.random.default_rng(1234)
    for _ in range(400):
        M, N, K = (int(x) for x in rng.integers(1, 20000, 3))
        if rng.random() < 0.3:
            M = int(rng.integers(1, 300))
        if rng.random() < 0.3:
            N = int(rng.integers(1, 300))
        sms = int(rng.choice([1, 8, 132, 148, 152, 160]))
        lda, ldb, ldc = K + int(rng.integers(0, 5)), N + int(rng.integers(0, 5)), N + int(rng.integers(0, 5))
        align = int(rng.integers(0, 8))
        p = sg.plan(M, N, K, lda=lda, ldb=ldb, ldc=ldc, align_flags=align, num_sms=sms)
        assert p.kernel == sg.KERNEL_FFMA
        tiles = p.tiles_m * p.tiles_n
        assert p.tiles_m == -(-M // p.bm) and p.tiles_n == -(-N // p.bn)
        kb = -(-K // 32)
        assert 1 <= p.splits <= min(kb, 16)
        slots = sms * p.ctas_per_sm
        if p.sk_tiles > 0:
            assert p.splits == 1 and 0 < p.sk_tiles < slots
            assert p.units == tiles - p.sk_tiles and p.units % slots == 0
            assert p.grid == (slots if p.units > 0 else min(slots, p.sk_tiles * kb))
            assert p.sk_grid == min(slots, p.sk_tiles * kb) <= p.grid
            assert p.workspace_bytes >= 2 * p.grid * p.bm * p.bn * 4
        else:
            assert p.units == tiles * p.splits
            if p.splits > 1 and not p.cluster_split:
                assert p.workspace_bytes >= p.splits * M * (-(-N // 4) * 4) * 4
        if p.cluster_split:
            # split-K within clusters: one CTA per (tile, slice), no partials in the workspace
            assert 2 <= p.splits <= 8 and p.sk_tiles == 0 and p.grid == p.units
        else:
            assert 1 <= p.grid <= (slots if p.sk_tiles else min(p.units, slots))
        assert p.transpose_a in (1, 2)  # A as given (0) only when forced
        assert p.repack_a == (0 if (p.transpose_a == 1 or (align & 1 and lda % 4 == 0)) else 1)
        assert p.repack_b == (0 if (align & 2 and ldb % 4 == 0) else 1)
        assert p.vec_c == (1 if (align & 4 and ldc % 4 == 0) else 0)
        if p.transpose_a == 1:
            assert p.workspace_bytes >= K * (-(-M // 4) * 4) * 4
        extra = 1 if ((p.splits > 1 and not p.cluster_split) or p.sk_tiles > 0) else 0
        # both operand copies go in one launch
        assert p.launches == 1 + int(p.transpose_a == 1 or p.repack_a or p.repack_b) + extra


def test_tf32_plan(lib):
    p = sg.plan(4096, 4096, 4096, math_mode=sg.MATH_TF32)
    # CTA pairs: 256 x 256 tiles, 76 pairs on 152 SMs
    assert p.kernel == sg.KERNEL_TF32 and p.config == 1 and (p.bm, p.bn, p.bk) == (256, 256, 32)
    # A read K-major and B MN-major as stored: no operand copy
    assert p.repack_a == 0 and p.repack_b == 0 and p.grid == 152 and p.transpose_a == 0
    # 256 tiles on 76 pairs: 3 whole rounds, then the 28 remaining tiles as a stream-K span
    assert p.units == 228 and p.sk_tiles == 28
    assert p.sk_grid == 56  # 2 equal K slices per span tile, one per pair
    assert p.launches == 2  # mainloop, stream-K reduction
    assert p.workspace_bytes == 2 * 56 * 256 * 256 * 4
    # an unaligned B (ldb not a multiple of 4) is repacked first
    p = sg.plan(4096, 4095, 4096, ldb=4095, ldc=4096, math_mode=sg.MATH_TF32)
    assert p.repack_b == 1 and p.launches == 2 + (1 if p.sk_tiles else 0)
    # an odd SM count: pairs = floor(SMs / 2), the grid is whole pairs
    p = sg.plan(4096, 4096, 4096, num_sms=151, math_mode=sg.MATH_TF32)
    assert p.config == 1 and p.grid == 150
    # C not 16-byte accessible (ldc not a multiple of 4): written in place, no copy of C
    p = sg.plan(2047, 3001, 1531, math_mode=sg.MATH_TF32)
    assert p.vec_c == 0 and p.repack_c == 0 and p.repack_a == 1 and p.repack_b == 1
    assert p.launches == 2 + (1 if p.sk_tiles else 0)  # both copies in one launch
    # at any size, and for an unaligned C base (align bit 2 clear) as well
    for (M, N, K, ldc, align) in [(8191, 8191, 512, 8191, 7), (4096, 4096, 4096, 4096, 3), (300, 301, 64, 301, 7),
                                  (4095, 4093, 4096, 4093, 7)]:
        p = sg.plan(M, N, K, ldc=ldc, align_flags=align, math_mode=sg.MATH_TF32)
        assert p.vec_c == 0 and p.repack_c == 0, (M, N, K, ldc, align)
        assert p.launches == int(p.repack_a or p.repack_b) + 1 + (1 if p.sk_tiles else 0)


def test_tf32_single_cta_plan(lib):
    # 128 rows: half of every pair tile would be empty, one CTA per 128 x 256 tile wins
    p = sg.plan(128, 4096, 4096, math_mode=sg.MATH_TF32)
    assert p.kernel == sg.KERNEL_TF32 and p.config == 0 and (p.bm, p.bn, p.bk) == (128, 256, 32)
    assert p.tiles_m == 1 and p.tiles_n == 16
    assert p.units + p.sk_tiles == 16 and p.grid <= 152
    if p.sk_tiles:
        assert p.grid == p.sk_grid and p.workspace_bytes >= 2 * p.sk_grid * 128 * 256 * 4


def test_plan_rows_follow_the_measured_epilogue_costs(lib):
    """Row 0 (128 x 128) writes its tiles out through epilogue warps: that hides the
    write-out behind the next tile but costs a tiny tile a few microseconds, so the
    planner leaves the smallest problems to row 1 (measured on GB300: 256^3 12.3 us
    and 512^3 16.4 us on row 1 against 14.3 and 18.4 on row 0) and takes row 0 from
    1024^3 up (1024^3 50.2 us, ragged 2047 x 3001 x 1531 328 us against 349 on row 1)."""
    for n in (256, 512):  # (or split-K within clusters, which has no epilogue warps' write-out)
        p = sg.plan(n, n, n)
        assert p.config == 1 or p.cluster_split == 1
    for shape in [(1024, 1024, 1024), (2048, 2048, 2048), (4096, 4096, 4096), (8192, 8192, 8192),
                  (2047, 3001, 1531)]:
        assert sg.plan(*shape).config == 0, shape
    p = sg.plan(4096, 4096, 4096)
    assert p.threads == (8 + 1 + 2) * 32  # 8 compute warps, the TMA warp, 2 epilogue warps


def test_plan_small_problems_reduce_within_clusters(lib):
    """Small problems: the split-K CTAs of a tile form one cluster and add their
    partial tiles in distributed shared memory, so the call is one launch with no
    workspace; large ones keep the persistent grid."""
    for n in (256, 512):
        p = sg.plan(n, n, n, num_sms=152)
        assert p.cluster_split == 1 and 2 <= p.splits <= 8 and p.launches == 1 and p.workspace_bytes == 0
        assert p.grid == p.units == p.tiles_m * p.tiles_n * p.splits
    for shape in ((4096, 4096, 4096), (2047, 3001, 1531), (16384, 64, 8192)):
        assert sg.plan(*shape, num_sms=152).cluster_split == 0
