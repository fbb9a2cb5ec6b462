"""GPU parity: the library (through its C ABI) against the FP64 oracle.

Bit-exact on integer-valued operands; within
(K + 2) * 2^-24 * (|alpha| sum |a||b| + |beta||c|) elementwise on real ones.
"""

import itertools

import numpy as np
import pytest

import dense_fp32_gemm_04_gb300 as sg
import oracle
from dense_fp32_gemm_04_gb300 import inputs
from gpu_helpers import check_against_oracle, problem_reference, run_gemm, sample_rows

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def h():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_fp32_gemm_04_gb300 import _build

    _build.build()
    handle = sg.Sgemm(0)
    yield handle
    handle.close()


def ops(M, N, K, seed, dist=("int", "int", "int")):
    return inputs.problem_operands(M=M, N=N, K=K, seed=seed, dist=dist)


def test_tiny_shapes_exact(h):
    """Every M, N, K in 1..9 with integer operands: bit-exact, guards intact."""
    for M, N, K in itertools.product(range(1, 10), repeat=3):
        A, B, C = ops(M, N, K, seed=M * 100 + N * 10 + K)
        got, guards, st = run_gemm(torch, h, A, B, C, 1.5, -0.5)
        assert st == sg.SGEMM_OK and guards, (M, N, K)
        check_against_oracle(got, A, B, C, 1.5, -0.5, exact=True)


def force(h, config=-1, splits=0, transpose_a=-1):
    h.set_option(sg.OPT_FORCE_CONFIG, config)
    h.set_option(sg.OPT_FORCE_SPLITS, splits)
    h.set_option(sg.OPT_FORCE_TRANSPOSE_A, transpose_a)


@pytest.mark.parametrize("cfg", range(4))
@pytest.mark.parametrize("splits", [1, 2, 3, 7])
@pytest.mark.parametrize("ta", [0, 1, 2])
def test_every_config_and_split(h, cfg, splits, ta):
    """Each tile-config row, split factor and A layout (as given / transposed first /
    transposed in shared memory), around tile multiples, integer and real operands."""
    force(h, cfg, splits, ta)
    try:
        for (M, N, K) in [(63, 65, 33), (129, 127, 95), (200, 300, 257), (256, 128, 224)]:
            A, B, C = ops(M, N, K, seed=cfg * 10 + splits)
            got, guards, st = run_gemm(torch, h, A, B, C, 1.5, 0.5)
            assert st == sg.SGEMM_OK and guards
            p = h.last_plan()
            assert p.config == cfg and p.splits == min(splits, (K + 31) // 32) and p.transpose_a == ta
            check_against_oracle(got, A, B, C, 1.5, 0.5, exact=True)
            Ar, Br, Cr = ops(M, N, K, seed=cfg * 10 + splits + 1, dist=("normal", "uniform", "uniform"))
            got, guards, st = run_gemm(torch, h, Ar, Br, Cr, -0.75, 1.25)
            assert st == sg.SGEMM_OK and guards
            check_against_oracle(got, Ar, Br, Cr, -0.75, 1.25)
    finally:
        force(h)


@pytest.mark.parametrize("cfg", range(4))
def test_a_layouts_give_identical_bits(h, cfg):
    """The three A layouts evaluate every output as the same FMA chain in ascending k:
    the results must agree bit for bit (real operands, every split path)."""
    for (M, N, K), splits in [((300, 260, 777), 1), ((129, 200, 500), 3), ((1000, 2500, 513), 0)]:
        A, B, C = ops(M, N, K, seed=cfg + M, dist=("normal", "normal", "uniform"))
        outs = []
        for ta in (0, 1, 2):
            force(h, cfg, splits, ta)
            try:
                got, guards, st = run_gemm(torch, h, A, B, C, 1.25, -0.5)
                assert st == sg.SGEMM_OK and guards and h.last_plan().transpose_a == ta
            finally:
                force(h)
            outs.append(got)
        for o in outs[1:]:
            assert np.array_equal(outs[0].view(np.uint32), o.view(np.uint32)), (cfg, M, N, K)
        check_against_oracle(outs[1], A, B, C, 1.25, -0.5)


@pytest.mark.parametrize("cfg", range(4))
@pytest.mark.parametrize("splits", [2, 3, 5, 8])
@pytest.mark.parametrize("ta", [1, 2])
def test_cluster_split_matches_workspace_split(h, cfg, splits, ta):
    """Split-K reduced within thread-block clusters (partials added in distributed
    shared memory, one launch) against the same plan with the partials going
    through the workspace to the reduction kernel: the same additions in the same
    order, so bit for bit the same C; exact on integers, inside the bound on reals.
    Shapes around tile multiples, ragged N and unaligned / padded C. The cluster form
    reads A transposed in shared memory: with A forced to be transposed first
    (ta = 1) the plan keeps the workspace even when clusters are asked for."""
    shapes = [((63, 65, 333), (None, None, None), (0, 0, 0)), ((129, 127, 500), (None, None, 130), (0, 0, 1)),
              ((256, 200, 1000), (1001, 203, 201), (0, 0, 0)), ((300, 260, 777), (None, None, None), (1, 0, 2))]
    for (M, N, K), lds, offs in shapes:
        for dist, alpha, beta in ((("int", "int", "int"), 1.5, 0.5), (("normal", "uniform", "uniform"), -0.75, 1.25),
                                  (("normal", "normal", "uniform"), 1.0, 0.0)):
            A, B, C = ops(M, N, K, seed=cfg * 100 + splits * 10 + M, dist=dist)
            outs = []
            for cl in (1, 0):
                force(h, cfg, splits, ta)
                h.set_option(sg.OPT_CLUSTER_SPLIT, cl)
                try:
                    got, guards, st = run_gemm(torch, h, A, B, C, alpha, beta, lds=lds, offsets=offs)
                    assert st == sg.SGEMM_OK and guards
                    assert h.check_device_status() == (sg.SGEMM_OK, 0)
                    p = h.last_plan()
                    assert p.cluster_split == (cl if ta == 2 else 0), p.as_dict()
                    assert p.splits == min(splits, (K + 31) // 32), p.as_dict()
                    if p.cluster_split:  # no reduction launch; the workspace holds operand copies at most
                        assert p.grid == p.units and p.launches == 1 + int(p.transpose_a == 1 or p.repack_a or p.repack_b)
                finally:
                    force(h)
                    h.set_option(sg.OPT_CLUSTER_SPLIT, -1)
                outs.append(got)
            assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32)), (cfg, splits, ta, M, N, K)
            check_against_oracle(outs[0], A, B, C, alpha, beta, exact=dist[0] == "int")


def test_cluster_split_beta_zero_never_reads_c(h):
    """Within clusters too, beta = 0 writes C without reading it (NaN in C stays out)."""
    M, N, K = 200, 190, 600
    A, B, _ = ops(M, N, K, seed=9, dist=("normal", "normal", "uniform"))
    nanC = np.full((M, N), np.nan, np.float32)
    h.set_option(sg.OPT_CLUSTER_SPLIT, 1)
    force(h, 3, 4, 2)
    try:
        got, guards, st = run_gemm(torch, h, A, B, nanC, 1.0, 0.0)
        assert st == sg.SGEMM_OK and guards and h.last_plan().cluster_split == 1
    finally:
        force(h)
        h.set_option(sg.OPT_CLUSTER_SPLIT, -1)
    assert np.all(np.isfinite(got))
    check_against_oracle(got, A, B, None, 1.0, 0.0)


def test_deterministic(h):
    A, B, C = ops(300, 260, 700, seed=5, dist=("normal", "normal", "uniform"))
    r1, _, _ = run_gemm(torch, h, A, B, C, 1.0, 1.0)
    r2, _, _ = run_gemm(torch, h, A, B, C, 1.0, 1.0)
    assert np.array_equal(r1.view(np.uint32), r2.view(np.uint32))


@pytest.mark.parametrize("ta", [0, 1, 2])
def test_leading_dimensions_and_misalignment(h, ta):
    """Padded leading dimensions keep pad columns untouched; misaligned pointers take
    the repack path (A as given or transposed in shared memory) or the transposition
    (A transposed first)."""
    M, N, K = 190, 170, 150
    A, B, C = ops(M, N, K, seed=77)
    force(h, transpose_a=ta)
    try:
        for lds, offs in [((K + 4, N + 8, N + 12), (0, 0, 0)),    # aligned, padded
                          ((K + 1, N + 3, N + 5), (0, 0, 0)),     # unaligned strides
                          ((None, None, None), (1, 2, 3)),        # unaligned pointers
                          ((K + 3, N, N + 1), (2, 0, 1))]:
            got, guards, st = run_gemm(torch, h, A, B, C, 2.0, -1.0, lds=lds, offsets=offs)
            assert st == sg.SGEMM_OK and guards, (lds, offs)
            check_against_oracle(got, A, B, C, 2.0, -1.0, exact=True)
        p = h.last_plan()
    finally:
        force(h)
    assert p.transpose_a == ta and p.repack_a == (0 if ta == 1 else 1) and p.vec_c == 0


def test_quick_returns(h):
    M, N, K = 70, 90, 40
    A, B, C = ops(M, N, K, seed=3, dist=("uniform", "uniform", "uniform"))
    nanA = np.full_like(A, np.nan)
    nanB = np.full_like(B, np.nan)
    # alpha == 0: A, B not read; C = beta * C
    got, guards, st = run_gemm(torch, h, nanA, nanB, C, 0.0, 0.5)
    assert st == sg.SGEMM_OK and guards and np.array_equal(got, 0.5 * C)
    # alpha == 0, beta == 1: C untouched
    got, guards, st = run_gemm(torch, h, nanA, nanB, C, 0.0, 1.0)
    assert st == sg.SGEMM_OK and guards and np.array_equal(got, C)
    # beta == 0: C not read (NaN in C must not appear)
    nanC = np.full_like(C, np.nan)
    got, guards, st = run_gemm(torch, h, A, B, nanC, 1.0, 0.0)
    assert st == sg.SGEMM_OK and guards and np.all(np.isfinite(got))
    check_against_oracle(got, A, B, None, 1.0, 0.0)
    # alpha == 0, beta == 0: C = 0 without reading it
    got, guards, st = run_gemm(torch, h, nanA, nanB, nanC, 0.0, 0.0)
    assert st == sg.SGEMM_OK and guards and np.all(got == 0)
    # K == 0
    A0 = np.zeros((M, 0), np.float32)
    B0 = np.zeros((0, N), np.float32)
    got, guards, st = run_gemm(torch, h, A0, B0, C, 1.0, 2.0)
    assert st == sg.SGEMM_OK and guards and np.array_equal(got, 2.0 * C)
    # M == 0 / N == 0: nothing touched
    for (m, n) in ((0, N), (M, 0)):
        Am = np.zeros((m, K), np.float32)
        Bn = np.zeros((K, n), np.float32)
        Cm = np.zeros((m, n), np.float32)
        got, guards, st = run_gemm(torch, h, Am, Bn, Cm, 1.0, 0.0)
        assert st == sg.SGEMM_OK and guards


def test_invalid_arguments_touch_nothing(h):
    M, N, K = 16, 16, 16
    A, B, C = ops(M, N, K, seed=1)
    bufs = [torch.from_numpy(x).cuda() for x in (A, B, C)]
    pA, pB, pC = (b.data_ptr() for b in bufs)
    bad = [(-1, N, K, K, N, N), (M, N, K, K - 1, N, N), (M, N, K, K, N - 1, N), (M, N, K, K, N, N - 1)]
    for (m, n, k, lda, ldb, ldc) in bad:
        assert h.run_ptr(m, n, k, 1.0, pA, lda, pB, ldb, 0.0, pC, ldc) == sg.SGEMM_ERR_INVALID_VALUE
    assert h.run_ptr(M, N, K, 1.0, None, K, pB, N, 0.0, pC, N) == sg.SGEMM_ERR_INVALID_VALUE
    assert h.run_ptr(M, N, K, 1.0, pA, K, pB, N, 0.0, None, N) == sg.SGEMM_ERR_INVALID_VALUE
    torch.cuda.synchronize()
    assert np.array_equal(bufs[2].cpu().numpy(), C)


def test_option_values_are_checked(h):
    """Out-of-range option values and unknown options are refused and change nothing."""
    lib = sg.library()
    for opt, bad in ((sg.OPT_FORCE_TF32_KERNEL, 2), (sg.OPT_FORCE_REPACK_C, 2), (sg.OPT_FORCE_REPACK_C, -2),
                     (sg.OPT_CLUSTER_SPLIT, 2), (sg.OPT_CLUSTER_SPLIT, -2),
                     (sg.OPT_FORCE_STREAMK, 2), (sg.OPT_FORCE_TRANSPOSE_A, -2), (sg.OPT_FORCE_TRANSPOSE_A, 3),
                     (99, 0)):
        assert lib.sgemm_set_option(h._h, opt, bad) == sg.SGEMM_ERR_INVALID_VALUE, (opt, bad)
    for opt in (sg.OPT_FORCE_TF32_KERNEL, sg.OPT_FORCE_REPACK_C, sg.OPT_FORCE_STREAMK, sg.OPT_FORCE_TRANSPOSE_A,
                sg.OPT_CLUSTER_SPLIT):
        assert lib.sgemm_set_option(h._h, opt, -1) == sg.SGEMM_OK


def test_non_default_stream(h):
    A, B, C = ops(333, 222, 111, seed=8)
    dA, dB, dC = (torch.from_numpy(x).cuda() for x in (A, B, C))
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        h.run(dA, dB, dC, 1.0, 1.0, stream=s)
    s.synchronize()
    check_against_oracle(dC.cpu().numpy(), A, B, C, 1.0, 1.0, exact=True)


def test_run_host(h):
    """Host-operand entry point (the e2e path): padded host strides, pinned and pageable."""
    M, N, K = 257, 131, 513
    A, B, C = ops(M, N, K, seed=21, dist=("normal", "normal", "uniform"))
    Ab = inputs.with_ld(A, K + 3)
    Cb = inputs.with_ld(C, N + 1)
    out = Cb.copy()
    h.run_host(Ab[:, :K], B, out[:, :N], 1.5, 0.5)
    check_against_oracle(out[:, :N], A, B, C, 1.5, 0.5)
    assert np.isnan(out[:, N:]).all()
    pinned = [torch.from_numpy(x).pin_memory() for x in (A, B, C)]
    h.run_host(pinned[0], pinned[1], pinned[2], 1.5, 0.5)
    check_against_oracle(pinned[2].numpy(), A, B, C, 1.5, 0.5)


# ---- the benchmark problems ------------------------------------------------

def _problem(name):
    p = inputs.PROBLEMS[name]
    A, B, C = inputs.problem_operands(name)
    return p, A, B, C


def test_square256(h):
    p, A, B, C = _problem("square256")
    got, guards, st = run_gemm(torch, h, A, B, C, p["alpha"], p["beta"])
    assert st == sg.SGEMM_OK and guards
    check_against_oracle(got, A, B, C, p["alpha"], p["beta"])


@pytest.mark.parametrize("name", ["square4096", "square4096_int"])
def test_square4096(h, name):
    """The headline problem and its integer companion, every element of C against the oracle."""
    p, A, B, C = _problem(name)
    got, guards, st = run_gemm(torch, h, A, B, C, p["alpha"], p["beta"])
    assert st == sg.SGEMM_OK and guards
    check_against_oracle(got, A, B, C, p["alpha"], p["beta"], exact=name.endswith("_int"),
                         ref=problem_reference(name))


@pytest.mark.parametrize("name", ["ragged", "ragged_int"])
def test_ragged(h, name):
    p, A, B, C = _problem(name)
    got, guards, st = run_gemm(torch, h, A, B, C, p["alpha"], p["beta"])
    assert st == sg.SGEMM_OK and guards
    plan = h.last_plan()
    # lda, ldb, ldc are not multiples of 4: A reaches the mainloop transposed (or
    # repacked), B through the aligned copy, C through scalar accesses
    assert (plan.transpose_a or plan.repack_a) and plan.repack_b and not plan.vec_c
    check_against_oracle(got, A, B, C, p["alpha"], p["beta"], exact=name.endswith("_int"))


@pytest.mark.parametrize("n", [512, 1024, 2048, 8192, 16384])
def test_sweep(h, n):
    p, A, B, C = _problem(f"sweep{n}")
    got, guards, st = run_gemm(torch, h, A, B, C, p["alpha"], p["beta"])
    assert st == sg.SGEMM_OK and guards
    # every element up to 8192^3 (about 35 s of oracle time on 16 host threads);
    # 16384^3 (8.8e12 flops) on the edge rows of the first and last two tile rows
    # and 16 seeded random rows
    rows = None if n <= 8192 else sample_rows(n, n_random=16)
    check_against_oracle(got, A, B, C, p["alpha"], p["beta"], rows=rows)


@pytest.mark.parametrize("name", ["skinny_tall", "skinny_wide"])
def test_skinny(h, name):
    p, A, B, C = _problem(name)
    got, guards, st = run_gemm(torch, h, A, B, C, p["alpha"], p["beta"])
    assert st == sg.SGEMM_OK and guards
    plan = h.last_plan()
    assert plan.splits > 1 or plan.sk_tiles > 0  # K shared: split-K or stream-K
    check_against_oracle(got, A, B, C, p["alpha"], p["beta"])


@pytest.mark.parametrize("shape", [(1000, 2500, 513), (1999, 3001, 1031), (1500, 4095, 2050), (1024, 1024, 1024),
                                   (300, 260, 777), (129, 127, 95)])
@pytest.mark.parametrize("ta", [0, 1, 2])
def test_stream_k(h, shape, ta):
    """Stream-K: the tiles of the last, partial round share one span of k-blocks cut
    evenly over the CTAs (whole tiles before it; for small problems the span is all
    of them). Exact on integers, bound on reals, bitwise repeatable."""
    h.set_option(sg.OPT_FORCE_TRANSPOSE_A, ta)
    h.set_option(sg.OPT_FORCE_STREAMK, 1)
    try:
        _stream_k_case(h, shape)
        assert h.last_plan().transpose_a == ta
    finally:
        h.set_option(sg.OPT_FORCE_TRANSPOSE_A, -1)
        h.set_option(sg.OPT_FORCE_STREAMK, -1)


@pytest.mark.parametrize("cfg", range(4))
def test_stream_k_every_config(h, cfg):
    """Each tile-config row (1-3 CTAs per SM) with a stream-K span."""
    force(h, config=cfg)
    h.set_option(sg.OPT_FORCE_STREAMK, 1)
    try:
        for shape in [(700, 900, 1500), (65, 4000, 333)]:
            _stream_k_case(h, shape)
            assert h.last_plan().config == cfg
    finally:
        force(h)
        h.set_option(sg.OPT_FORCE_STREAMK, -1)


def _stream_k_case(h, shape):
    M, N, K = shape
    A, B, C = ops(M, N, K, seed=M + N, dist=("int", "int", "int"))
    got, guards, st = run_gemm(torch, h, A, B, C, 1.5, 0.5)
    assert st == sg.SGEMM_OK and guards
    plan = h.last_plan()
    assert plan.sk_tiles > 0 and plan.splits == 1, plan.as_dict()
    check_against_oracle(got, A, B, C, 1.5, 0.5, exact=True)
    Ar, Br, Cr = ops(M, N, K, seed=M + N + 1, dist=("normal", "uniform", "uniform"))
    got, guards, st = run_gemm(torch, h, Ar, Br, Cr, -1.0, 0.25)
    assert st == sg.SGEMM_OK and guards
    check_against_oracle(got, Ar, Br, Cr, -1.0, 0.25)
    r2, _, _ = run_gemm(torch, h, Ar, Br, Cr, -1.0, 0.25)
    assert np.array_equal(got.view(np.uint32), r2.view(np.uint32))
    assert h.check_device_status() == (sg.SGEMM_OK, 0)


@pytest.mark.parametrize("shape", [(4100, 3001, 300), (6000, 1100, 160)])
def test_run_host_pipelined_panels(h, shape):
    """Large host-buffer calls are pipelined over row panels (the first panel over
    column blocks of B; N = 1100 makes the first block a single 128-column tile):
    results match the oracle."""
    M, N, K = shape
    A, B, C = ops(M, N, K, seed=41, dist=("int", "int", "int"))
    Ab = inputs.with_ld(A, K + 3)
    Cb = inputs.with_ld(C, N + 5)
    for alpha, beta in [(1.5, 0.5), (1.0, 0.0), (0.0, 1.0), (0.0, 2.0)]:
        out = Cb.copy()
        h.run_host(Ab[:, :K], B, out[:, :N], alpha, beta)
        assert np.isnan(out[:, N:]).all()
        check_against_oracle(out[:, :N], A, B, C, alpha, beta, exact=True)
    pinned = [torch.from_numpy(x).pin_memory() for x in (A, B, C)]
    h.run_host(pinned[0], pinned[1], pinned[2], 1.5, 0.5)
    check_against_oracle(pinned[2].numpy(), A, B, C, 1.5, 0.5, exact=True)


def test_offsets_beyond_2_31_elements(h):
    """C with 2.6e9 elements (row offsets past 2^31): the tail rows are still exact.

    Integer A and B, beta = 0 (C never read, allocated uninitialised on the device).
    Every output below row 53687 has an offset under 2^31; the checked rows are the
    first ones and rows far past that point.
    """
    M, N, K = 65536, 40000, 64
    free, _ = torch.cuda.mem_get_info()
    if free < 16 * 2**30:
        pytest.skip("needs 16 GiB of free device memory")
    A = inputs.matrix(51, 0, M, K, "int")
    B = inputs.matrix(51, 1, K, N, "int")
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dC = torch.empty((M, N), dtype=torch.float32, device="cuda")
    h.run(dA, dB, dC, 1.0, 0.0)
    torch.cuda.synchronize()
    assert h.check_device_status() == (sg.SGEMM_OK, 0)
    rows = np.array([0, 1, 53686, 53687, 53688, 60000, M - 2, M - 1])
    got = dC[torch.from_numpy(rows).cuda()].cpu().numpy()
    ref, _ = oracle.sgemm_f64(A, B, None, 1.0, 0.0, rows=rows, with_mag=False)
    assert oracle.exact(got, ref)
    del dC
    torch.cuda.empty_cache()


@pytest.mark.parametrize("skew", [3000, -3000])
def test_timing_skew_is_race_free(h, skew):
    """A slow producer (skew > 0) or slow consumers (skew < 0) change only timing:
    results stay bitwise identical (a race on the shared-memory ring would show here)."""
    cases = [((1999, 3001, 1031), dict()), ((700, 900, 1500), dict(config=1, splits=3, transpose_a=0)),
             ((700, 900, 1500), dict(config=1, splits=3, transpose_a=1)),
             ((300, 260, 777), dict(config=3, splits=1, transpose_a=0)),
             ((300, 260, 777), dict(config=3, splits=1, transpose_a=1)),
             ((1999, 3001, 1031), dict(config=0, splits=1, transpose_a=2)),
             ((700, 900, 1500), dict(config=1, splits=3, transpose_a=2)),
             ((300, 260, 777), dict(config=3, splits=1, transpose_a=2)),
             ((333, 700, 900), dict(config=2, splits=2, transpose_a=2))]
    for (M, N, K), forced in cases:
        A, B, C = ops(M, N, K, seed=M + skew, dist=("normal", "uniform", "uniform"))
        force(h, **forced)
        try:
            ref_run, _, st = run_gemm(torch, h, A, B, C, 1.0, 1.0)
            assert st == sg.SGEMM_OK
            h.set_option(sg.OPT_SKEW_NS, skew)
            skewed, guards, st = run_gemm(torch, h, A, B, C, 1.0, 1.0)
            assert st == sg.SGEMM_OK and guards
            assert h.check_device_status() == (sg.SGEMM_OK, 0)
        finally:
            h.set_option(sg.OPT_SKEW_NS, 0)
            force(h)
        assert np.array_equal(ref_run.view(np.uint32), skewed.view(np.uint32)), (M, N, K, skew)
        check_against_oracle(skewed, A, B, C, 1.0, 1.0)
