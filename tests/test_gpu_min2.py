"""sgemm_run_min2: C and its two smallest elements with their (row, column).

Integer operands: C is exact, so values and positions must equal the oracle's
two minimums of the exact product (ties ranked by row-major position).
Real operands: the reported pair must be the two smallest elements of the
GPU's own C (the definition applied to that C) and lie within the FP32 bound of
the oracle's values at those positions.
"""

import numpy as np
import pytest

import dense_fp32_gemm_04_gb300 as sg
import oracle
from dense_fp32_gemm_04_gb300 import inputs

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


def _run(h, A, B, C, alpha, beta):
    dA, dB, dC = (torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in (A, B, C))
    vals, ij = h.run_min2(dA, dB, dC, alpha, beta)
    torch.cuda.synchronize()
    assert h.check_device_status() == (sg.SGEMM_OK, 0)
    return dC.cpu().numpy(), vals.cpu().numpy(), ij.cpu().numpy()


@pytest.mark.parametrize("shape", [(1, 1, 5), (1, 37, 9), (64, 64, 64), (300, 200, 100), (1000, 2500, 513),
                                   (2047, 3001, 1531), (16384, 64, 512)])
def test_integer_exact(h, shape):
    M, N, K = shape
    A, B, C = inputs.problem_operands(M=M, N=N, K=K, seed=M + 3 * N, dist=("int", "int", "int"))
    got, vals, ij = _run(h, A, B, C, 1.0, 1.0)
    ref, _ = oracle.sgemm_f64(A, B, C, 1.0, 1.0, with_mag=False)
    assert oracle.exact(got, ref)
    rv, rr, rc = oracle.min2(ref)
    assert list(vals.astype(np.float64)) == rv
    assert list(ij) == [rr[0], rc[0], rr[1], rc[1]]


@pytest.mark.parametrize("name", ["square256", "ragged", "skinny_wide"])
def test_real(h, name):
    p = inputs.PROBLEMS[name]
    A, B, C = inputs.problem_operands(name)
    got, vals, ij = _run(h, A, B, C, p["alpha"], p["beta"])
    # the definition applied to the GPU's own C
    gv, gr, gc = oracle.min2(got)
    assert list(vals.astype(np.float64)) == gv and list(ij) == [gr[0], gc[0], gr[1], gc[1]]
    # and those elements are within the FP32 bound of the exact product
    rows = np.array([gr[0], gr[1]])
    ref, mag = oracle.sgemm_f64(A, B, C, p["alpha"], p["beta"], rows=rows)
    for t in range(2):
        e = abs(float(vals[t]) - ref[t, gc[t]])
        assert e <= oracle.bound(p["K"], mag[t, gc[t]])
    # the true (FP64) minimum is within two bounds of the reported one
    full, fmag = oracle.sgemm_f64(A, B, C, p["alpha"], p["beta"], with_mag=True)
    tv, _, _ = oracle.min2(full)
    assert abs(tv[0] - float(vals[0])) <= 2 * oracle.bound(p["K"], fmag.max())


def test_empty_and_degenerate(h):
    A = np.zeros((0, 4), np.float32)
    B = np.ones((4, 3), np.float32)
    C = np.zeros((0, 3), np.float32)
    dA, dB, dC = (torch.from_numpy(x).cuda() for x in (A, B, C))
    vals, ij = h.run_min2(dA, dB, dC, 1.0, 0.0)
    torch.cuda.synchronize()
    assert np.all(np.isinf(vals.cpu().numpy())) and list(ij.cpu().numpy()) == [-1, -1, -1, -1]
    # a single element: second entry is +inf at (-1, -1)
    A = np.full((1, 3), 2.0, np.float32)
    B = np.full((3, 1), -1.0, np.float32)
    got, vals, ij = _run(h, A, B, np.zeros((1, 1), np.float32), 1.0, 0.0)
    assert vals[0] == -6.0 and np.isinf(vals[1]) and list(ij) == [0, 0, -1, -1]


def test_deterministic_under_ties(h):
    # all-equal product: every element ties, the first two positions win
    A = np.ones((300, 17), np.float32)
    B = np.ones((17, 500), np.float32)
    got, vals, ij = _run(h, A, B, np.zeros((300, 500), np.float32), 1.0, 0.0)
    assert list(vals) == [17.0, 17.0] and list(ij) == [0, 0, 0, 1]


@pytest.mark.parametrize("force", [dict(), dict(config=1, splits=3), dict(config=3, splits=1),
                                   dict(config=0, splits=1, transpose_a=0), dict(config=2, splits=5, transpose_a=1),
                                   dict(config=0, splits=1, transpose_a=2)])
@pytest.mark.parametrize("shape", [(300, 200, 100), (1000, 2500, 513), (2047, 3001, 1531)])
def test_every_plan(h, force, shape):
    """Whichever kernel writes the final C values (whole-tile epilogue with either A
    layout, tail-split reduction, split-K reduction), the pass over C finds the two
    minima. Integer operands: values and positions equal the oracle's."""
    M, N, K = shape
    A, B, C = inputs.problem_operands(M=M, N=N, K=K, seed=7 * M + N, dist=("int", "int", "int"))
    h.set_option(sg.OPT_FORCE_CONFIG, force.get("config", -1))
    h.set_option(sg.OPT_FORCE_SPLITS, force.get("splits", 0))
    h.set_option(sg.OPT_FORCE_TRANSPOSE_A, force.get("transpose_a", -1))
    try:
        got, vals, ij = _run(h, A, B, C, -1.0, 1.0)
    finally:
        h.set_option(sg.OPT_FORCE_CONFIG, -1)
        h.set_option(sg.OPT_FORCE_SPLITS, 0)
        h.set_option(sg.OPT_FORCE_TRANSPOSE_A, -1)
    ref, _ = oracle.sgemm_f64(A, B, C, -1.0, 1.0, with_mag=False)
    assert oracle.exact(got, ref)
    rv, rr, rc = oracle.min2(ref)
    assert list(vals.astype(np.float64)) == rv and list(ij) == [rr[0], rc[0], rr[1], rc[1]]


def test_tail_split_plan(h):
    # whole tiles plus a stream-K last round (104 tiles shared by 152 CTAs)
    M, N, K = 2048, 2048, 2048
    A, B, C = inputs.problem_operands(M=M, N=N, K=K, seed=99, dist=("int", "int", "zero"))
    got, vals, ij = _run(h, A, B, C, 1.0, 0.0)
    plan = h.last_plan()
    ref, _ = oracle.sgemm_f64(A, B, None, 1.0, 0.0, with_mag=False)
    assert oracle.exact(got, ref)
    rv, rr, rc = oracle.min2(ref)
    assert list(vals.astype(np.float64)) == rv and list(ij) == [rr[0], rc[0], rr[1], rc[1]]
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert plan.sk_tiles > 0, plan.as_dict()


def test_tf32_and_scale_only_plans(h):
    """TF32 mode and C = beta * C (alpha == 0): the same pass over C."""
    A, B, C = inputs.problem_operands(M=333, N=444, K=96, seed=5, dist=("int", "int", "int"))
    got, vals, ij = _run(h, A, B, C, 0.0, 2.0)
    rv, rr, rc = oracle.min2(2.0 * C.astype(np.float64))
    assert list(vals.astype(np.float64)) == rv and list(ij) == [rr[0], rc[0], rr[1], rc[1]]
    h.set_math_mode(sg.MATH_TF32)
    try:
        got, vals, ij = _run(h, A, B, C, 1.0, 1.0)
    finally:
        h.set_math_mode(sg.MATH_FP32)
    ref, _ = oracle.sgemm_f64(A, B, C, 1.0, 1.0, with_mag=False)
    assert oracle.exact(got, ref)  # integer operands are exact in TF32
    rv, rr, rc = oracle.min2(ref)
    assert list(vals.astype(np.float64)) == rv and list(ij) == [rr[0], rc[0], rr[1], rc[1]]


def _min2_reference(C):
    """The definition on a given C: NaN ranks as +inf, equal values by row-major position."""
    flat = np.where(np.isnan(C), np.inf, C).astype(np.float64).ravel()
    order = np.lexsort((np.arange(flat.size), flat))[:2]
    return flat[order], [(int(i) // C.shape[1], int(i) % C.shape[1]) for i in order]


@pytest.mark.parametrize("N", [520, 517])  # 16-byte loads of C, and element loads
def test_nan_ranks_as_infinity(h, N):
    """NaN in C (through beta * C) ranks as +inf: it is never chosen while two other
    values exist, and an all-NaN C gives +inf at the first two positions."""
    M, K = 300, 40
    A, B, C = inputs.problem_operands(M=M, N=N, K=K, seed=N, dist=("int", "int", "int"))
    rng = np.random.default_rng(N)
    for kind in ("some", "all_but_one", "all"):
        Cn = C.copy()
        if kind == "some":
            Cn[rng.random(Cn.shape) < 0.3] = np.nan
        else:
            Cn[:] = np.nan
            if kind == "all_but_one":
                Cn[M // 2, N // 3] = 0.0
        got, vals, ij = _run(h, A, B, Cn, 1.0, 1.0)
        want_vals, want_pos = _min2_reference(got)
        assert [float(v) for v in vals] == [float(v) for v in want_vals], kind
        assert [tuple(ij[:2]), tuple(ij[2:])] == want_pos, kind
