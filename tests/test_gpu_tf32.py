"""GPU parity of the flagged TF32 tensor-core mode (SGEMM_MATH_TF32).

Bounds: the stated TF32 bound (K + 2) * 2^-10 * (|alpha| sum |a||b| + |beta||c|)
is very loose at large K, so every case is also held to a tighter one that
follows the same rounding argument more closely: each operand is rounded to
TF32 (relative error below 2^-10, so a product is off by below 2^-9 + 2^-20),
then K products are summed in FP32 (depth K + 2 with alpha/beta):
|err| <= (2^-9 + 2^-20 + (K + 2) * 2^-24) * magnitude. A wrong descriptor or
layout would fail the tight bound by orders of magnitude. Integer operands in
{-2..2} are exact in TF32, so those runs must be bit-exact. Every case runs on
both TF32 kernels (one CTA per tile, and CTA pairs).
"""

import numpy as np
import pytest

import dense_fp32_gemm_04_gb300 as sg
import oracle
from dense_fp32_gemm_04_gb300 import inputs
from gpu_helpers import problem_reference, run_gemm

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", params=[0, 1], ids=["one_cta", "cta_pair"])
def h(request):
    """A TF32-mode handle forced to one kernel: 0 = one CTA per 128 x 256 tile,
    1 = a CTA pair (cluster of two, tcgen05 .cta_group::2) per 256 x 256 tile."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_fp32_gemm_04_gb300 import _build

    _build.build()
    handle = sg.Sgemm(0)
    handle.set_math_mode(sg.MATH_TF32)
    handle.set_option(sg.OPT_FORCE_TF32_KERNEL, request.param)
    handle.tf32_kernel = request.param
    yield handle
    handle.close()


def _assert_kernel(h):
    plan = h.last_plan()
    assert plan.kernel == sg.KERNEL_TF32 and plan.config == h.tf32_kernel, plan.as_dict()
    if plan.config == 1:
        assert (plan.bm, plan.bn) == (256, 256) and plan.grid % 2 == 0


def _check(got, A, B, C, alpha, beta, rows=None, exact=False, ref=None):
    K = A.shape[1]
    ref, mag = ref if ref is not None else oracle.sgemm_f64(A, B, C, alpha, beta, rows=rows)
    g = (got if rows is None else got[rows]).astype(np.float64)
    assert np.all(np.isfinite(g))
    err = np.abs(g - ref)
    assert np.all(err <= oracle.bound(K, mag, oracle.U_TF32)), "outside the TF32 bound"
    tight = (2.0**-9 + 2.0**-20 + (K + 2) * 2.0**-24) * mag
    bad = err > tight
    assert not bad.any(), f"{int(bad.sum())} elements outside the tight TF32 bound, worst ratio {float(np.max(err / np.maximum(tight, 1e-300))):.3g}"
    if exact:
        assert oracle.exact(got if rows is None else got[rows], ref)


@pytest.mark.parametrize("shape", [(1, 1, 1), (128, 256, 32), (129, 257, 33), (256, 256, 256), (300, 500, 200),
                                   (77, 1000, 517), (520, 1030, 96)])
def test_integer_exact(h, shape):
    M, N, K = shape
    A, B, C = inputs.problem_operands(M=M, N=N, K=K, seed=M + N + K, dist=("int", "int", "int"))
    got, guards, st = run_gemm(torch, h, A, B, C, 1.5, 0.5)
    assert st == sg.SGEMM_OK and guards
    _assert_kernel(h)
    assert h.check_device_status() == (sg.SGEMM_OK, 0)
    _check(got, A, B, C, 1.5, 0.5, exact=True)


def test_real_square(h):
    A, B, C = inputs.problem_operands(M=512, N=512, K=512, seed=5, dist=("uniform", "uniform", "uniform"))
    got, guards, st = run_gemm(torch, h, A, B, C, 1.5, 0.5)
    assert st == sg.SGEMM_OK and guards
    _check(got, A, B, C, 1.5, 0.5)


def test_ragged_problem(h):
    p = inputs.PROBLEMS["ragged"]
    A, B, C = inputs.problem_operands("ragged")
    got, guards, st = run_gemm(torch, h, A, B, C, p["alpha"], p["beta"])
    assert st == sg.SGEMM_OK and guards
    plan = h.last_plan()
    # lda, ldb and ldc are not multiples of 4: both operands repacked, C written in
    # place (16-byte accesses inside each row)
    assert plan.repack_a == 1 and plan.repack_b == 1 and plan.repack_c == 0 and plan.vec_c == 0
    # the copies of A and B (one launch), mainloop, [stream-K reduction]
    assert plan.launches == 2 + (1 if plan.sk_tiles else 0)
    _check(got, A, B, C, p["alpha"], p["beta"])


def test_unaligned_and_padded(h):
    """Padded and unaligned operands; C small enough to be written in place."""
    M, N, K = 190, 300, 130
    A, B, C = inputs.problem_operands(M=M, N=N, K=K, seed=6, dist=("int", "int", "int"))
    for lds, offs in [((K + 4, N + 8, N + 4), (0, 0, 0)), ((K + 1, N + 3, N + 1), (1, 2, 3))]:
        got, guards, st = run_gemm(torch, h, A, B, C, 1.0, -1.0, lds=lds, offsets=offs)
        assert st == sg.SGEMM_OK and guards
        _check(got, A, B, C, 1.0, -1.0, exact=True)


@pytest.mark.parametrize("K", [130, 700])
def test_aligned_c_with_a_partial_last_chunk(h, K):
    """C 16-byte accessible (ldc a multiple of 4) but N = 301: the write-out's last
    16-byte chunk of every row is cut by N and goes element by element; rows past M
    in the last tile row are skipped. Pad columns and guard bands stay untouched."""
    M, N = 190, 301
    A, B, C = inputs.problem_operands(M=M, N=N, K=K, seed=23, dist=("int", "int", "int"))
    for beta in (0.5, 0.0):
        got, guards, st = run_gemm(torch, h, A, B, C, 1.5, beta, lds=(K + 4, N + 7, 304))
        assert st == sg.SGEMM_OK and guards
        plan = h.last_plan()
        assert plan.vec_c == 1 and plan.repack_c == 0, plan.as_dict()
        _check(got, A, B, C, 1.5, beta, exact=True)


@pytest.mark.parametrize("name", ["square4096", "square4096_int"])
def test_square4096(h, name):
    p = inputs.PROBLEMS[name]
    A, B, C = inputs.problem_operands(name)
    got, guards, st = run_gemm(torch, h, A, B, C, p["alpha"], p["beta"])
    assert st == sg.SGEMM_OK and guards
    _assert_kernel(h)
    assert h.check_device_status() == (sg.SGEMM_OK, 0)
    _check(got, A, B, C, p["alpha"], p["beta"], exact=name.endswith("_int"), ref=problem_reference(name))


def test_deterministic(h):
    A, B, C = inputs.problem_operands(M=384, N=512, K=640, seed=7, dist=("normal", "normal", "uniform"))
    r1, _, _ = run_gemm(torch, h, A, B, C, 1.0, 1.0)
    r2, _, _ = run_gemm(torch, h, A, B, C, 1.0, 1.0)
    assert np.array_equal(r1.view(np.uint32), r2.view(np.uint32))


def test_mode_switch_back_to_fp32(h):
    A, B, C = inputs.problem_operands(M=200, N=200, K=300, seed=8, dist=("normal", "normal", "uniform"))
    h.set_math_mode(sg.MATH_FP32)
    try:
        got, _, st = run_gemm(torch, h, A, B, C, 1.0, 1.0)
        assert st == sg.SGEMM_OK and h.last_plan().kernel == sg.KERNEL_FFMA
        ref, mag = oracle.sgemm_f64(A, B, C, 1.0, 1.0)
        assert oracle.check(got, ref, mag, 300)[0]
    finally:
        h.set_math_mode(sg.MATH_TF32)


@pytest.mark.parametrize("shape", [(4096, 4000, 2048), (512, 512, 512), (77, 1000, 517), (300, 700, 1000)])
def test_stream_k(h, shape):
    """The last partial round's tiles form a stream-K span (the whole problem when it is
    a single round): partial tiles are added in k order by the reduction; exact on
    integers, tight bound on reals, and bitwise repeatable."""
    h.set_option(sg.OPT_FORCE_STREAMK, 1)
    try:
        _stream_k_case(h, shape)
    finally:
        h.set_option(sg.OPT_FORCE_STREAMK, -1)


def _stream_k_case(h, shape):
    M, N, K = shape
    A, B, C = inputs.problem_operands(M=M, N=N, K=K, seed=M + K, dist=("int", "int", "int"))
    got, guards, st = run_gemm(torch, h, A, B, C, 1.5, 0.5)
    assert st == sg.SGEMM_OK and guards
    plan = h.last_plan()
    _assert_kernel(h)
    assert plan.sk_tiles > 0 and plan.launches == 2 + int(plan.repack_a or plan.repack_b) + 2 * plan.repack_c, \
        plan.as_dict()
    # every element (4096 x 4000 x 2048: about 2 s of oracle time per run)
    _check(got, A, B, C, 1.5, 0.5, exact=True)
    Ar, Br, Cr = inputs.problem_operands(M=M, N=N, K=K, seed=M + K + 1, dist=("normal", "uniform", "uniform"))
    r1, guards, st = run_gemm(torch, h, Ar, Br, Cr, -1.0, 0.25)
    assert st == sg.SGEMM_OK and guards
    _check(r1, Ar, Br, Cr, -1.0, 0.25)
    r2, _, _ = run_gemm(torch, h, Ar, Br, Cr, -1.0, 0.25)
    assert np.array_equal(r1.view(np.uint32), r2.view(np.uint32))


@pytest.mark.parametrize("repack_c", [0, 1])
@pytest.mark.parametrize("K", [96, 600])
def test_unaligned_c_in_place_or_through_a_copy(h, repack_c, K):
    """A C that is not 16-byte accessible, written in place (4-byte accesses, lane l
    on column l of each staged row, whatever the row's alignment) or computed in an
    aligned workspace copy (filled from C first when beta != 0). Short K (3 k-blocks)
    and long K (19); N = 700 leaves a partial last tile. Pad columns and guard bands
    around C stay untouched."""
    M, N = 600, 700
    A, B, C = inputs.problem_operands(M=M, N=N, K=K, seed=17, dist=("int", "int", "int"))
    h.set_option(sg.OPT_FORCE_REPACK_C, repack_c)
    try:
        for beta, pad, off in ((0.5, 1, 1), (0.0, 1, 1), (1.0, 2, 3), (-1.0, 3, 2), (0.5, 4, 1)):
            got, guards, st = run_gemm(torch, h, A, B, C, 1.5, beta, lds=(K, N, N + pad), offsets=(0, 0, off))
            assert st == sg.SGEMM_OK and guards
            plan = h.last_plan()
            assert plan.repack_c == repack_c and plan.vec_c == 0, plan.as_dict()
            _check(got, A, B, C, 1.5, beta, exact=True)
    finally:
        h.set_option(sg.OPT_FORCE_REPACK_C, -1)
