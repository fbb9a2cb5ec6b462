"""Randomised GPU parity sweep: seeded random shapes, leading-dimension pads,
pointer offsets, alpha / beta and forced plan options, on the FP32 path and on
both TF32 kernel forms, every result checked against the FP64 oracle.

The fixed cases of the other GPU tests sit on chosen edges (tile multiples +-1,
the benchmark problems); this sweep draws the combinations in between, where a
scheduling or indexing mistake (a stream-K range boundary, a split slice, a
partial pair tile, a repacked operand with an offset, a ragged row or column of
the staged 128 x 128 epilogue, an unaligned row of C written in place or through
its aligned copy) would show up. The FP32 cases also force a random
tile-config row. Integer
operands must be bit-exact; real ones must lie inside the mode's bound (for
TF32 also the tight bound of test_gpu_tf32). Every case also checks the canary
guards around C and the device status word.
"""

import numpy as np
import pytest

import dense_fp32_gemm_04_gb300 as sg
import oracle
from dense_fp32_gemm_04_gb300 import inputs
from gpu_helpers import check_against_oracle, run_gemm

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

CASES = 150
ALPHAS = (1.0, 1.5, -0.75, 2.0, 0.0)
BETAS = (0.0, 1.0, 0.5, -1.0)


@pytest.fixture(scope="module")
def lib_built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_fp32_gemm_04_gb300 import _build

    _build.build()


def _draw_case(rng):
    """One random problem: shape, pads, offsets, scalars, distribution, plan options."""
    M = int(rng.integers(1, 520))
    N = int(rng.integers(1, 600))
    K = int(rng.integers(1, 800))
    pads = tuple(int(rng.choice([0, 0, 1, 3, 4, 9])) for _ in range(3))
    offsets = tuple(int(rng.choice([0, 0, 0, 1, 2, 4])) for _ in range(3))
    alpha = float(rng.choice(ALPHAS, p=[0.3, 0.25, 0.2, 0.15, 0.1]))
    beta = float(rng.choice(BETAS))
    dist = ("int", "int", "int") if rng.random() < 0.5 else ("normal", "uniform", "uniform")
    opts = {
        "config": int(rng.choice([-1, -1, 0, 0, 1, 2, 3])),
        "streamk": int(rng.choice([-1, -1, 0, 1])),
        "splits": int(rng.choice([0, 0, 0, 2, 3, 5, 8])),
        "transpose_a": int(rng.choice([-1, -1, 0, 1, 2])),
    }
    return M, N, K, pads, offsets, alpha, beta, dist, opts


def _tf32_check(got, A, B, C, alpha, beta, exact):
    K = A.shape[1]
    ref, mag = oracle.sgemm_f64(A, B, C, alpha, beta)
    g = got.astype(np.float64)
    assert np.all(np.isfinite(g))
    err = np.abs(g - ref)
    assert np.all(err <= oracle.bound(K, mag, oracle.U_TF32)), "outside the TF32 bound"
    tight = (2.0**-9 + 2.0**-20 + (K + 2) * 2.0**-24) * mag
    assert np.all(err <= tight), "outside the tight TF32 bound"
    if exact:
        assert oracle.exact(got, ref)


@pytest.mark.parametrize("mode", ["fp32", "tf32_one_cta", "tf32_cta_pair"])
def test_random_problems(lib_built, mode):
    rng = np.random.default_rng({"fp32": 101, "tf32_one_cta": 202, "tf32_cta_pair": 303}[mode])
    h = sg.Sgemm(0)
    try:
        if mode != "fp32":
            h.set_math_mode(sg.MATH_TF32)
            h.set_option(sg.OPT_FORCE_TF32_KERNEL, 0 if mode == "tf32_one_cta" else 1)
        for case in range(CASES):
            M, N, K, pads, offsets, alpha, beta, dist, opts = _draw_case(rng)
            h.set_option(sg.OPT_FORCE_STREAMK, opts["streamk"])
            if mode == "fp32":
                h.set_option(sg.OPT_FORCE_CONFIG, opts["config"])
                h.set_option(sg.OPT_FORCE_SPLITS, opts["splits"])
                h.set_option(sg.OPT_FORCE_TRANSPOSE_A, opts["transpose_a"])
                # split-K within clusters or through the workspace (own generator: the
                # cases drawn above stay the same)
                h.set_option(sg.OPT_CLUSTER_SPLIT, int(np.random.default_rng(7000 + case).choice([-1, -1, 0, 1])))
            else:
                # C written in place or through an aligned copy (own generator: the
                # cases drawn above stay the same)
                h.set_option(sg.OPT_FORCE_REPACK_C, int(np.random.default_rng(case).choice([-1, 0, 1])))
            A, B, C = inputs.problem_operands(M=M, N=N, K=K, seed=1000 + case, dist=dist)
            lds = (K + pads[0], N + pads[1], N + pads[2])
            got, guards, st = run_gemm(torch, h, A, B, C, alpha, beta, lds=lds, offsets=offsets)
            what = (mode, case, M, N, K, pads, offsets, alpha, beta, dist[0], opts, h.last_plan().as_dict())
            assert st == sg.SGEMM_OK and guards, what
            assert h.check_device_status() == (sg.SGEMM_OK, 0), what
            exact = dist[0] == "int"
            if mode == "fp32":
                check_against_oracle(got, A, B, C, alpha, beta, exact=exact)
            else:
                plan = h.last_plan()
                if plan.kernel == sg.KERNEL_TF32:
                    assert plan.config == (0 if mode == "tf32_one_cta" else 1), what
                _tf32_check(got, A, B, C, alpha, beta, exact)
    finally:
        h.close()
