"""The FP64 oracle against its pins, and the FP32 error bound against the pages' FP32 loop."""

import numpy as np
import pytest

import oracle
import oracle_pins
from dense_fp32_gemm_04_gb300 import inputs


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle._default())


def test_fp32_ground_truth_inside_bound():
    """The pages' FP32 i-j-k loop (float accumulator) stays inside the FP32 bound."""
    for (M, N, K, alpha, beta, dist) in [(32, 48, 1024, 1.0, 0.0, "uniform"),
                                         (40, 24, 777, 1.5, 0.5, "normal")]:
        A = inputs.matrix(1, 0, M, K, dist)
        B = inputs.matrix(1, 1, K, N, dist)
        C = inputs.matrix(1, 2, M, N, "uniform")
        ref, mag = oracle.sgemm_f64(A, B, C, alpha, beta)
        got = oracle.sgemm_f32_ijk(A, B, C, alpha, beta)
        ok, worst, nbad = oracle.check(got, ref, mag, K)
        assert ok, (worst, nbad)
        # the FP32 loop does round: the result is not exactly the FP64 one
        assert not oracle.exact(got, ref)


def test_bound_catches_dropped_term():
    """A result missing one product (k = 0) is outside the bound: the bound is not vacuous."""
    M, N, K = 32, 32, 512
    A = inputs.matrix(2, 0, M, K, "uniform")
    B = inputs.matrix(2, 1, K, N, "uniform")
    ref, mag = oracle.sgemm_f64(A, B, None, 1.0, 0.0)
    dropped = oracle.sgemm_f32_ijk(np.ascontiguousarray(A[:, 1:]), np.ascontiguousarray(B[1:, :]), None, 1.0, 0.0)
    ok, worst, nbad = oracle.check(dropped, ref, mag, K)
    assert not ok and nbad > 0.9 * M * N


def test_bound_catches_one_ulp_per_step_drift():
    """A result off by K ulps in the wrong direction everywhere is rejected for large |sum|."""
    M, N, K = 16, 16, 256
    A = inputs.matrix(6, 0, M, K, "int")
    B = inputs.matrix(6, 1, K, N, "int")
    ref, mag = oracle.sgemm_f64(A, B, None, 1.0, 0.0)
    bad = (ref + np.sign(ref + 0.5) * oracle.bound(K, mag) * 1.01).astype(np.float32)
    ok, worst, _ = oracle.check(bad, ref, mag, K)
    assert not ok and worst > 1.0


def test_check_rejects_nan():
    ref = np.zeros((2, 2))
    mag = np.ones((2, 2))
    got = np.zeros((2, 2), dtype=np.float32)
    got[1, 1] = np.nan
    ok, _, nbad = oracle.check(got, ref, mag, 4)
    assert not ok and nbad == 1


def test_threads_reported():
    assert oracle.max_threads() >= 1


def test_empty_shapes():
    A = np.zeros((0, 5), dtype=np.float32)
    B = np.zeros((5, 3), dtype=np.float32)
    out, mag = oracle.sgemm_f64(A, B, None, 1.0, 0.0)
    assert out.shape == (0, 3)
    A = np.zeros((4, 0), dtype=np.float32)
    B = np.zeros((0, 3), dtype=np.float32)
    C = inputs.matrix(1, 2, 4, 3, "uniform")
    out, mag = oracle.sgemm_f64(A, B, C, 1.0, 2.0)
    assert np.array_equal(out, 2.0 * C.astype(np.float64))


def _min2_brute(v):
    """Sort every (value, row-major position) pair: the definition, by brute force."""
    M, N = v.shape
    pairs = sorted((float(v[i, j]), i * N + j) for i in range(M) for j in range(N))
    out = pairs[:2] + [(float("inf"), None)] * (2 - len(pairs[:2]))
    vals = [p[0] for p in out]
    rows = [p[1] // N if p[1] is not None else -1 for p in out]
    cols = [p[1] % N if p[1] is not None else -1 for p in out]
    return vals, rows, cols


@pytest.mark.parametrize("shape", [(1, 1), (1, 7), (5, 1), (3, 4), (9, 13), (16, 16)])
def test_min2_matches_brute_force(shape):
    M, N = shape
    for seed in range(5):
        v = inputs.matrix(seed, 0, M, N, "int")  # many ties
        assert oracle.min2(v) == _min2_brute(v)
        w = inputs.matrix(seed, 1, M, N, "normal")
        assert oracle.min2(w) == _min2_brute(w)


def test_min2_ties_take_the_first_position():
    v = np.array([[3.0, -1.0, 2.0], [-1.0, 0.0, -1.0]], dtype=np.float32)
    assert oracle.min2(v) == ([-1.0, -1.0], [0, 1], [1, 0])
