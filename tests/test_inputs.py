"""The seeded input generator: SplitMix64 published outputs, determinism and value sets."""

import numpy as np

from dense_fp32_gemm_04_gb300 import inputs


def test_splitmix64_published_outputs():
    # First three outputs of splitmix64 started at state 0 (Vigna's reference
    # implementation of Steele et al.'s SplitMix64 finaliser).
    got = inputs.draws(0, np.arange(3))
    assert [int(x) for x in got] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_deterministic_and_distinct():
    a = inputs.matrix(1, 0, 33, 17, "uniform")
    b = inputs.matrix(1, 0, 33, 17, "uniform")
    c = inputs.matrix(1, 1, 33, 17, "uniform")
    d = inputs.matrix(2, 0, 33, 17, "uniform")
    assert np.array_equal(a, b)
    assert not np.array_equal(a, c) and not np.array_equal(a, d)


def test_uniform_grid_and_range():
    x = inputs.matrix(3, 0, 256, 256, "uniform").astype(np.float64)
    assert x.min() >= -1.0 and x.max() < 1.0
    assert np.all((x + 1.0) * 2**23 == np.round((x + 1.0) * 2**23))
    assert abs(x.mean()) < 0.01


def test_int_values():
    x = inputs.matrix(3, 0, 200, 200, "int")
    vals, counts = np.unique(x, return_counts=True)
    assert list(vals) == [-2, -1, 0, 1, 2]
    assert counts.min() > 0.18 * x.size


def test_normal_moments():
    x = inputs.matrix(4, 0, 300, 300, "normal").astype(np.float64)
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1.0) < 0.02


def test_chunking_is_invisible():
    old = inputs._CHUNK
    try:
        full = inputs.matrix(5, 1, 70, 90, "normal")
        inputs._CHUNK = 1000
        chunked = inputs.matrix(5, 1, 70, 90, "normal")
    finally:
        inputs._CHUNK = old
    assert np.array_equal(full, chunked)


def test_problem_shapes():
    A, B, C = inputs.problem_operands("square256")
    assert A.shape == (256, 256) and B.shape == (256, 256) and not C.any()
    p = inputs.PROBLEMS["ragged"]
    assert (p["M"], p["N"], p["K"]) == (2047, 3001, 1531)
