"""Pins that tie the FP64 oracle to facts other than itself.

Each ``pin_*`` takes an :class:`oracle.Oracle` and raises AssertionError when
the oracle disagrees with something the pages or the mathematics fix:

* the pages' special case alpha = 1, beta = 0 ("SGEMM CUDA kernel (First
  Half)", opening definition) against exact integer arithmetic;
* brute force on every shape 1..8 x 1..8 x 1..8 against exact rationals;
* identity and permutation operands (closed forms);
* alpha = 0 passthrough and beta = 0 not reading C (the reading of the
  FP32 page kernel's beta == 0 branch, "Optimizing Matrix Multiplication in
  CUDA", 1D thread tiling epilogue);
* integer-valued inputs whose sums stay below 2**24, against int64;
* a library cross-check (numpy float64 matmul) on real inputs;
* the error-bound magnitude against its closed form.

``tests/test_oracle.py`` runs them on the real build; ``tests/test_oracle_mutants.py``
runs them on builds with planted mistakes and requires each to be caught.
"""

from __future__ import annotations

import itertools
from fractions import Fraction

import numpy as np

from dense_fp32_gemm_04_gb300 import inputs


def _ints(seed, tag, r, c):
    return inputs.matrix(seed, tag, r, c, "int")


def _exact_gemm(A, B, C, alpha, beta):
    """Exact rational alpha*A@B + beta*C for small float inputs (pure Python)."""
    M, K = A.shape
    N = B.shape[1]
    a, b = Fraction(float(alpha)), Fraction(float(beta))
    out = [[None] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            s = Fraction(0)
            for k in range(K):
                s += Fraction(float(A[i, k])) * Fraction(float(B[k, j]))
            v = a * s
            if beta != 0.0:
                v += b * Fraction(float(C[i, j]))
            out[i][j] = v
    return out


def pin_alpha1_beta0_int64(orc):
    """alpha = 1, beta = 0 on integer operands equals an int64 triple loop exactly."""
    for (M, N, K) in [(5, 7, 3), (13, 9, 31), (17, 1, 40), (1, 23, 19)]:
        A = _ints(11, 0, M, K)
        B = _ints(11, 1, K, N)
        out, _ = orc.sgemm_f64(A, B, None, 1.0, 0.0)
        Ai, Bi = A.astype(np.int64), B.astype(np.int64)
        ref = np.zeros((M, N), dtype=np.int64)
        for i in range(M):
            for j in range(N):
                acc = 0
                for k in range(K):
                    acc += int(Ai[i, k]) * int(Bi[k, j])
                ref[i, j] = acc
        assert np.array_equal(out, ref.astype(np.float64)), (M, N, K)


def pin_bruteforce_tiny(orc):
    """Every M, N, K in 1..8 with integer operands, alpha=1.5, beta=-0.5: exact."""
    for M, N, K in itertools.product(range(1, 9), repeat=3):
        seed = 100 + M * 64 + N * 8 + K
        A = _ints(seed, 0, M, K)
        B = _ints(seed, 1, K, N)
        C = _ints(seed, 2, M, N)
        out, mag = orc.sgemm_f64(A, B, C, 1.5, -0.5)
        ref = _exact_gemm(A, B, C, 1.5, -0.5)
        for i in range(M):
            for j in range(N):
                assert Fraction(out[i, j]) == ref[i][j], (M, N, K, i, j)
        # magnitude: |alpha| * |A|@|B| + |beta| * |C|, exact in integers / 2
        magref = 1.5 * (np.abs(A).astype(np.int64) @ np.abs(B).astype(np.int64)) + 0.5 * np.abs(C)
        assert np.array_equal(mag, magref), (M, N, K)


def pin_identity(orc):
    """A = I (K = M): C_out = alpha*B + beta*C, exact for powers of two."""
    M, N = 37, 29
    A = np.eye(M, dtype=np.float32)
    B = inputs.matrix(5, 1, M, N, "uniform")
    C = inputs.matrix(5, 2, M, N, "uniform")
    out, _ = orc.sgemm_f64(A, B, C, 2.0, 0.25)
    assert np.array_equal(out, 2.0 * B.astype(np.float64) + 0.25 * C.astype(np.float64))
    out, _ = orc.sgemm_f64(A, B, C, 1.3, -0.7)
    ref = np.float64(np.float32(1.3)) * B.astype(np.float64) + np.float64(np.float32(-0.7)) * C
    assert np.max(np.abs(out - ref)) <= 1e-15 * np.max(np.abs(ref))


def pin_permutation(orc):
    """A = permutation matrix P: row i of C_out is row perm[i] of B, exactly."""
    M, N = 41, 33
    perm = np.argsort(inputs.draws(9, np.arange(M)).astype(np.float64))
    A = np.zeros((M, M), dtype=np.float32)
    A[np.arange(M), perm] = 1.0
    B = inputs.matrix(9, 1, M, N, "normal")
    out, _ = orc.sgemm_f64(A, B, None, 1.0, 0.0)
    assert np.array_equal(out, B[perm].astype(np.float64))
    # a non-square left factor: rows of P restricted to the first 17 rows of A
    out, _ = orc.sgemm_f64(A[:17], B, None, 1.0, 0.0)
    assert np.array_equal(out, B[perm[:17]].astype(np.float64))


def pin_alpha_zero(orc):
    """alpha = 0: C_out = beta * C_in exactly, A and B never read (NaN there is harmless)."""
    M, N, K = 19, 21, 12
    A = np.full((M, K), np.nan, dtype=np.float32)
    B = np.full((K, N), np.nan, dtype=np.float32)
    C = inputs.matrix(3, 2, M, N, "uniform")
    out, mag = orc.sgemm_f64(A, B, C, 0.0, 0.5)
    assert np.array_equal(out, 0.5 * C.astype(np.float64))
    assert np.array_equal(mag, 0.5 * np.abs(C.astype(np.float64)))


def pin_beta_zero_no_read(orc):
    """beta = 0: C_in is not read, so NaN in C does not reach the output."""
    M, N, K = 23, 17, 9
    A = _ints(4, 0, M, K)
    B = _ints(4, 1, K, N)
    C = np.full((M, N), np.nan, dtype=np.float32)
    out, _ = orc.sgemm_f64(A, B, C, 1.0, 0.0)
    assert np.all(np.isfinite(out))
    assert np.array_equal(out, (A.astype(np.int64) @ B.astype(np.int64)).astype(np.float64))


def pin_integer_padded(orc):
    """Integer operands in buffers with padded leading dimensions: exact against int64."""
    M, N, K = 96, 80, 700
    A = _ints(21, 0, M, K)
    B = _ints(21, 1, K, N)
    C = _ints(21, 2, M, N)
    Ab = inputs.with_ld(A, K + 5)
    Bb = inputs.with_ld(B, N + 3)
    Cb = inputs.with_ld(C, N + 7)
    out, _ = orc.sgemm_f64(Ab[:, :K], Bb[:, :N], Cb[:, :N], 1.0, 1.0)
    ref = A.astype(np.int64) @ B.astype(np.int64) + C.astype(np.int64)
    assert np.array_equal(out, ref.astype(np.float64))
    # the sums stay far below 2**24, so the FP32 ground truth is exact as well
    g = orc.sgemm_f32_ijk(A, B, C, 1.0, 1.0)
    assert np.array_equal(g.astype(np.int64), ref)


def pin_library_crosscheck(orc):
    """Real operands: agrees with numpy's float64 matmul to 1e-12 of the bound magnitude."""
    M, N, K = 37, 53, 129
    A = inputs.matrix(7, 0, M, K, "uniform")
    B = inputs.matrix(7, 1, K, N, "normal")
    C = inputs.matrix(7, 2, M, N, "uniform")
    Ab = inputs.with_ld(A, K + 3)
    out, mag = orc.sgemm_f64(Ab[:, :K], B, C, 1.5, 0.5)
    A64, B64, C64 = A.astype(np.float64), B.astype(np.float64), C.astype(np.float64)
    ref = 1.5 * (A64 @ B64) + 0.5 * C64
    magref = 1.5 * (np.abs(A64) @ np.abs(B64)) + 0.5 * np.abs(C64)
    assert np.all(np.abs(out - ref) <= 1e-12 * magref)
    assert np.all(np.abs(mag - magref) <= 1e-12 * magref)


def pin_rows_subset(orc):
    """Selected rows equal the same rows of the full product (sampling is faithful)."""
    M, N, K = 50, 40, 30
    A = inputs.matrix(8, 0, M, K, "uniform")
    B = inputs.matrix(8, 1, K, N, "uniform")
    C = inputs.matrix(8, 2, M, N, "uniform")
    full, fmag = orc.sgemm_f64(A, B, C, 1.5, 0.5)
    rows = np.array([49, 0, 17, 17, 3])
    part, pmag = orc.sgemm_f64(A, B, C, 1.5, 0.5, rows=rows)
    assert np.array_equal(part, full[rows]) and np.array_equal(pmag, fmag[rows])


ALL_PINS = [
    pin_alpha1_beta0_int64,
    pin_bruteforce_tiny,
    pin_identity,
    pin_permutation,
    pin_alpha_zero,
    pin_beta_zero_no_read,
    pin_integer_padded,
    pin_library_crosscheck,
    pin_rows_subset,
]
