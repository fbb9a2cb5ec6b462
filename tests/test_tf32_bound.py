"""The TF32 mode's error bounds, against a CPU emulation of its input rounding.

`tcgen05.mma .kind::tf32` reads each FP32 operand as TF32: sign, 8 exponent bits
and 10 explicit mantissa bits, that is an FP32 pattern with its low 13 bits gone
(PTX ISA, "Warp Level Matrix Multiply-Accumulate Instructions", TF32 format).
Dropping them (truncation) or rounding them to nearest changes each input by less
than 2^-10 (truncation) or 2^-11 (nearest) of its value, so a product is off by at
most 2^-9 + 2^-20 of its magnitude. The FP32 accumulation adds at most (K + 2)
2^-24. The GPU TF32 tests use that sum, (2^-9 + 2^-20 + (K+2) 2^-24) * mag, beside
the stated (K + 2) 2^-10 * mag.

Here both rounding forms are applied to the operands on the CPU, and the products
are summed exactly (FP64 over FP32 values). This checks three things:
- both bounds hold;
- the tighter bound is not vacuous: same-signed inputs reach a third of it;
- integer operands in {-2..2}, which the bit-exact TF32 tests use, pass through TF32
  unchanged.
"""

import numpy as np

import oracle
from dense_fp32_gemm_04_gb300 import inputs

LOW13 = np.uint32(0xFFFFE000)


def tf32_truncate(x: np.ndarray) -> np.ndarray:
    return (x.astype(np.float32).view(np.uint32) & LOW13).view(np.float32)


def tf32_nearest(x: np.ndarray) -> np.ndarray:
    """Round to nearest, ties to even, at bit 13 (finite inputs far from overflow)."""
    u = x.astype(np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0xFFF + ((u >> 13) & 1)) & 0xFFFFE000
    return u.astype(np.uint32).view(np.float32)


def tight_bound(K, mag):
    return (2.0**-9 + 2.0**-20 + (K + 2) * 2.0**-24) * mag


def _emulate(rounding, A, B, C, alpha, beta):
    prod = rounding(A).astype(np.float64) @ rounding(B).astype(np.float64)
    out = alpha * prod
    if beta != 0.0:
        out = out + beta * C.astype(np.float64)
    return out


def test_rounding_helpers_keep_ten_mantissa_bits():
    x = np.array([1.0, 1.0 + 2.0**-10, 1.0 + 2.0**-11, 1.0 + 3 * 2.0**-11, -(1.0 + 2.0**-10 + 2.0**-12)],
                 dtype=np.float32)
    assert tf32_truncate(x).tolist() == [1.0, 1.0 + 2.0**-10, 1.0, 1.0 + 2.0**-10, -(1.0 + 2.0**-10)]
    # ties go to the even mantissa: 1 + 2^-11 -> 1, 1 + 3 * 2^-11 -> 1 + 2^-9
    assert tf32_nearest(x).tolist() == [1.0, 1.0 + 2.0**-10, 1.0, 1.0 + 2.0**-9, -(1.0 + 2.0**-10)]


def test_integer_operands_pass_through_tf32_unchanged():
    A, B, C = inputs.problem_operands(M=33, N=40, K=70, seed=5, dist=("int", "int", "int"))
    for x in (A, B, C):
        assert np.array_equal(tf32_truncate(x), x) and np.array_equal(tf32_nearest(x), x)


def test_both_bounds_hold_and_the_tight_one_is_reached():
    M, N, K = 64, 48, 1024
    A, B, C = inputs.problem_operands(M=M, N=N, K=K, seed=21, dist=("uniform", "uniform", "uniform"))
    # same-signed operands: the truncation errors add up instead of cancelling
    A, B = np.abs(A), np.abs(B)
    ref, mag = oracle.sgemm_f64(A, B, C, 1.0, 0.0)
    worst = {}
    for rounding in (tf32_truncate, tf32_nearest):
        err = np.abs(_emulate(rounding, A, B, C, 1.0, 0.0) - ref)
        assert np.all(err <= oracle.bound(K, mag, oracle.U_TF32)), rounding.__name__
        assert np.all(err <= tight_bound(K, mag)), rounding.__name__
        worst[rounding.__name__] = float(np.max(err / tight_bound(K, mag)))
    assert worst["tf32_truncate"] >= 0.25, worst
    # the FP32 bound alone would be exceeded ten times over: the input rounding dominates
    assert worst["tf32_truncate"] * tight_bound(K, 1.0) > 10 * oracle.bound(K, 1.0, oracle.U_FP32)


def test_signed_operands_with_beta():
    M, N, K = 50, 70, 300
    A, B, C = inputs.problem_operands(M=M, N=N, K=K, seed=22, dist=("normal", "uniform", "uniform"))
    ref, mag = oracle.sgemm_f64(A, B, C, 1.5, 0.5)
    for rounding in (tf32_truncate, tf32_nearest):
        err = np.abs(_emulate(rounding, A, B, C, 1.5, 0.5) - ref)
        assert np.all(err <= tight_bound(K, mag)), rounding.__name__
