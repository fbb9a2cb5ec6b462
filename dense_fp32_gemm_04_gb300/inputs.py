"""Seeded synthetic inputs for the SGEMM problems (shared by tests, bench and oracle checks).

This module holds no GEMM arithmetic. It only turns (seed, matrix tag, element
index) into a float, so both the CUDA path and the FP64 oracle can be fed the
same operands without either one producing the other's inputs.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014; the 64-bit finaliser constants are Vigna's
public-domain splitmix64.c). It is used in counter form: draw number ``c`` of a
stream started at state ``seed`` is ``mix(seed + (c + 1) * GAMMA)``, which is
exactly the c-th output of the sequential generator. Matrix ``tag`` (A=0, B=1,
C=2) owns the counter range ``[tag << 48, (tag + 1) << 48)``, and element ``e``
of a row-major ``rows x cols`` matrix (packed index ``e = i * cols + j``,
independent of any leading dimension) uses counters ``tag << 48 | (e * d + t)``
for its ``d`` draws ``t = 0..d-1``.

Distributions (the pages name none; these are this library's readings):

* ``uniform``: ``(u >> 40) * 2**-23 - 1``, 24 random bits, values in [-1, 1)
  on a 2**-23 grid, every one exactly representable in FP32.
* ``normal``: Box-Muller from two 53-bit uniforms, computed in float64 and
  rounded once to FP32 (one normal per element, two draws).
* ``int``: integers in {-2, -1, 0, 1, 2} by Lemire's multiply-shift on the top
  32 bits (``((u >> 32) * 5) >> 32``); bias below 2**-32.
"""

from __future__ import annotations

import concurrent.futures
import os

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

TAG_A, TAG_B, TAG_C = 0, 1, 2
_CHUNK = 1 << 20  # elements generated per numpy pass (bounds temporaries)
_WORKERS = max(1, min(16, os.cpu_count() or 1))


def mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output finaliser on a uint64 array (wrapping arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def draws(seed: int, counters: np.ndarray) -> np.ndarray:
    """Outputs number ``counters`` (0-based) of the SplitMix64 stream started at ``seed``."""
    c = np.asarray(counters, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + (c + np.uint64(1)) * GAMMA
    return mix64(z)


def _fill(seed: int, tag: int, rows: int, cols: int, per_elem: int, convert) -> np.ndarray:
    n = rows * cols
    out = np.empty(n, dtype=np.float32)
    base = np.uint64(tag) << np.uint64(48)

    def chunk(lo):
        hi = min(n, lo + _CHUNK)
        e = np.arange(lo, hi, dtype=np.uint64)
        if per_elem == 1:
            out[lo:hi] = convert(draws(seed, base | e))
        else:
            d0 = draws(seed, base | (e * np.uint64(2)))
            d1 = draws(seed, base | (e * np.uint64(2) + np.uint64(1)))
            out[lo:hi] = convert(d0, d1)

    starts = range(0, n, _CHUNK)
    if n > 4 * _CHUNK and _WORKERS > 1:
        # Chunks are independent (counter-based draws), so threads change nothing but speed.
        with concurrent.futures.ThreadPoolExecutor(_WORKERS) as ex:
            list(ex.map(chunk, starts))
    else:
        for lo in starts:
            chunk(lo)
    return out.reshape(rows, cols)


def _to_uniform(u: np.ndarray) -> np.ndarray:
    return ((u >> np.uint64(40)).astype(np.float64) * 2.0**-23 - 1.0).astype(np.float32)


def _to_normal(u0: np.ndarray, u1: np.ndarray) -> np.ndarray:
    r1 = ((u0 >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0**-53  # (0, 1]
    r2 = (u1 >> np.uint64(11)).astype(np.float64) * 2.0**-53          # [0, 1)
    return (np.sqrt(-2.0 * np.log(r1)) * np.cos(2.0 * np.pi * r2)).astype(np.float32)


def _to_int(u: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        k = ((u >> np.uint64(32)) * np.uint64(5)) >> np.uint64(32)
    return (k.astype(np.int64) - 2).astype(np.float32)


def matrix(seed: int, tag: int, rows: int, cols: int, dist: str) -> np.ndarray:
    """A packed row-major float32 ``rows x cols`` matrix from the given distribution."""
    if rows < 0 or cols < 0:
        raise ValueError("negative matrix shape")
    if dist == "uniform":
        return _fill(seed, tag, rows, cols, 1, _to_uniform)
    if dist == "normal":
        return _fill(seed, tag, rows, cols, 2, _to_normal)
    if dist == "int":
        return _fill(seed, tag, rows, cols, 1, _to_int)
    if dist == "zero":
        return np.zeros((rows, cols), dtype=np.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def with_ld(x: np.ndarray, ld: int, fill: float = np.nan) -> np.ndarray:
    """Embed a packed matrix in a buffer of row stride ``ld`` (pad columns set to ``fill``).

    Returns the full ``rows x ld`` buffer; the logical matrix is ``buf[:, :cols]``.
    """
    rows, cols = x.shape
    if ld < max(1, cols):
        raise ValueError("ld smaller than the column count")
    buf = np.full((rows, ld), fill, dtype=np.float32)
    buf[:, :cols] = x
    return buf


# The problems the benchmarks and parity tests are quoted on: operand shapes,
# scalars, seeds and distributions (A, B, C).
PROBLEMS = {
    "square256": dict(M=256, N=256, K=256, alpha=1.0, beta=0.0, seed=0,
                      dist=("uniform", "uniform", "zero")),
    "square4096": dict(M=4096, N=4096, K=4096, alpha=1.5, beta=0.5, seed=1,
                       dist=("uniform", "uniform", "uniform")),
    "square4096_int": dict(M=4096, N=4096, K=4096, alpha=1.5, beta=0.5, seed=1,
                           dist=("int", "int", "zero")),
    "ragged": dict(M=2047, N=3001, K=1531, alpha=1.0, beta=1.0, seed=2,
                   dist=("normal", "normal", "uniform")),
    "ragged_int": dict(M=2047, N=3001, K=1531, alpha=1.0, beta=1.0, seed=2,
                       dist=("int", "int", "int")),
    "skinny_tall": dict(M=16384, N=64, K=8192, alpha=1.0, beta=0.0, seed=4,
                        dist=("uniform", "uniform", "zero")),
    "skinny_wide": dict(M=64, N=16384, K=8192, alpha=1.0, beta=0.0, seed=4,
                        dist=("uniform", "uniform", "zero")),
}
for _n in (512, 1024, 2048, 8192, 16384):
    PROBLEMS[f"sweep{_n}"] = dict(M=_n, N=_n, K=_n, alpha=1.0, beta=0.0, seed=3,
                                  dist=("uniform", "uniform", "zero"))


def problem_operands(name: str = None, **spec):
    """(A, B, C) packed float32 operands of a named problem (or an explicit spec)."""
    p = dict(PROBLEMS[name]) if name is not None else {}
    p.update(spec)
    M, N, K, seed = p["M"], p["N"], p["K"], p["seed"]
    da, db, dc = p["dist"]
    A = matrix(seed, TAG_A, M, K, da)
    B = matrix(seed, TAG_B, K, N, db)
    C = matrix(seed, TAG_C, M, N, dc)
    return A, B, C
