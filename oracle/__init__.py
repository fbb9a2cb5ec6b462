"""FP64 CPU oracle for C = alpha*A*B + beta*C — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference arm may import this package. The GPU library never does.

The arithmetic lives in ``sgemm_oracle.c`` (plain C, FP64 accumulation, i-k-j
loop; see its header for the passages it follows). This module only builds
that file with gcc, marshals numpy arrays into it, and states the error bound
the GPU result is held to:

    |C_gpu - C_ref64| <= (K + 2) * u * (|alpha| sum_k |a_ik||b_kj| + |beta||c_ij|)

with u = 2**-24 for the FP32 path and u = 2**-10 for the flagged TF32 mode.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sgemm_oracle.c")
_LIB = os.path.join(_HERE, "libsgemm_oracle.so")
_lock = threading.Lock()
_lib = None

U_FP32 = 2.0**-24
U_TF32 = 2.0**-10


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libsgemm_oracle.so`` (OpenMP when available)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-std=c11", _SRC, "-o", _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


class Oracle:
    """ctypes view of one build of ``sgemm_oracle.c`` (the default build, or a test's mutant)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        f64 = lib.oracle_sgemm_f64
        f64.restype = ctypes.c_int
        f64.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                        ctypes.c_void_p, ctypes.c_longlong,
                        ctypes.c_void_p, ctypes.c_longlong,
                        ctypes.c_float, ctypes.c_void_p, ctypes.c_longlong,
                        ctypes.c_void_p, ctypes.c_int,
                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        f32 = lib.oracle_sgemm_f32_ijk
        f32.restype = ctypes.c_int
        f32.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                        ctypes.c_void_p, ctypes.c_longlong,
                        ctypes.c_void_p, ctypes.c_longlong,
                        ctypes.c_float, ctypes.c_void_p, ctypes.c_longlong,
                        ctypes.c_void_p]
        lib.oracle_max_threads.restype = ctypes.c_int
        self._lib = lib

    def max_threads(self) -> int:
        return int(self._lib.oracle_max_threads())

    def sgemm_f64(self, A, B, C, alpha: float, beta: float, M=None, N=None, K=None,
                  rows=None, with_mag: bool = True, nthreads: int = 0):
        """Reference result (and bound magnitude) in float64.

        ``A``, ``B``, ``C`` are 2-D float32 arrays (views with a row stride
        larger than their width are allowed: that stride is the leading
        dimension). ``rows`` restricts the output to those row indices. Returns
        ``(out, mag)``, each ``len(rows) x N`` (or ``M x N``); ``mag`` is None
        when ``with_mag`` is False.
        """
        M = A.shape[0] if M is None else M
        K = A.shape[1] if K is None else K
        N = B.shape[1] if N is None else N
        # Operands are passed as given; whether C (beta == 0) or A, B (alpha == 0)
        # are read is decided in the C code, which the pins check with NaN fills.
        pa, lda = _operand(A, M, K, "A")
        pb, ldb = _operand(B, K, N, "B")
        pc, ldc = _operand(C, M, N, "C")
        if rows is not None:
            rows = np.ascontiguousarray(rows, dtype=np.int32)
            R = rows.shape[0]
        else:
            R = M
        out = np.empty((R, N), dtype=np.float64)
        mag = np.empty((R, N), dtype=np.float64) if with_mag else None
        rc = self._lib.oracle_sgemm_f64(M, N, K, ctypes.c_float(alpha), pa, lda, pb, ldb,
                                        ctypes.c_float(beta), pc, ldc,
                                        rows.ctypes.data if rows is not None else None,
                                        R, out.ctypes.data,
                                        mag.ctypes.data if mag is not None else None, nthreads)
        if rc != 0:
            raise ValueError("oracle_sgemm_f64 rejected its arguments")
        return out, mag

    def sgemm_f32_ijk(self, A, B, C, alpha: float, beta: float):
        """The pages' FP32 i-j-k ground truth (float accumulator), generalised to alpha/beta."""
        M, K = A.shape
        N = B.shape[1]
        pa, lda = _operand(A, M, K, "A")
        pb, ldb = _operand(B, K, N, "B")
        pc, ldc = _operand(C, M, N, "C")
        out = np.empty((M, N), dtype=np.float32)
        rc = self._lib.oracle_sgemm_f32_ijk(M, N, K, ctypes.c_float(alpha), pa, lda, pb, ldb,
                                            ctypes.c_float(beta), pc, ldc, out.ctypes.data)
        if rc != 0:
            raise ValueError("oracle_sgemm_f32_ijk rejected its arguments")
        return out


def _default() -> Oracle:
    global _lib
    with _lock:
        if _lib is None:
            _lib = Oracle(build())
    return _lib


def _operand(x, rows, cols, name):
    """Pointer and leading dimension of a row-major float32 view (unit column stride)."""
    if x is None:
        return None, max(1, cols)
    if x.dtype != np.float32 or x.ndim != 2:
        raise TypeError(f"{name} must be a 2-D float32 array")
    if x.shape[0] < rows or x.shape[1] < cols:
        raise ValueError(f"{name} is smaller than {rows} x {cols}")
    if rows > 0 and cols > 0 and x.strides[1] != 4:
        raise ValueError(f"{name} must have unit column stride")
    ld = x.strides[0] // 4 if x.shape[0] > 1 else max(1, x.shape[1])
    return x.ctypes.data, ld


def max_threads() -> int:
    return _default().max_threads()


def sgemm_f64(*args, **kwargs):
    """See :meth:`Oracle.sgemm_f64` (default build)."""
    return _default().sgemm_f64(*args, **kwargs)


def sgemm_f32_ijk(*args, **kwargs):
    """See :meth:`Oracle.sgemm_f32_ijk` (default build)."""
    return _default().sgemm_f32_ijk(*args, **kwargs)


def min2(values):
    """The two smallest entries of a matrix and their (row, column).

    The pages' follow-up task ("SGEMM CUDA kernel (First Half)", Additionally
    Required: the two minimums of the product C and their 2D indices), taken as
    a total order on (value, row-major position): equal values are ordered by
    the smaller row-major index. Returns ``(vals, rows, cols)`` of length 2; a
    matrix with one element reports (+inf, -1, -1) second.
    """
    v = np.asarray(values, dtype=np.float64)
    M, N = v.shape
    flat = v.reshape(-1)
    order = np.lexsort((np.arange(flat.size), flat))  # by value, then position
    vals, rows, cols = [], [], []
    for t in range(2):
        if t < flat.size:
            e = int(order[t])
            vals.append(float(flat[e]))
            rows.append(e // N)
            cols.append(e % N)
        else:
            vals.append(float("inf"))
            rows.append(-1)
            cols.append(-1)
    return vals, rows, cols


def bound(K: int, mag, u: float = U_FP32):
    """Elementwise error bound (K + 2) * u * mag."""
    return (K + 2) * u * mag


def check(got, ref, mag, K: int, u: float = U_FP32):
    """Return (ok, worst_ratio, n_bad) for a float32 result against the FP64 reference.

    NaN or Inf in ``got`` always fails. ``worst_ratio`` is max |err| / bound
    (0/0 counted as 0).
    """
    got64 = np.asarray(got, dtype=np.float64)
    err = np.abs(got64 - ref)
    b = bound(K, mag, u)
    finite = np.isfinite(got64)
    bad = (err > b) | ~finite
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(b > 0, err / b, np.where(err > 0, np.inf, 0.0))
    worst = float(np.max(ratio)) if ratio.size else 0.0
    return (not bad.any()), worst, int(bad.sum())


def exact(got, ref) -> bool:
    """Bit-exact comparison after rounding the FP64 reference to FP32 (+0 == -0)."""
    return bool(np.array_equal(np.asarray(got, dtype=np.float32), ref.astype(np.float32)))
