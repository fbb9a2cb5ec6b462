"""Shared helpers of the GPU parity tests: run the library through its C ABI on
seeded operands, and compare with the FP64 oracle."""

from __future__ import annotations

import functools

import numpy as np

import oracle
from dense_fp32_gemm_04_gb300 import inputs

CANARY = np.float32(-7.0e30)  # written around and between the rows of C; must survive


def device_buffer(torch, x: np.ndarray, ld: int = None, offset: int = 0, guard: int = 64):
    """Copy a packed matrix into a device buffer with row stride ``ld``.

    The buffer has ``guard`` canary floats before and after the matrix and
    canaries in the pad columns; ``offset`` extra floats shift the matrix start
    (offset % 4 != 0 makes the pointer not 16-byte aligned). Returns
    (buffer, pointer, ld, view-extractor).
    """
    rows, cols = x.shape
    ld = max(1, cols) if ld is None else ld
    n = guard + offset + rows * ld + guard
    host = np.full(n, CANARY, dtype=np.float32)
    start = guard + offset
    if rows and cols:
        body = host[start:start + rows * ld].reshape(rows, ld)
        body[:, :cols] = x
    buf = torch.from_numpy(host).cuda()
    ptr = buf.data_ptr() + 4 * start

    def extract(dev_buf):
        h = dev_buf.cpu().numpy()
        mat = h[start:start + rows * ld].reshape(rows, ld)[:, :cols] if rows else np.zeros((0, cols), np.float32)
        pads_ok = True
        if rows and ld > cols:
            pads_ok = bool(np.all(h[start:start + rows * ld].reshape(rows, ld)[:, cols:] == CANARY))
        guards_ok = bool(np.all(h[:start] == CANARY) and np.all(h[start + rows * ld:] == CANARY))
        return mat.copy(), pads_ok and guards_ok

    return buf, ptr, ld, extract


def run_gemm(torch, h, A, B, C, alpha, beta, lds=(None, None, None), offsets=(0, 0, 0), stream=None):
    """C_out of the library for packed operands (placed with the given ld / offsets).

    Returns (C_out, guards_intact, status).
    """
    M, K = A.shape
    N = B.shape[1]
    bA, pA, lda, _ = device_buffer(torch, A, lds[0], offsets[0])
    bB, pB, ldb, _ = device_buffer(torch, B, lds[1], offsets[1])
    bC, pC, ldc, ext = device_buffer(torch, C, lds[2], offsets[2])
    st = h.run_ptr(M, N, K, alpha, pA, lda, pB, ldb, beta, pC, ldc, stream)
    torch.cuda.synchronize()
    out, guards = ext(bC)
    return out, guards, st


@functools.lru_cache(maxsize=2)
def problem_reference(name: str):
    """FP64 oracle result and bound magnitude over all of C for one configured problem.

    Kept for the two most recent problems, so the FP32 and TF32 tests of the
    4096^3 problems share one oracle run per problem (a few seconds on all host
    threads each)."""
    p = inputs.PROBLEMS[name]
    A, B, C = inputs.problem_operands(name)
    return oracle.sgemm_f64(A, B, C, p["alpha"], p["beta"])


def check_against_oracle(got, A, B, C, alpha, beta, rows=None, exact=False, u=oracle.U_FP32, ref=None):
    """Assert the FP32 bound (and bit-exactness when ``exact``) on all or selected rows.

    ``ref`` is an already computed ``(ref, mag)`` pair over all of C (see
    ``problem_reference``); otherwise the oracle runs here."""
    K = A.shape[1]
    if ref is not None:
        assert rows is None
        ref, mag = ref
    else:
        ref, mag = oracle.sgemm_f64(A, B, C, alpha, beta, rows=rows)
    g = got if rows is None else got[rows]
    ok, worst, nbad = oracle.check(g, ref, mag, K, u)
    assert ok, f"{nbad} elements outside the bound (worst ratio {worst:.3g})"
    if exact:
        assert oracle.exact(g, ref), "integer-valued problem is not bit-exact"
    return worst


def sample_rows(M: int, bm: int = 128, n_random: int = 64, seed: int = 12345):
    """Rows to check on large problems: the edges of the first two and last two tile rows plus seeded random rows."""
    rows = {0, 1, M - 1, M - 2}
    last = (M - 1) // bm * bm
    for t in {0, bm, max(0, last - bm), last}:
        rows.update((t, t + 1, min(M - 1, t + bm - 1), min(M - 1, t + bm)))
    rnd = inputs.draws(seed, np.arange(n_random)) % np.uint64(max(M, 1))
    rows.update(int(r) for r in rnd)
    rows = sorted(r for r in rows if 0 <= r < M)
    return np.array(rows, dtype=np.int64)
