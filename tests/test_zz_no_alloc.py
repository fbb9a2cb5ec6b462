"""sgemm_run_splitk_static: the split-K SGEMM entry point that allocates nothing.

It exists for callers that cannot call cudaMalloc (code inside another
runtime's memory pool, latency-sensitive loops that cannot take the implicit
device synchronization of cudaMalloc/cudaFree): its split-K partials live in a
32 MiB file-scope static device array instead of a handle workspace.

The tests call it through the C ABI twice in a row on different problems (the
second call reuses the array the first one left behind) and compare each
result with the existing entry point sgemm_run on the same operands and split
factor, within the FP32 error bound the other parity tests use (bit-exact on
integer operands). Besides packed, aligned operands they cover operands that
are copied into the array first (row strides that are not a multiple of 4
floats, pointers one float off a 16-byte boundary), one split (C written by the
GEMM kernel itself, no partials), and the caller's status word: it is cleared
by every successful call, quick returns included. This file is named so pytest
collects it last.
"""

import ctypes

import numpy as np
import pytest

import dense_fp32_gemm_04_gb300 as sg
import oracle
from dense_fp32_gemm_04_gb300 import inputs
from gpu_helpers import device_buffer

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _device(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _run_both(h, M, N, K, alpha, beta, splits, seed):
    A, B, C = inputs.problem_operands(M=M, N=N, K=K, seed=seed, dist=("normal", "uniform", "uniform"))
    dA, dB = _device(A), _device(B)
    c_static = _device(C)
    c_handle = _device(C)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = sg.run_splitk_static(M, N, K, alpha, dA.data_ptr(), K, dB.data_ptr(), N, beta, c_static.data_ptr(), N,
                              splits, status.data_ptr())
    assert st == sg.SGEMM_OK, sg.status_string(st)
    h.set_option(sg.OPT_FORCE_SPLITS, splits)
    try:
        h.run(dA, dB, c_handle, alpha, beta)
    finally:
        h.set_option(sg.OPT_FORCE_SPLITS, 0)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got_static = c_static.cpu().numpy()
    got_handle = c_handle.cpu().numpy()
    # against the existing entry point, within the FP32 bound of the problem
    ref, mag = oracle.sgemm_f64(A, B, C, alpha, beta)
    diff = np.abs(got_static.astype(np.float64) - got_handle.astype(np.float64))
    assert np.all(np.isfinite(got_static))
    assert np.all(diff <= oracle.bound(K, mag))
    # and against the oracle itself
    assert oracle.check(got_static, ref, mag, K)[0]
    return got_static


def test_static_scratch_matches_sgemm_run_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_fp32_gemm_04_gb300 import _build

    _build.build()
    h = sg.Sgemm(0)
    try:
        # two calls in a row, different shapes and split factors, sharing the static scratch
        _run_both(h, 640, 384, 1024, 1.5, 0.5, 4, seed=31)
        _run_both(h, 333, 200, 777, -1.0, 2.0, 3, seed=32)
        # steady state: further calls do not change the device's free memory
        A, B, C = inputs.problem_operands(M=256, N=256, K=512, seed=33, dist=("int", "int", "int"))
        dA, dB, dC = _device(A), _device(B), _device(C)
        torch.cuda.synchronize()
        free0, _ = torch.cuda.mem_get_info()
        for _ in range(2):
            assert sg.run_splitk_static(256, 256, 512, 1.0, dA.data_ptr(), 512, dB.data_ptr(), 256, 0.0,
                                        dC.data_ptr(), 256, 5, None) == sg.SGEMM_OK
        torch.cuda.synchronize()
        free1, _ = torch.cuda.mem_get_info()
        assert free1 == free0
        ref, _ = oracle.sgemm_f64(A, B, None, 1.0, 0.0, with_mag=False)
        assert oracle.exact(dC.cpu().numpy(), ref)
    finally:
        h.close()


def test_static_scratch_rejects_oversized_problem():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_fp32_gemm_04_gb300 import _build

    _build.build()
    # 16 splits x 1024 x 1024 floats = 64 MiB of partials > 32 MiB: rejected before any launch
    M = N = 1024
    K = 4096
    dA = torch.zeros((M, K), device="cuda")
    dB = torch.zeros((K, N), device="cuda")
    dC = torch.full((M, N), 3.0, device="cuda")
    st = sg.run_splitk_static(M, N, K, 1.0, dA.data_ptr(), K, dB.data_ptr(), N, 0.0, dC.data_ptr(), N, 16, None)
    assert st == sg.SGEMM_ERR_NOT_SUPPORTED
    torch.cuda.synchronize()
    assert bool((dC == 3.0).all())
    # invalid arguments are still invalid
    assert sg.run_splitk_static(M, N, K, 1.0, dA.data_ptr(), K - 1, dB.data_ptr(), N, 0.0, dC.data_ptr(), N, 2,
                                None) == sg.SGEMM_ERR_INVALID_VALUE
    assert sg.run_splitk_static(M, N, K, 1.0, dA.data_ptr(), K, dB.data_ptr(), N, 0.0, dC.data_ptr(), N, 17,
                                None) == sg.SGEMM_ERR_INVALID_VALUE


STALE = 0x5A5A  # a status code left over from some earlier call of the caller's


def _status_word():
    return torch.full((1,), STALE, dtype=torch.int32, device="cuda")


def _placed_pair(h, M, N, K, alpha, beta, splits, seed, dist, lds, offsets):
    """Both entry points on the same placed operands (row strides ``lds``, pointer
    offsets ``offsets`` in floats); returns (static C, handle C, status after the
    static call, guards of both C buffers intact)."""
    A, B, C = inputs.problem_operands(M=M, N=N, K=K, seed=seed, dist=dist)
    bA, pA, lda, _ = device_buffer(torch, A, lds[0], offsets[0])
    bB, pB, ldb, _ = device_buffer(torch, B, lds[1], offsets[1])
    bCs, pCs, ldc, ext_s = device_buffer(torch, C, lds[2], offsets[2])
    bCh, pCh, _, ext_h = device_buffer(torch, C, lds[2], offsets[2])
    status = _status_word()
    st = sg.run_splitk_static(M, N, K, alpha, pA, lda, pB, ldb, beta, pCs, ldc, splits, status.data_ptr())
    assert st == sg.SGEMM_OK, sg.status_string(st)
    h.set_option(sg.OPT_FORCE_SPLITS, splits)
    try:
        assert h.run_ptr(M, N, K, alpha, pA, lda, pB, ldb, beta, pCh, ldc) == sg.SGEMM_OK
    finally:
        h.set_option(sg.OPT_FORCE_SPLITS, 0)
    torch.cuda.synchronize()
    got_s, guards_s = ext_s(bCs)
    got_h, guards_h = ext_h(bCh)
    return (A, B, C), got_s, got_h, int(status.item()), guards_s and guards_h


def _compare(ops, got_s, got_h, alpha, beta, exact):
    A, B, C = ops
    K = A.shape[1]
    ref, mag = oracle.sgemm_f64(A, B, C, alpha, beta)
    assert np.all(np.isfinite(got_s))
    diff = np.abs(got_s.astype(np.float64) - got_h.astype(np.float64))
    assert np.all(diff <= oracle.bound(K, mag))
    assert oracle.check(got_s, ref, mag, K)[0]
    if exact:
        assert oracle.exact(got_s, ref) and oracle.exact(got_h, ref)


@pytest.mark.parametrize("dist", [("int", "int", "int"), ("normal", "normal", "uniform")], ids=["int", "real"])
def test_static_scratch_unaligned_operands(dist):
    """Row strides K + 1 and N + 3 and pointers one float past a 16-byte boundary:
    A and B are first copied into aligned regions of the static array (after the
    partials' share of it), C is read and written in place with 4-byte accesses.
    Two calls in a row with different shapes and splits."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_fp32_gemm_04_gb300 import _build

    _build.build()
    h = sg.Sgemm(0)
    try:
        for (M, N, K, splits, seed, offs) in [(300, 260, 777, 4, 41, (1, 1, 3)), (129, 515, 1031, 3, 42, (1, 3, 1))]:
            ops, got_s, got_h, status, guards = _placed_pair(h, M, N, K, 1.5, -0.5, splits, seed, dist,
                                                             (K + 1, N + 3, N + 1), offs)
            assert guards and status == 0
            _compare(ops, got_s, got_h, 1.5, -0.5, exact=dist[0] == "int")
    finally:
        h.close()


def test_static_scratch_one_split():
    """splits = 1: the GEMM kernel writes C itself and the array holds no partials
    (aligned operands), then the same with operand copies in the array."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_fp32_gemm_04_gb300 import _build

    _build.build()
    h = sg.Sgemm(0)
    try:
        for (M, N, K, lds, offs) in [(384, 256, 640, (640, 256, 256), (0, 0, 0)),
                                     (211, 301, 333, (334, 304, 303), (1, 0, 2))]:
            for dist in (("int", "int", "int"), ("normal", "uniform", "uniform")):
                ops, got_s, got_h, status, guards = _placed_pair(h, M, N, K, 1.0, 1.0, 1, M + N, dist, lds, offs)
                assert guards and status == 0
                _compare(ops, got_s, got_h, 1.0, 1.0, exact=dist[0] == "int")
                # one split: one FMA chain per output in both entry points, so the same bits
                assert np.array_equal(got_s.view(np.uint32), got_h.view(np.uint32))
    finally:
        h.close()


def test_static_scratch_clears_callers_status_word():
    """A caller's status word holding an old code reads 0 after every successful
    call, the quick returns (M == 0; K == 0, which only scales C by beta) included,
    and an invalid call leaves it untouched."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_fp32_gemm_04_gb300 import _build

    _build.build()
    M, N, K = 96, 80, 200
    A, B, C = inputs.problem_operands(M=M, N=N, K=K, seed=44, dist=("int", "int", "int"))
    dA, dB, dC = _device(A), _device(B), _device(C)
    cases = [(M, N, K, 2), (0, N, K, 2), (M, N, 0, 2)]
    for (m, n, k, splits) in cases:
        status = _status_word()
        c0 = dC.clone()
        st = sg.run_splitk_static(m, n, k, 1.0, dA.data_ptr(), K, dB.data_ptr(), N, 2.0, dC.data_ptr(), N, splits,
                                  status.data_ptr())
        assert st == sg.SGEMM_OK, sg.status_string(st)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, (m, n, k)
        if k == 0 and m > 0:
            assert torch.equal(dC, 2.0 * c0)  # C = beta * C
        elif m == 0:
            assert torch.equal(dC, c0)
        else:
            ref, _ = oracle.sgemm_f64(A, B, c0.cpu().numpy(), 1.0, 2.0, with_mag=False)
            assert oracle.exact(dC.cpu().numpy(), ref)
    status = _status_word()
    assert sg.run_splitk_static(M, N, K, 1.0, dA.data_ptr(), K - 1, dB.data_ptr(), N, 0.0, dC.data_ptr(), N, 2,
                                status.data_ptr()) == sg.SGEMM_ERR_INVALID_VALUE
    torch.cuda.synchronize()
    assert int(status.item()) == STALE
