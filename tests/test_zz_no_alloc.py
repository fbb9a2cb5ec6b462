"""sgemm_run_splitk_static: the split-K SGEMM entry point that allocates nothing.

It exists for callers that cannot call cudaMalloc (code inside another
runtime's memory pool, latency-sensitive loops that cannot take the implicit
device synchronization of cudaMalloc/cudaFree): its split-K partials live in a
32 MiB file-scope static device array instead of a handle workspace.

The test calls it through the C ABI twice in a row on different problems (the
second call reuses the array the first one left behind) and compares each
result with the existing entry point sgemm_run on the same operands and split
factor, within the FP32 error bound the other parity tests use. This file is
named so pytest collects it last.
"""

import ctypes

import numpy as np
import pytest

import dense_fp32_gemm_04_gb300 as sg
import oracle
from dense_fp32_gemm_04_gb300 import inputs

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
