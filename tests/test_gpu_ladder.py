"""The pages' kernel ladder (context kernels, include/sgemm_ladder.h) against the oracle."""

import numpy as np
import pytest

import dense_fp32_gemm_04_gb300 as sg
import oracle
from dense_fp32_gemm_04_gb300 import inputs

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_fp32_gemm_04_gb300 import _build

    _build.build()


def _run(rung, A, B, C, alpha, beta):
    dA, dB, dC = (torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in (A, B, C))
    st = sg.ladder_run(rung, dA, dB, dC, alpha, beta)
    torch.cuda.synchronize()
    return st, dC.cpu().numpy()


@pytest.mark.parametrize("rung", range(1, 9))
def test_rung_parity(rung):
    shapes = [(1, 4, 4), (33, 68, 40), (130, 260, 100), (256, 256, 256)] if rung >= 6 else \
             [(1, 1, 1), (33, 65, 17), (130, 257, 99), (256, 256, 256)]
    for (M, N, K) in shapes:
        A, B, C = inputs.problem_operands(M=M, N=N, K=K, seed=rung * 7 + M, dist=("int", "int", "int"))
        st, got = _run(rung, A, B, C, 1.5, 0.5)
        assert st == sg.SGEMM_OK, (rung, M, N, K)
        ref, mag = oracle.sgemm_f64(A, B, C, 1.5, 0.5)
        assert oracle.exact(got, ref), (rung, M, N, K)
        Ar, Br, Cr = inputs.problem_operands(M=M, N=N, K=K, seed=rung, dist=("normal", "uniform", "uniform"))
        st, got = _run(rung, Ar, Br, Cr, 1.0, 0.0)
        ref, mag = oracle.sgemm_f64(Ar, Br, Cr, 1.0, 0.0)
        assert oracle.check(got, ref, mag, K)[0], (rung, M, N, K)


def test_vector_rungs_reject_unaligned_shapes():
    A, B, C = inputs.problem_operands(M=16, N=16, K=15, seed=1, dist=("int", "int", "int"))
    for rung in (6, 7, 8):
        st, got = _run(rung, A, B, C, 1.0, 0.0)
        assert st == sg.SGEMM_ERR_NOT_SUPPORTED
        assert np.array_equal(got, C)
    for rung in (0, 9):
        st, _ = _run(rung, A, B, C, 1.0, 0.0)
        assert st == sg.SGEMM_ERR_INVALID_VALUE
