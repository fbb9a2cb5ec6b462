"""CUDA graph capture of library calls.

A handle whose workspace was sized beforehand (sgemm_reserve with the plan's
workspace_bytes) can be captured into a CUDA graph: the capture runs nothing,
and every replay gives bit for bit the result of the same call run eagerly.
Covers the split-K path (two launches), the transposed-A + stream-K path
(three launches, programmatic dependent launch between them), two minima of C,
and the TF32 mode on CTA pairs (cluster launch). A capture that would have to
grow the workspace is refused with SGEMM_ERR_NOT_SUPPORTED and captures nothing.
"""

import numpy as np
import pytest

import dense_fp32_gemm_04_gb300 as sg
import oracle
from dense_fp32_gemm_04_gb300 import inputs

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

CASES = [
    ((512, 512, 512), sg.MATH_FP32),      # split-K + reduction
    ((1000, 2500, 513), sg.MATH_FP32),    # A^T + stream-K + reduction
    ((777, 1300, 513), sg.MATH_TF32),     # TF32 on CTA pairs
]


@pytest.fixture(scope="module")
def num_sms():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_fp32_gemm_04_gb300 import _build

    _build.build()
    return torch.cuda.get_device_properties(0).multi_processor_count


def _operands(M, N, K, seed):
    A, B, C = inputs.problem_operands(M=M, N=N, K=K, seed=seed, dist=("int", "int", "int"))
    return A, B, C, tuple(torch.from_numpy(x).cuda() for x in (A, B, C))


@pytest.mark.parametrize("shape,mode", CASES)
def test_graph_replay_matches_eager(num_sms, shape, mode):
    M, N, K = shape
    A, B, C, (dA, dB, dC) = _operands(M, N, K, seed=M + N)
    h = sg.Sgemm(0)
    try:
        h.set_math_mode(mode)
        plan = sg.plan(M, N, K, num_sms=num_sms, math_mode=mode)
        h.reserve(2 * plan.workspace_bytes)  # the plan on this handle may differ in detail
        out = dC.clone()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            st = h.run_ptr(M, N, K, 1.5, dA.data_ptr(), K, dB.data_ptr(), N, 0.5, out.data_ptr(), N, s)
        assert st == sg.SGEMM_OK
        torch.cuda.synchronize()
        assert torch.equal(out, dC), "the capture itself must not run the GEMM"
        eager = dC.clone()
        h.run(dA, dB, eager, 1.5, 0.5)
        torch.cuda.synchronize()
        ref = eager.cpu().numpy()
        for _ in range(3):
            out.copy_(dC)
            g.replay()
            torch.cuda.synchronize()
            assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))
        assert h.check_device_status() == (sg.SGEMM_OK, 0)
        want, _ = oracle.sgemm_f64(A, B, C, 1.5, 0.5)
        assert oracle.exact(ref, want)
    finally:
        h.close()


def test_graph_of_min2(num_sms):
    M, N, K = 900, 700, 300
    A, B, C, (dA, dB, dC) = _operands(M, N, K, seed=77)
    h = sg.Sgemm(0)
    try:
        h.reserve(2 * sg.plan(M, N, K, num_sms=num_sms).workspace_bytes)
        out = dC.clone()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            vals, ij = h.run_min2(dA, dB, out, 1.5, 0.5, stream=s)
        out.copy_(dC)
        g.replay()
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        want, _ = oracle.sgemm_f64(A, B, C, 1.5, 0.5)
        assert oracle.exact(got, want)
        flat = np.sort(got.ravel())
        assert vals.cpu().numpy().tolist() == flat[:2].tolist()
        i = ij.cpu().numpy()
        assert got[i[0], i[1]] == flat[0] and got[i[2], i[3]] == flat[1] and (i[0], i[1]) != (i[2], i[3])
    finally:
        h.close()


def test_capture_that_needs_a_larger_workspace_is_refused(num_sms):
    M, N, K = 1000, 2500, 513  # A^T and stream-K partials need workspace
    _, _, _, (dA, dB, dC) = _operands(M, N, K, seed=5)
    h = sg.Sgemm(0)  # fresh handle: no workspace yet
    try:
        out = dC.clone()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            st = h.run_ptr(M, N, K, 1.0, dA.data_ptr(), K, dB.data_ptr(), N, 0.0, out.data_ptr(), N, s)
            out.add_(0.0)  # keep the graph non-empty
        assert st == sg.SGEMM_ERR_NOT_SUPPORTED
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, dC)  # nothing of the GEMM was captured
        # outside a capture the same call grows the workspace and runs
        h.run(dA, dB, out, 1.0, 0.0)
        torch.cuda.synchronize()
        assert h.check_device_status() == (sg.SGEMM_OK, 0)
    finally:
        h.close()
