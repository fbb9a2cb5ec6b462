"""Handles running at the same time on different streams.

Three handles (FP32, TF32 on one CTA per tile, TF32 on CTA pairs) each queue
several calls on their own stream before anything is synchronised, so their
persistent grids compete for SMs. Nothing of one handle (workspace, status
word, plan) may leak into another, and no kernel depends on another CTA of its
grid being resident, so every result must equal that handle's result when run
alone: bit for bit, and exact on integer operands.
"""

import numpy as np
import pytest

import dense_fp32_gemm_04_gb300 as sg
import oracle
from dense_fp32_gemm_04_gb300 import inputs

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

MODES = (("fp32", None), ("tf32_one_cta", 0), ("tf32_cta_pair", 1))
SHAPES = ((1024, 1024, 1024), (777, 1300, 513), (2048, 512, 1024))


@pytest.fixture(scope="module")
def handles():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_fp32_gemm_04_gb300 import _build

    _build.build()
    hs = {}
    for name, kernel in MODES:
        h = sg.Sgemm(0)
        if kernel is not None:
            h.set_math_mode(sg.MATH_TF32)
            h.set_option(sg.OPT_FORCE_TF32_KERNEL, kernel)
        hs[name] = h
    yield hs
    for h in hs.values():
        h.close()


def _operands(shape, seed):
    M, N, K = shape
    A, B, C = inputs.problem_operands(M=M, N=N, K=K, seed=seed, dist=("int", "int", "int"))
    return A, B, C, tuple(torch.from_numpy(x).cuda() for x in (A, B, C))


def test_concurrent_handles_match_serial_runs(handles):
    problems = [_operands(s, 500 + i) for i, s in enumerate(SHAPES)]
    # serial reference per handle
    serial = {}
    for name, h in handles.items():
        for i, (A, B, C, (dA, dB, dC)) in enumerate(problems):
            out = dC.clone()
            h.run(dA, dB, out, 1.5, 0.5)
            torch.cuda.synchronize()
            assert h.check_device_status() == (sg.SGEMM_OK, 0), (name, i)
            serial[name, i] = out.cpu().numpy()
    # every handle on its own stream, all calls queued before any synchronisation
    streams = {name: torch.cuda.Stream() for name in handles}
    outs = {}
    torch.cuda.synchronize()
    for rep in range(3):
        for i, (A, B, C, (dA, dB, dC)) in enumerate(problems):
            for name, h in handles.items():
                with torch.cuda.stream(streams[name]):
                    out = dC.clone()
                    h.run(dA, dB, out, 1.5, 0.5, stream=streams[name])
                outs[name, i, rep] = out
    torch.cuda.synchronize()
    for name, h in handles.items():
        assert h.check_device_status() == (sg.SGEMM_OK, 0), name
    for (name, i, rep), out in outs.items():
        got = out.cpu().numpy()
        assert np.array_equal(got.view(np.uint32), serial[name, i].view(np.uint32)), (name, i, rep)
    for i, (A, B, C, _) in enumerate(problems):
        ref, _ = oracle.sgemm_f64(A, B, C, 1.5, 0.5)
        for name, _ in MODES:
            assert oracle.exact(serial[name, i], ref), (name, i)
