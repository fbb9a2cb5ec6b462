"""The kernels' bounded waits: a stage that is never filled ends the launch with
SGEMM_ERR_TIMEOUT (no trap, no hang) and the GPU stays usable afterwards.

The missing fill is made on purpose by the test-only option SGEMM_OPT_INJECT_SKIP:
CTA 0's producer skips one stage, so its consumers' wait runs out after the short
limit set here. Nothing faults; the kernel returns on its own.
"""

import numpy as np
import pytest

import dense_fp32_gemm_04_gb300 as sg
from dense_fp32_gemm_04_gb300 import inputs
from gpu_helpers import check_against_oracle, run_gemm

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.mark.parametrize("ta", [0, 1, 2])
def test_timeout_is_reported_and_gpu_recovers(ta):
    """Each A layout: with A transposed in shared memory the transposer warp waits
    for the missing stage too, and whichever wait runs out first reports."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_fp32_gemm_04_gb300 import _build

    _build.build()
    h = sg.Sgemm(0)
    try:
        M, N, K = 256, 256, 512
        A, B, C = inputs.problem_operands(M=M, N=N, K=K, seed=2, dist=("int", "int", "int"))
        h.set_option(sg.OPT_FORCE_CONFIG, 0)
        h.set_option(sg.OPT_FORCE_SPLITS, 1)  # CTA 0 then walks all 16 k-blocks of its tile
        h.set_option(sg.OPT_FORCE_TRANSPOSE_A, ta)
        h.set_option(sg.OPT_WAIT_TIMEOUT_NS, 50_000_000)  # 50 ms
        h.set_option(sg.OPT_INJECT_SKIP, 3)
        _, _, st = run_gemm(torch, h, A, B, C, 1.0, 1.0)
        assert st == sg.SGEMM_OK  # the launch itself is accepted
        status, code = h.check_device_status()
        assert status == sg.SGEMM_ERR_TIMEOUT and (code >> 16) == sg.SGEMM_ERR_TIMEOUT, hex(code)
        assert h.last_plan().transpose_a == ta
        # the status word is cleared and the context is healthy
        h.set_option(sg.OPT_INJECT_SKIP, -1)
        h.set_option(sg.OPT_WAIT_TIMEOUT_NS, 4_000_000_000)
        got, guards, st = run_gemm(torch, h, A, B, C, 1.0, 1.0)
        assert st == sg.SGEMM_OK and guards
        assert h.check_device_status() == (sg.SGEMM_OK, 0)
        check_against_oracle(got, A, B, C, 1.0, 1.0, exact=True)
    finally:
        h.close()
