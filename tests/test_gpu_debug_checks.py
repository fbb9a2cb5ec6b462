"""The debug build of the library: its kernels check the indices of their memory
accesses (TMA tile coordinates, ring / staging / M-major buffer offsets, workspace
slots of split-K slices and stream-K partial tiles, stores to C, distributed shared
memory reads) and report a failed check as SGEMM_ERR_INDEX instead of touching
memory out of range. This stands in for a memory checker: a suite of small problems
over every plan form (tests/debug_checks_run.py) runs through that build in a
process of its own and must leave the status word at 0 with exact results."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

HERE = os.path.dirname(os.path.abspath(__file__))


def test_debug_build_index_checks_stay_silent():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_fp32_gemm_04_gb300 import _build

    lib = _build.build(debug=True)
    assert lib.endswith("libsgemm_gb300_debug.so")
    env = dict(os.environ, SGEMM_GB300_DEBUG_CHECKS="1")
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_checks_run.py")], env=env, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "status word 0 after each" in r.stdout
