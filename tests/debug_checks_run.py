"""Run by tests/test_gpu_debug_checks.py in a process of its own, against the debug
build of the library (SGEMM_GB300_DEBUG_CHECKS=1: every kernel checks the indices of
its accesses; a failed check records SGEMM_ERR_INDEX and skips the access).

A suite of small problems covering every plan form goes through it: tiny shapes,
tile multiples +-1 on every tile-config row with 1, 2, 3 and 7 splits and each A
layout, split-K within clusters, stream-K, unaligned / padded operands, and the TF32
mode (both kernels). After every call the device status word must read 0 and C
must match the FP64 oracle (bit-exact on integer operands)."""

import itertools
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import torch  # noqa: E402

import dense_fp32_gemm_04_gb300 as sg  # noqa: E402
import oracle  # noqa: E402
from dense_fp32_gemm_04_gb300 import inputs  # noqa: E402
from gpu_helpers import check_against_oracle, run_gemm  # noqa: E402

assert sg.LIB_PATH.endswith("_debug.so"), sg.LIB_PATH
calls = 0


def one(h, M, N, K, opts, lds=(None, None, None), offs=(0, 0, 0), tf32=False):
    global calls
    for opt, v in opts.items():
        h.set_option(opt, v)
    try:
        A, B, C = inputs.problem_operands(M=M, N=N, K=K, seed=M * 7 + N * 3 + K, dist=("int", "int", "int"))
        got, guards, st = run_gemm(torch, h, A, B, C, 1.5, 0.5, lds=lds, offsets=offs)
        plan = h.last_plan().as_dict()
        assert st == sg.SGEMM_OK and guards, (M, N, K, opts, plan)
        status, code = h.check_device_status()
        assert (status, code) == (sg.SGEMM_OK, 0), (hex(code), M, N, K, opts, plan)
        if tf32:
            ref, _ = oracle.sgemm_f64(A, B, C, 1.5, 0.5)
            assert oracle.exact(got, ref), (M, N, K, opts, plan)
        else:
            check_against_oracle(got, A, B, C, 1.5, 0.5, exact=True)
        calls += 1
    finally:
        for opt in opts:
            h.set_option(opt, 0 if opt == sg.OPT_FORCE_SPLITS else -1)


h = sg.Sgemm(0)
for M, N, K in itertools.product((1, 3, 8), (1, 5, 9), (1, 4, 7)):
    one(h, M, N, K, {})
for cfg, splits, ta in itertools.product(range(4), (1, 2, 3, 7), (0, 1, 2)):
    for M, N, K in ((63, 65, 33), (129, 127, 95), (256, 128, 224)):
        one(h, M, N, K, {sg.OPT_FORCE_CONFIG: cfg, sg.OPT_FORCE_SPLITS: splits, sg.OPT_FORCE_TRANSPOSE_A: ta})
for cfg, splits in itertools.product(range(4), (2, 4, 8)):
    one(h, 200, 190, 600, {sg.OPT_FORCE_CONFIG: cfg, sg.OPT_FORCE_SPLITS: splits, sg.OPT_CLUSTER_SPLIT: 1})
for ta in (0, 1, 2):
    for M, N, K in ((1000, 2500, 513), (300, 260, 777), (129, 127, 95)):
        one(h, M, N, K, {sg.OPT_FORCE_STREAMK: 1, sg.OPT_FORCE_TRANSPOSE_A: ta})
for cfg in range(4):
    one(h, 700, 900, 1500, {sg.OPT_FORCE_CONFIG: cfg, sg.OPT_FORCE_STREAMK: 1})
one(h, 190, 170, 150, {}, lds=(151, 173, 175), offs=(1, 2, 3))
one(h, 333, 222, 111, {}, lds=(115, 224, 230), offs=(0, 0, 1))
h.close()
for kernel in (0, 1):
    h = sg.Sgemm(0)
    h.set_math_mode(sg.MATH_TF32)
    for M, N, K in ((1, 1, 1), (129, 257, 33), (300, 500, 200), (77, 1000, 517)):
        one(h, M, N, K, {sg.OPT_FORCE_TF32_KERNEL: kernel}, tf32=True)
    one(h, 512, 600, 900, {sg.OPT_FORCE_TF32_KERNEL: kernel, sg.OPT_FORCE_STREAMK: 1}, tf32=True)
    one(h, 300, 301, 299, {sg.OPT_FORCE_TF32_KERNEL: kernel}, lds=(301, 303, 303), offs=(1, 1, 1), tf32=True)
    h.close()
print(f"debug build: {calls} calls, status word 0 after each, results exact")
