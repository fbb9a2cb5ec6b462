"""Time the pages' kernel ladder (include/sgemm_ladder.h) and the library on one problem.

    python -m dense_fp32_gemm_04_gb300.ladder [--n 4096] [--out ladder.json]

Prints TFLOP/s per rung and the step-to-step speedups, next to the ratios the
pages report for the same steps on their (older) GPUs: coalescing 7.1x over the
naive kernel and shared-memory tiling 1.41x over coalescing ("Global Memory
Coalescing"), 1D register tiling 3.17x over shared-memory tiling ("1D Register
Tiling: One Thread, TM Outputs"); and, from "Shared memory and register
blocking", cache blocking at 3762 against 825 GFLOP/s for 32 x 32 shared-memory
tiles (4.56x) and register blocking on shared memory at 6172, 1.64x cache
blocking.
"""

from __future__ import annotations

import argparse
import json
import sys

RUNGS = {1: "naive", 2: "coalesced", 3: "smem tiling", 4: "1D register tiling", 5: "2D register tiling",
         6: "transposed A + float4", 7: "warp tiling", 8: "cache blocking", 9: "library (sgemm_run)"}
PAGE_RATIOS = {(1, 2): 7.1, (2, 3): 1.41, (3, 4): 3.17}
# (faster rung, slower rung): the pages' ratio of the two ("Shared memory and register blocking")
PAGE_PAIRS = {(8, 3): 3762 / 825, (6, 8): 6172 / 3762}
LIBRARY = 9


def main(argv=None):
    import torch

    import dense_fp32_gemm_04_gb300 as sg

    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--n", type=int, default=4096)
    ap.add_argument("--out", default=None)
    args = ap.parse_args(argv)
    n = args.n
    g = torch.Generator(device="cuda").manual_seed(0)
    A = torch.rand((n, n), device="cuda", generator=g) * 2 - 1
    B = torch.rand((n, n), device="cuda", generator=g) * 2 - 1
    C = torch.zeros((n, n), device="cuda")
    h = sg.Sgemm()
    flops = 2.0 * n * n * n
    res = {}
    for rung in range(1, LIBRARY + 1):
        call = (lambda: h.run(A, B, C, 1.0, 0.0)) if rung == LIBRARY else (lambda: sg.ladder_run(rung, A, B, C, 1.0, 0.0))
        st = call()
        if rung != LIBRARY and st != sg.SGEMM_OK:
            raise RuntimeError(f"rung {rung}: {sg.status_string(st)}")
        torch.cuda.synchronize()
        reps = 3 if rung <= 3 else 10
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            call()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        res[rung] = {"name": RUNGS[rung], "ms": ms, "tflops": flops / ms / 1e9}
    h.close()
    print(f"M=N=K={n}, alpha=1, beta=0")
    for rung, r in res.items():
        line = f"{rung} {r['name']:24s} {r['ms']:9.3f} ms {r['tflops']:7.2f} TFLOP/s"
        if rung > 1:
            line += f"  x{res[rung - 1]['ms'] / r['ms']:.2f} over rung {rung - 1}"
            if (rung - 1, rung) in PAGE_RATIOS:
                line += f" (pages: x{PAGE_RATIOS[(rung - 1, rung)]})"
        print(line)
    for (fast, slow), page in PAGE_PAIRS.items():
        print(f"rung {fast} ({res[fast]['name']}) over rung {slow} ({res[slow]['name']}): "
              f"x{res[slow]['ms'] / res[fast]['ms']:.2f} (pages: x{page:.2f})")
    if args.out:
        json.dump(res, open(args.out, "w"), indent=1)
    return 0


if __name__ == "__main__":
    sys.exit(main())
