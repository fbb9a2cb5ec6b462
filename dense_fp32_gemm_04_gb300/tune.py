"""Measure every tile-config row and split-K factor on a set of shapes.

    python -m dense_fp32_gemm_04_gb300.tune [--out sweep.json] [--shapes bench|all|small] [--layout-only]

For each shape it times the library's automatic plan and every forced
(config, splits) combination with CUDA events (operands uniform[-1,1), alpha=1,
beta=0, packed unless the shape says otherwise) and prints one line per shape:
the automatic plan's time, the best forced combination and the ratio. It also
times the automatic plan with A read as given, transposed first and transposed
in shared memory (``--layout-only``: only that). The planner's cost model, table and
transposition rule are checked against this sweep.
"""

from __future__ import annotations

import argparse
import json
import sys

SHAPES = {
    "bench": [(256, 256, 256), (512, 512, 512), (1024, 1024, 1024), (2048, 2048, 2048), (4096, 4096, 4096),
              (8192, 8192, 8192), (2047, 3001, 1531), (16384, 64, 8192), (64, 16384, 8192)],
}
SHAPES["all"] = SHAPES["bench"] + [(16384, 16384, 16384), (1000, 2500, 513), (1999, 3001, 1031),
                                   (4096, 1024, 4096), (1024, 4096, 4096), (8192, 128, 8192), (128, 8192, 8192)]
SHAPES["small"] = [(256, 256, 256), (512, 512, 512), (768, 768, 768), (1024, 1024, 1024), (1536, 1536, 1536),
                   (64, 16384, 8192), (128, 8192, 8192), (256, 4096, 4096), (4096, 256, 4096), (16384, 256, 4096),
                   (1000, 2500, 513), (2047, 3001, 1531)]
SPLITS = (1, 2, 3, 4, 6, 8, 12, 16)


def time_call(torch, fn, budget_flops, flops):
    for _ in range(2):
        fn()
    torch.cuda.synchronize()
    n = max(3, min(200, int(budget_flops / flops)))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(n):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n


LAYOUTS = {0: "as given", 1: "transposed first", 2: "transposed in shared memory"}


def layouts(torch, sg, h, run, budget_flops, flops):
    """Time of the automatic plan with each A layout: as given (0), transposed
    first in global memory (1), transposed in shared memory (2)."""
    out = {}
    for ta in LAYOUTS:
        h.set_option(sg.OPT_FORCE_TRANSPOSE_A, ta)
        out[ta] = time_call(torch, run, budget_flops, flops)
    h.set_option(sg.OPT_FORCE_TRANSPOSE_A, -1)
    return out


def sweep(shapes, budget_flops=4e11, layout_only=False):
    import torch

    import dense_fp32_gemm_04_gb300 as sg

    h = sg.Sgemm()
    results = []
    for (M, N, K) in shapes:
        g = torch.Generator(device="cuda").manual_seed(M + N + K)
        A = torch.rand((M, K), device="cuda", generator=g) * 2 - 1
        B = torch.rand((K, N), device="cuda", generator=g) * 2 - 1
        C = torch.zeros((M, N), device="cuda")
        flops = 2.0 * M * N * K
        run = lambda: h.run(A, B, C, 1.0, 0.0)  # noqa: E731
        auto_ms = time_call(torch, run, budget_flops, flops)
        auto = h.last_plan().as_dict()
        lay = layouts(torch, sg, h, run, budget_flops, flops)
        lay_line = (f"A as given {lay[0]:8.3f} ms, transposed first {lay[1]:8.3f} ms, in shared memory "
                    f"{lay[2]:8.3f} ms (auto picks {LAYOUTS[auto['transpose_a']]})")
        if layout_only:
            print(f"{M:6d} {N:6d} {K:6d}  auto cfg {auto['config']} S {auto['splits']}: {auto_ms:8.3f} ms | {lay_line}",
                  flush=True)
            results.append({"shape": [M, N, K], "auto_ms": auto_ms, "auto_plan": auto, "a_as_given_ms": lay[0],
                            "a_transposed_ms": lay[1], "a_smem_transposed_ms": lay[2]})
            continue
        rows = []
        for cfg in range(len(sg.configs())):
            h.set_option(sg.OPT_FORCE_CONFIG, cfg)
            for s in SPLITS:
                if s > (K + 31) // 32:
                    continue
                h.set_option(sg.OPT_FORCE_SPLITS, s)
                ms = time_call(torch, run, budget_flops, flops)
                rows.append({"config": cfg, "splits": s, "ms": ms, "tflops": flops / ms / 1e9})
        h.set_option(sg.OPT_FORCE_CONFIG, -1)
        h.set_option(sg.OPT_FORCE_SPLITS, 0)
        st, code = h.check_device_status()
        best = min(rows, key=lambda r: r["ms"])
        rec = {"shape": [M, N, K], "auto_ms": auto_ms, "auto_tflops": flops / auto_ms / 1e9, "auto_plan": auto,
               "best": best, "auto_over_best": auto_ms / best["ms"], "status": st, "forced": rows,
               "a_as_given_ms": lay[0], "a_transposed_ms": lay[1], "a_smem_transposed_ms": lay[2]}
        results.append(rec)
        print(f"{M:6d} {N:6d} {K:6d}  auto cfg {auto['config']} S {auto['splits']} sk {auto['sk_tiles']}"
              f": {auto_ms:8.3f} ms {rec['auto_tflops']:6.2f} TFLOP/s | best cfg {best['config']} "
              f"S {best['splits']}: {best['ms']:8.3f} ms {best['tflops']:6.2f} | auto/best {rec['auto_over_best']:.3f}"
              f" | {lay_line}", flush=True)
    h.close()
    return results


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--out", default=None)
    ap.add_argument("--shapes", default="bench", choices=sorted(SHAPES))
    ap.add_argument("--layout-only", action="store_true", help="time only the three A layouts of the automatic plan")
    args = ap.parse_args(argv)
    res = sweep(SHAPES[args.shapes], layout_only=args.layout_only)
    if args.out:
        with open(args.out, "w") as f:
            json.dump(res, f, indent=1)
    return 0


if __name__ == "__main__":
    sys.exit(main())
