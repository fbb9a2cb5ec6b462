"""bench.py prints one JSON line with the contract's keys (reference arm on CPU; our arm on a GPU)."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, timeout=600):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, capture_output=True, text=True,
                       timeout=timeout, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def test_reference_arm_line():
    d = _run(["--impl", "reference", "--workload", "square256", "--steps", "2", "--warmup", "1"])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1 and d["cpu_baseline"]["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


@pytest.mark.gpu
def test_our_arm_line():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = _run(["--steps", "20", "--warmup", "3", "--e2e-steps", "3", "--tf32-steps", "3", "--cpu-seconds", "0.5"])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks",
              "cpu_baseline"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 20 and d["dtype"] == "f32" and d["data"] == "synthetic"
    assert d["config"]["workload"].startswith("sgemm M=N=K=4096")
    r = d["roofline"]
    assert r["bound"] == "alu" and r["unit"] == "TFLOP/s" and 0 < r["frac"] < 1.2
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    e = d["e2e"]
    assert e["h2d_bytes_per_step"] == 3 * 4096 * 4096 * 4 and e["d2h_bytes_per_step"] == 4096 * 4096 * 4
    assert d["gpu_launches"] == d["config"]["plan"]["launches"] * 20
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] > 0
    assert d["tf32_mode"]["status"] == 0 and d["tf32_mode"]["roofline"]["bound"] == "tensor"
    probs = d["configs"]["problems"]
    assert [r["problem"] for r in probs] == ["square256", "sweep512", "sweep1024", "sweep2048", "sweep8192",
                                             "sweep16384", "ragged", "skinny_tall", "skinny_wide"]
    for r in probs:
        assert r["status"] == 0 and r["calls"] >= 20 and r["tflops"] > 0 and r["bound"] == "alu"
    assert {c["problem"] for c in d["cpu_baseline"]["configs"]} == {"square256", "square4096", "ragged", "skinny_tall"}
