"""Host-side logic of bench.py and the planner, pinned to figures the pages print
(tests/golden/page_figures.json), plus the multi-rank aggregation on 2 gloo ranks."""

import json
import os
import socket

import pytest

import bench

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")))


@pytest.mark.parametrize("case", GOLDEN["timings"])
def test_flop_count_matches_page_timings(case):
    gflops = bench.gemm_flops(case["M"], case["N"], case["K"]) / (case["ms"] * 1e-3) / 1e9
    assert abs(gflops - case["gflops"]) / case["gflops"] < 1e-4


def test_operand_traffic_model_matches_page():
    c = GOLDEN["global_traffic"][0]
    per_output = c["K"] * (1 / c["BM"] + 1 / c["BN"])
    assert per_output == c["loads_per_output"]
    gb = bench.operand_load_bytes(c["M"], c["N"], c["K"], c["BM"], c["BN"]) / 1e9
    assert round(gb, 2) == c["total_gb"]


def test_smem_reads_model_matches_page():
    one_d, naive = GOLDEN["smem_accesses_per_result"]
    assert bench.smem_reads_per_output(one_d["K"], one_d["TM"]) == one_d["value"]
    assert bench.smem_reads_per_output(naive["K"], naive["TM"]) == naive["value"]
    # the 8 x 8 microtile used here: K * 16 / 64 = K / 4
    assert bench.smem_reads_per_output(4096, 8, 8) == 1024


def test_float4_alignment_example(lib):
    import dense_fp32_gemm_04_gb300 as sg

    g = GOLDEN["float4_alignment"]
    cols = g["cols"]
    for off in g["legal_offsets"]:
        assert (off * 4) % 16 == 0 and off % cols == 0
    for off in g["illegal_offsets"]:
        assert (off * 4) % 16 != 0
    # a 15-wide packed matrix has rows that are not 16-byte aligned: the library
    # copies it to an aligned workspace instead of issuing vector/TMA loads on it
    p = sg.plan(15, 15, 15, lda=15, ldb=15, ldc=15)
    assert p.repack_a == 1 and p.repack_b == 1 and p.vec_c == 0


def test_clock_summary_parsing():
    s = bench.ClockSampler("0")
    s.lines = [(1.0, "1965, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active"),
               (1.1, "2070, 2070, 1000.0, 0x4, Not Active, Not Active, Not Active, Active"),
               (1.2, "2040, 2070, 1010.0, 0x0, Not Active, Not Active, Not Active, Not Active"),
               (9.0, "300, 2070, 100.0, 0x0, Not Active, Not Active, Not Active, Not Active")]
    out = s.summary(0.9, 1.3)
    assert out["sm_mhz"] == 2040 and out["sm_max_mhz"] == 2070 and out["reasons"] == ["sw_power_cap"]
    assert out["samples"] == 3


def test_traffic_is_ignored_for_a_changed_kernel(tmp_path, monkeypatch):
    f = tmp_path / "t.md"
    f.write_text("kernel_source_sha256_16: 0000000000000000\ndram_bytes_per_launch: 123\n")
    monkeypatch.setattr(bench, "TRAFFIC_SUMMARY", str(f))
    assert bench.recorded_traffic() is None
    f.write_text(f"kernel_source_sha256_16: {bench.kernel_source_hash()}\ndram_bytes_per_launch: 123\n")
    assert bench.recorded_traffic() == 123.0


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    w = bench.World()
    w.init("gloo")
    w.barrier()
    t = [0.5, 0.8][rank]
    q.put((rank, w.max(t)))
    w.close()


def test_two_gloo_ranks_take_the_max():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=5) for _ in range(2))
    assert got == {0: 0.8, 1: 0.8}
    value, t = bench.aggregate([0.5, 0.8], [2e12, 2e12])
    assert t == 0.8 and abs(value - 4e12 / 0.8 / 1e12) < 1e-12


def test_kernel_hash_ignores_comments():
    src = 'int a = 1; // note\n/* block\n note */ const char *s = "x // kept"; char c = \'/\';\n'
    assert bench.strip_comments(src) == 'int a = 1; const char *s = "x // kept"; char c = \'/\';'
    assert bench.strip_comments("a  =\n b;") == bench.strip_comments("a = b;".replace(" b", "\n  b"))
    assert bench.strip_comments("x = 1; // a") == bench.strip_comments("x = 1; // b")
    assert bench.strip_comments("x = 1;") != bench.strip_comments("x = 2;")


def test_optional_sections_report_failures_instead_of_raising(capsys):
    def boom():
        raise ValueError("no TF32 today")

    assert bench.optional("tf32_mode", boom) == {"error": "tf32_mode: ValueError: no TF32 today"}
    assert "ValueError" in capsys.readouterr().err
    assert bench.optional("min2", lambda a, b=0: a + b, 2, b=3) == 5
