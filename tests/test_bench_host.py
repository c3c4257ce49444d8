"""Host logic of bench.py on CPU: the replica timing reduction over gloo
ranks, the reference arm's rank handling, and the traffic record guard."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _rank_main(rank, world, port, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    r, w, _ = bench.dist_env()
    bench.dist_init(w, "gloo")
    v = bench.max_over_ranks(1.5 + r, w)
    bench.barrier(w)
    out.put((r, v))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # each rank's step time is the slowest rank's
    assert res == [(0, 2.5), (1, 2.5)]


def test_reference_arm_only_rank0_prints():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny",
                        "--steps", "1", "--warmup", "0"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_reference_arm_line_on_rank0():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny",
                        "--steps", "1", "--warmup", "0"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    for key in ("metric", "value", "unit", "higher_is_better", "config", "cpu_baseline", "e2e"):
        assert key in line
    assert line["value"] > 0 and line["e2e"]["value"] == line["value"]
    assert line["config"] == bench.workload_config(bench.wl.WORKLOADS["tiny"], line["config"]["lm_batch"],
                                                   line["config"]["k"], 1 if line["config"]["wire"] == "f16"
                                                   else (2 if line["config"]["wire"] == "i8" else 0),
                                                   line["config"]["embed_ids"], 1)


def test_recorded_traffic_is_dropped_when_kernels_change(tmp_path):
    d = bench.kernel_digest("qwen05b/lm_head")
    assert len(d) == 16
    recs = bench.load_traffic_records()
    assert recs and set(recs) <= set(bench.KERNEL_SOURCES)
    f = tmp_path / "t.txt"
    f.write_text(f"# comment\nqwen05b/lm_head {d} 1.0e6 cap_a  # trailing\n"
                 f"batched/lm_head {'0' * 16} 2e6 cap_b\n")
    recs = bench.load_traffic_records(str(f))
    assert bench.recorded_traffic("qwen05b/lm_head", recs) == (1.0e6, "cap_a")
    v, why = bench.recorded_traffic("batched/lm_head", recs)
    assert v is None and "changed" in why
    assert bench.recorded_traffic("no-such/measurement", recs)[0] is None


def test_bench_source_names_no_markdown_file():
    with open(os.path.join(ROOT, "bench.py")) as fh:
        assert ".md" not in fh.read()


def test_clock_lines_and_windows():
    assert bench.parse_clock_line("1965, 2070, 1010.5, 0x0, Not Active, Not Active, Not Active, Active") == \
        (1965.0, 2070.0, {"sw_power_cap"})
    assert bench.parse_clock_line("[N/A], 2070, 1, 0, a, b, c, d") is None
    assert bench.parse_clock_line("1, 2") is None
    s = bench.ClockSampler(0)
    s.samples = [(10.0, 2070.0, 2070.0, set()), (10.2, 1900.0, 2070.0, {"sw_power_cap"}),
                 (11.0, 1500.0, 2070.0, {"hw_slowdown"})]
    w = s.window(9.9, 10.5)
    assert w["samples"] == 2 and w["sm_mhz"] == 1985.0 and w["reasons"] == ["sw_power_cap"]
    assert s.window(20.0, 21.0)["samples"] == 0


def test_l2_policy_and_chunks():
    L2 = bench.L2_BYTES
    assert bench.l2_policy(8 << 20) == "flush"
    assert bench.l2_policy(bench.wl.WORKLOADS["qwen05b"].table_bytes) == "two_copies"
    assert bench.l2_policy(bench.wl.WORKLOADS["gemma_q8"].table_bytes) == "two_copies"
    assert bench.l2_policy(bench.wl.WORKLOADS["gemma31b"].table_bytes) == "stream"
    # a copy that alternates with another must itself exceed the L2
    assert bench.wl.WORKLOADS["gemma_q8"].table_bytes > L2
    assert bench.chunk_size(50e-6, False) == 10 and bench.chunk_size(300e-6, False) == 1
    assert bench.chunk_size(50e-6, True) == 1


def test_cpu_baseline_entry_single_and_all_cores():
    w = bench.wl.WORKLOADS["tiny"]
    T = bench.wl.table_for(w, threads=1)
    ids = bench.wl.ids_for(w)
    R = bench.wl.residuals_for(w, 4)
    e = bench.cpu_baseline_entry(w, T, ids, R, 4, 5, bench.wl.WIRE_F16, 0.2)
    assert e["single_thread"]["threads"] == 1 and e["all_cores"]["threads"] == e["cores"]
    assert e["value"] == e["all_cores"]["value"] > 0 and e["unit"] == "residuals/s"
    g = bench.cpu_baseline_entry(w, T, ids, R, 0, 5, bench.wl.WIRE_F16, 0.2)
    assert g["unit"] == "rows/s" and g["single_thread"]["value"] > 0
