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


def test_recorded_traffic_is_dropped_when_kernels_change(monkeypatch):
    d = bench.kernel_digest("qwen05b")
    assert len(d) == 16 and set(bench.TRAFFIC_RECORDS) <= set(bench.KERNEL_SOURCES)
    monkeypatch.setitem(bench.TRAFFIC_RECORDS, "qwen05b", (d, 1.0e6, "x"))
    assert bench.recorded_traffic("qwen05b") == (1.0e6, "x")
    monkeypatch.setitem(bench.TRAFFIC_RECORDS, "qwen05b", ("0" * 16, 1.0e6, "x"))
    v, why = bench.recorded_traffic("qwen05b")
    assert v is None and "changed" in why
    assert bench.recorded_traffic("no-such-workload")[0] is None
