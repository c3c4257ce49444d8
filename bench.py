#!/usr/bin/env python3
"""Benchmark of the embed / tied lm_head service hot path on GB300.

One step = one pass of the whole hot path over one batch of the workload:
  embed gather of the workload's token ids (x sqrt(hidden)),
  tied lm_head projection with fused top-k (+ probabilities),
  wire encode + decode of the residual batch in the workload's format.
Inputs are seeded synthetic data (workloads/), resident in HBM before the
timed region.  Tables between 64 MB and 4x the L2 are kept as two copies
that alternate from call to call, so no call finds its table in L2; smaller
tables are preceded by an L2 flush outside the timed events; larger ones
are streamed as they are.

The device step and the lm_head roofline loops replay CUDA graphs of the
C-ABI calls (captured once; --eager times eager calls), as a serving loop
would, so the host's launch cost and the per-launch submission gaps stay
out of the device figures.

Prints one JSON line.  `value` is lm_head top-k residuals per second of the
headline workload (qwen05b) for the whole job (all ranks).  Under torchrun
every rank runs its own replica (weak scaling; the path needs no exchange
between GPUs).  The line also carries, under `configs`, every workload's own
measurements: each bandwidth-bound call timed for >= 1.5 s of device time
(mean, median and min per call), its algorithmic bytes, its fraction of the
measured HBM copy bandwidth and the SM clocks sampled while it ran; the
launch-bound calls as latencies; and the oracle's rate on host cores, single
threaded and on all cores.

  python bench.py [--workload qwen05b] [--steps K] [--warmup W] [--no-configs]
  python bench.py --impl reference      # the CPU oracle, timed on host cores
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as wl  # noqa: E402

METRIC = "lm_head top-k residuals/s + HBM GB/s (% roofline); embed gather rows/s"
UNIT = "residuals/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1700.0
L2_BYTES = 129 * 1024 * 1024
ROOFLINE_SECONDS = 1.5          # device time of every bandwidth-bound timing loop
CONFIG_ORDER = ("tiny", "qwen05b", "gemma_q8", "gemma31b", "batched")


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="lhs", choices=["lhs", "reference"])
    ap.add_argument("--workload", default="qwen05b", choices=sorted(wl.WORKLOADS))
    ap.add_argument("--batch", type=int, default=None, help="lm_head batch (default: workload's first)")
    ap.add_argument("--vocab", type=int, default=None,
                    help="override the workload's vocab rows (small cases for profiling)")
    ap.add_argument("--no-configs", action="store_true",
                    help="only the headline workload (no per-workload `configs` block)")
    ap.add_argument("--configs", default=",".join(CONFIG_ORDER) + ",codec",
                    help="comma list of the `configs` entries to measure")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=5.0,
                    help="oracle seconds per timing (headline; the configs take a third of it)")
    ap.add_argument("--roofline-seconds", type=float, default=ROOFLINE_SECONDS)
    ap.add_argument("--untied", action="store_true",
                    help="lm_head on a second table of the same shape (an untied lm_head)")
    ap.add_argument("--e2e-eager", action="store_true",
                    help="time the end-to-end step as eager calls instead of replaying it as a CUDA graph")
    ap.add_argument("--profile-case", default=None,
                    help="run a few calls of one measurement and exit, for an ncu launch list: "
                         "lm_head:<workload>[:<vocab>[:<batch>]], gather:<workload>[:<ids>], "
                         "embed_wire_i8:<workload>[:<ids>], codec:<f16|i8>:<encode|decode>[:<positions>]")
    ap.add_argument("--eager", action="store_true",
                    help="time the device step and the lm_head loops as eager calls instead of CUDA graph replays")
    ap.add_argument("--raw-logits", action="store_true",
                    help="the step's lm_head call returns the full logits (raw-logits mode)")
    ap.add_argument("--wire-accuracy", action="store_true",
                    help="top-k agreement of logits from wire-decoded residuals with the "
                         "originals (f16: top-5, i8: top-1) on the gemma31b and batched workloads")
    ap.add_argument("--sweep", action="store_true",
                    help="steady-state sweep of the sub-10-us steps (gather, wire codecs): one "
                         "JSON line per point instead of the step line")
    return ap.parse_args(argv)


def default_steps(name):
    return {"tiny": 2000, "qwen05b": 2000, "gemma_q8": 2000, "gemma31b": 400,
            "batched": 200}[name]


# ---------------------------------------------------------------------------
# distributed plumbing (replicas: one process per GPU, no data-path collective)
# ---------------------------------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world, backend):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world, device=None) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# peaks and clocks
# ---------------------------------------------------------------------------

def load_peaks():
    """(hbm GB/s, bf16 TFLOP/s sustained, source) from the measured peaks
    file, else the fallback figures."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return (float(d["hbm_gbs"]), float(d.get("bf16_tflops_sustained", d.get("bf16_tflops"))),
                "measured")
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


_REASON_COLS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


def parse_clock_line(line: str):
    """(sm MHz, max sm MHz, set of active reasons) of one nvidia-smi CSV
    line, or None."""
    parts = [p.strip() for p in line.split(",")]
    if len(parts) < 8:
        return None
    try:
        sm, mx = float(parts[0]), float(parts[1])
    except ValueError:
        return None
    reasons = {name for name, val in zip(_REASON_COLS, parts[4:8]) if val.lower().startswith("active")}
    return sm, mx, reasons


def summarize_clocks(samples):
    """Clock record of a list of (time, sm, max, reasons) samples."""
    if not samples:
        return {"samples": 0, "sm_mhz": None, "sm_max_mhz": None, "reasons": []}
    sm = [s[1] for s in samples]
    reasons = set()
    for s in samples:
        reasons |= s[3]
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(s[2] for s in samples),
            "sm_mhz_min": min(sm), "samples": len(samples), "reasons": sorted(reasons)}


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons every 200 ms
    for the whole run; each timed loop takes the samples that arrived while
    it ran (host time window)."""

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.samples = []
        self.thread = None

    def start(self):
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.5)   # nvidia-smi's own start-up
        return self

    def _read(self):
        for line in self.proc.stdout:
            r = parse_clock_line(line)
            if r is not None:
                self.samples.append((time.time(), *r))

    def window(self, t0, t1):
        return summarize_clocks([s for s in list(self.samples) if t0 <= s[0] <= t1 + 0.05])

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)


class NoSampler:
    samples = []

    def window(self, t0, t1):
        return summarize_clocks([])

    def stop(self):
        pass


# ---------------------------------------------------------------------------
# DRAM traffic records (ncu captures, one text file beside their summaries)
# ---------------------------------------------------------------------------

TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")
_LM = ("embedding_lookup_tied_gb300/csrc/lm_head.cu", "embedding_lookup_tied_gb300/csrc/lm_topk.cuh",
       "embedding_lookup_tied_gb300/csrc/lhs_internal.cuh")
# the files each recorded measurement's kernels are compiled from: a change
# to any of them voids its record
KERNEL_SOURCES = {
    "tiny/lm_head": _LM,
    "qwen05b/lm_head": _LM,
    "gemma31b/lm_head_b1": _LM,
    "gemma31b/lm_head_b8": _LM,
    "gemma_q8/lm_head": ("embedding_lookup_tied_gb300/csrc/gemv_q8.cu",) + _LM,
    "batched/lm_head": ("embedding_lookup_tied_gb300/csrc/gemm_tc.cu",) + _LM,
    "gemma_q8/gather_steady": ("embedding_lookup_tied_gb300/csrc/gather.cu",
                               "embedding_lookup_tied_gb300/csrc/lhs_internal.cuh"),
    "codec/f16_encode": ("embedding_lookup_tied_gb300/csrc/wire.cu",
                         "embedding_lookup_tied_gb300/csrc/lhs_internal.cuh"),
    "codec/f16_decode": ("embedding_lookup_tied_gb300/csrc/wire.cu",
                         "embedding_lookup_tied_gb300/csrc/lhs_internal.cuh"),
    "codec/i8_encode": ("embedding_lookup_tied_gb300/csrc/wire.cu",
                        "embedding_lookup_tied_gb300/csrc/lhs_internal.cuh"),
    "codec/i8_decode": ("embedding_lookup_tied_gb300/csrc/wire.cu",
                        "embedding_lookup_tied_gb300/csrc/lhs_internal.cuh"),
    "gemma_q8/embed_wire_i8_steady": ("embedding_lookup_tied_gb300/csrc/embed_wire.cu",
                                      "embedding_lookup_tied_gb300/csrc/lhs_internal.cuh"),
}


def load_traffic_records(path=TRAFFIC_FILE):
    """{measurement: (sources digest, DRAM bytes per call, capture name)}."""
    recs = {}
    try:
        with open(path) as f:
            for line in f:
                line = line.split("#", 1)[0].strip()
                if not line:
                    continue
                name, digest, nbytes, capture = line.split()[:4]
                recs[name] = (digest, float(nbytes), capture)
    except FileNotFoundError:
        pass
    return recs


def kernel_digest(name) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[name]:
        p = os.path.join(ROOT, f)
        if os.path.exists(p):
            with open(p, "rb") as fh:
                h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(name, records=None):
    """(DRAM bytes per call, capture name) or (None, why not)."""
    rec = (load_traffic_records() if records is None else records).get(name)
    if rec is None or name not in KERNEL_SOURCES:
        return None, "no ncu capture recorded for this measurement"
    digest, nbytes, src = rec
    if kernel_digest(name) != digest:
        return None, f"kernel sources changed since the capture {src}"
    return nbytes, src


# ---------------------------------------------------------------------------
# workload setup
# ---------------------------------------------------------------------------

class Ctx:
    pass


def l2_policy(table_bytes: int) -> str:
    """How a timing loop keeps the table out of L2 between calls."""
    if table_bytes < 64 * 1000 * 1000:
        return "flush"
    if table_bytes < 4 * L2_BYTES:
        return "two_copies"
    return "stream"


def l2_note(policy: str) -> str:
    return {"flush": "a 258 MB buffer is rewritten before every timed call, outside the events "
                     "(the table fits in L2)",
            "two_copies": "two copies of the table alternate from call to call (each larger than "
                          "the L2), so no call finds its table in L2",
            "stream": "the table is more than 4x the L2 and is streamed by every call"}[policy]


def up(a, device):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(device)


def setup(name, batch, device, vocab=None, untied=False, raw=False, T_host=None):
    import ctypes
    import dataclasses

    import torch

    import embedding_lookup_tied_gb300 as lhs
    c = Ctx()
    c.w = w = wl.WORKLOADS[name]
    if vocab:
        c.w = w = dataclasses.replace(w, vocab=vocab)
    c.B = batch or (w.batches[0] if w.batches else 1)
    c.k = w.k or 10
    c.fmt = w.wire[0] if w.wire else wl.WIRE_F16
    c.n_ids = w.n_ids or 1
    c.lhs = lhs
    c.dev = device
    c.T_host = wl.table_for(w) if T_host is None else T_host
    c.policy = l2_policy(w.table_bytes)
    ncopy = 2 if c.policy == "two_copies" else 1
    t_dev = up(c.T_host, device)
    c.table_tensors = [t_dev] + [t_dev.clone() for _ in range(ncopy - 1)]
    c.tables = [lhs.lhs_table_init(t, w.vocab, w.hidden, w.dtype) for t in c.table_tensors]
    c.table = c.tables[0]
    c.untied, c.raw = untied, raw
    if untied:
        # a second table, same shape and distribution, other seed
        u = up(wl.make_table(w.dtype, w.vocab, w.hidden, 0.02, cid=w.cid + 50), device)
        c.lm_tensors = [u] + [u.clone() for _ in range(ncopy - 1)]
        c.lm_tables = [lhs.lhs_table_init(t, w.vocab, w.hidden, w.dtype) for t in c.lm_tensors]
    else:
        c.lm_tables = c.tables
    c.lm_table = c.lm_tables[0]
    c.ids_host = wl.ids_for(w) if w.n_ids else wl.zipf_ids(w.cid, 1, w.vocab)
    c.R_host = wl.residuals_for(w, c.B)
    c.ids = up(c.ids_host, device)
    c.resid = up(c.R_host, device)
    if w.resid_dtype == wl.BF16:
        c.resid = c.resid.view(torch.bfloat16)
    c.scale = float(w.embed_scale)
    H = w.hidden
    c.emb_out = torch.empty((c.n_ids, H), dtype=torch.float32, device=device)
    rd = lhs.LHS_F32 if w.resid_dtype == wl.F32 else lhs.LHS_BF16
    c.rd = rd
    c.ws = torch.empty(lhs.lhs_logits_topk_workspace(c.lm_table, c.B, 0 if raw else c.k, rd),
                       dtype=torch.uint8, device=device)
    c.raw_out = torch.empty((c.B, w.vocab), dtype=torch.float32, device=device) if raw else None
    c.top_ids = torch.empty((c.B, c.k), dtype=torch.int32, device=device)
    c.top_logits = torch.empty((c.B, c.k), dtype=torch.float32, device=device)
    c.top_probs = torch.empty((c.B, c.k), dtype=torch.float32, device=device)
    c.wire_bytes = lhs.lhs_wire_bytes(c.fmt, c.B, H)
    c.wire_buf = torch.empty(c.wire_bytes, dtype=torch.uint8, device=device)
    c.dec = torch.empty((c.B, H), dtype=torch.float32, device=device)
    c.err = torch.zeros(1, dtype=torch.int32, device=device)
    c.stream = torch.cuda.current_stream(device)
    c.sptr = c.stream.cuda_stream
    # direct C-ABI argument lists (no per-call marshalling in the timed loop),
    # one list per table copy
    L = lhs.lib()
    c.L = L
    c.steps_by_copy, c.lm_by_copy, c.embed_by_copy = [], [], []
    for tab, lmt in zip(c.tables, c.lm_tables):
        tb, lb = ctypes.byref(tab.c), ctypes.byref(lmt.c)
        if raw:
            lm_call = (L.lhs_logits, (lb, c.resid.data_ptr(), rd, c.B, c.raw_out.data_ptr(), c.ws.data_ptr(),
                                      c.ws.numel(), c.err.data_ptr(), c.sptr))
        else:
            lm_call = (L.lhs_logits_topk, (lb, c.resid.data_ptr(), rd, c.B, c.k, ctypes.c_float(1.0),
                                           c.top_ids.data_ptr(), c.top_logits.data_ptr(),
                                           c.top_probs.data_ptr(), c.ws.data_ptr(), c.ws.numel(),
                                           c.err.data_ptr(), c.sptr))
        embed_call = (L.lhs_embed, (tb, c.ids.data_ptr(), c.n_ids, ctypes.c_float(c.scale),
                                    c.emb_out.data_ptr(), c.err.data_ptr(), c.sptr))
        c.lm_by_copy.append(lm_call)
        c.embed_by_copy.append(embed_call)
        c.steps_by_copy.append([embed_call, lm_call] + wire_calls(c))
    c.lm_call = c.lm_by_copy[0]
    if c.policy == "flush":
        c.flush_buf = torch.zeros(2 * L2_BYTES // 4, dtype=torch.int32, device=device)
    # kernels per step: embed 1, the lm_head call as the library reports it
    # for this plan, wire encode 1, decode 1
    lm = lhs.lhs_logits_topk_launches(c.lm_table, c.B, 0 if raw else c.k, rd)
    c.lm_launches = lm
    c.gemm = (w.dtype == wl.BF16 and w.resid_dtype == wl.BF16 and c.B > 8)
    c.launches_per_step = 1 + lm + 1 + 1
    return c


def wire_calls(c):
    L, H = c.L, c.w.hidden
    return [(L.lhs_wire_encode, (c.fmt, c.resid.data_ptr(), c.rd, c.B, H, 0, 0, c.k,
                                 c.wire_buf.data_ptr(), c.wire_bytes, c.err.data_ptr(), c.sptr)),
            (L.lhs_wire_decode, (c.fmt, c.wire_buf.data_ptr(), c.wire_bytes, c.B, H,
                                 c.dec.data_ptr(), c.err.data_ptr(), c.sptr))]


def call(fn_args):
    fn, args = fn_args
    rc = fn(*args)
    if rc != 0:
        raise RuntimeError(f"{fn.__name__} -> {rc}")


GRAPH_CALLS = 20  # lm_head calls per replayed graph in the roofline loops
EAGER = False     # --eager: no graphs in the device step and roofline loops


def graph_of(calls):
    """A CUDA graph of direct C-ABI calls ((fn, args) with the stream handle
    last), captured on torch's capture stream; replay() re-issues them on the
    current stream, without the host's per-launch cost."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        sp = torch.cuda.current_stream().cuda_stream
        for fn, args in calls:
            args = list(args)
            args[-1] = sp
            rc = fn(*args)
            if rc != 0:
                raise RuntimeError(f"{fn.__name__} -> {rc} during capture")
    torch.cuda.synchronize()
    return g


def run_step(c, i=0):
    for fa in c.steps_by_copy[i % len(c.steps_by_copy)]:
        call(fa)


def workload_config(w, B, k, fmt, n_ids, world, untied=False, raw=False):
    """The `config` object of the JSON line (both arms)."""
    return {"workload": w.name, "vocab": w.vocab, "hidden": w.hidden,
            "table_dtype": wl.DTYPE_NAMES[w.dtype], "table_bytes": w.table_bytes,
            "embed_ids": n_ids, "lm_batch": B, "k": k,
            "lm_table": "untied (second table, same shape)" if untied else "tied (the embedding table)",
            "lm_output": "raw logits [batch x vocab]" if raw else "top-k ids, logits, probs",
            "wire": {0: "f32", 1: "f16", 2: "i8"}[fmt],
            "l2": l2_note(l2_policy(w.table_bytes)),
            "parallelism": f"replicas x{world}"}


def lm_bytes(w, B, k, raw=False):
    """Algorithmic bytes of one lm_head call: every table row once, the
    residuals once, the top-k outputs (or the raw logits) once."""
    relt = 4 if w.resid_dtype == wl.F32 else 2
    out = B * w.vocab * 4 if raw else B * k * 12
    return w.vocab * w.row_bytes + B * w.hidden * relt + out


def embed_bytes(w, n_ids, distinct):
    """Algorithmic bytes of one gather: the ids, each distinct row once
    (repeats hit L2), the f32 output."""
    return n_ids * (4 + w.hidden * 4) + distinct * w.row_bytes


def wire_bytes_rt(B, H, relt, msg_bytes):
    """Encode reads the residuals and writes the message; decode reads the
    message and writes f32 residuals."""
    return (B * H * relt + msg_bytes) + (msg_bytes + B * H * 4)


def step_bytes(c):
    w = c.w
    relt = 4 if w.resid_dtype == wl.F32 else 2
    distinct = len(np.unique(c.ids_host)) if w.n_ids else 0
    emb = embed_bytes(w, c.n_ids, distinct) if w.n_ids else c.n_ids * (4 + w.hidden * 4) + w.row_bytes
    return lm_bytes(w, c.B, c.k, c.raw) + emb + wire_bytes_rt(c.B, w.hidden, relt, c.wire_bytes)


# ---------------------------------------------------------------------------
# timing
# ---------------------------------------------------------------------------

def timed_loop(c, body, n):
    """Device time of `body(i)` per iteration (ms), CUDA events on the
    calls' stream.  With the flush policy a buffer larger than L2 is
    overwritten before every iteration, outside the timed events."""
    import torch
    if c.policy != "flush":
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(c.stream)
        for i in range(n):
            body(i)
        e1.record(c.stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / n
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for i, (a, b) in enumerate(ev):
        c.flush_buf.add_(1)
        a.record(c.stream)
        body(i)
        b.record(c.stream)
    ev[-1][1].synchronize()
    return sum(a.elapsed_time(b) for a, b in ev) / n


def chunk_size(per_call_s: float, flush: bool) -> int:
    """Calls between two events of a long loop: one for calls of 200 us or
    more (or when each call is preceded by a flush), else about 0.5 ms."""
    if flush or per_call_s >= 200e-6:
        return 1
    return max(1, int(500e-6 / max(per_call_s, 1e-7)))


def measure(c, body, seconds=ROOFLINE_SECONDS, sampler=None, min_iters=50, warm=5, calls_per_body=1):
    """Time `body(i)` for >= `seconds` of device time.  Returns per-call
    mean (over all calls), median and min (over chunks of calls between two
    events), the iteration count and the clocks sampled while it ran.  One
    body(i) may issue several calls (a graph replay): calls_per_body."""
    import torch
    for i in range(warm):
        body(i)
    torch.cuda.synchronize()
    flush = c.policy == "flush"
    est = timed_loop(c, body, 10) * 1e-3
    chunk = chunk_size(est, flush)
    n = max(min_iters, int(math.ceil(seconds / max(est, 1e-7))))
    n = int(math.ceil(n / chunk)) * chunk
    nch = n // chunk
    t0 = time.time()
    if flush:
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(nch)]
        for j, (a, b) in enumerate(ev):
            c.flush_buf.add_(1)
            a.record(c.stream)
            body(j)
            b.record(c.stream)
        ev[-1][1].synchronize()
        per = [a.elapsed_time(b) * 1e3 for a, b in ev]
    else:
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(nch + 1)]
        ev[0].record(c.stream)
        i = 0
        for j in range(nch):
            for _ in range(chunk):
                body(i)
                i += 1
            ev[j + 1].record(c.stream)
        ev[-1].synchronize()
        per = [ev[j].elapsed_time(ev[j + 1]) * 1e3 / chunk for j in range(nch)]
    t1 = time.time()
    if int(c.err.item()) != 0:
        raise RuntimeError(f"error word {int(c.err.item())} in a timing loop")
    per = [x / calls_per_body for x in per]
    return {"avg_us": sum(per) / len(per), "median_us": statistics.median(per), "min_us": min(per),
            "iters": n * calls_per_body, "chunk": chunk * calls_per_body, "device_s": sum(per) * chunk * calls_per_body * 1e-6,
            "clocks": (sampler or NoSampler()).window(t0, t1)}


def latency(c, body, n=200):
    """Per-call device time (us) of a launch-bound call: mean, median and
    min over `n` single calls between events."""
    import torch
    for i in range(5):
        body(i)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for i, (a, b) in enumerate(ev):
        if c.policy == "flush":
            c.flush_buf.add_(1)
        a.record(c.stream)
        body(i)
        b.record(c.stream)
    ev[-1][1].synchronize()
    per = [a.elapsed_time(b) * 1e3 for a, b in ev]
    return {"avg_us": sum(per) / n, "median_us": statistics.median(per), "min_us": min(per), "iters": n}


def roofline_entry(name, kernel, m, nbytes, peak_gbs, peak_src, records=None):
    """`roofline` object of one bandwidth-bound measurement."""
    achieved = nbytes / (m["avg_us"] * 1e-6) / 1e9
    traffic, tsrc = recorded_traffic(name, records)
    return {"kernel": kernel, "bound": "hbm", "achieved": achieved, "peak": peak_gbs, "unit": "GB/s",
            "frac": achieved / peak_gbs, "frac_median": nbytes / (m["median_us"] * 1e-6) / 1e9 / peak_gbs,
            "peak_source": f"{peak_src} hbm_gbs", "traffic": traffic, "traffic_source": tsrc,
            "traffic_ratio": traffic / nbytes if traffic else None,
            "algorithmic_bytes": nbytes, "avg_us": m["avg_us"], "median_us": m["median_us"],
            "min_us": m["min_us"], "iters": m["iters"], "events_every": m["chunk"],
            "device_s": m["device_s"], "clocks": m["clocks"]}


def time_device(c, steps, warmup, world):
    """The headline step loop: exactly `steps` steps between events (after
    `warmup` untimed ones), the table copies alternating."""
    import torch
    for i in range(warmup):
        run_step(c, i)
    torch.cuda.synchronize()
    if int(c.err.item()) != 0:
        raise RuntimeError(f"error word {int(c.err.item())} during warm-up")
    per = 1  # steps per timed body
    if EAGER or c.policy == "flush":
        step = lambda i: run_step(c, i)
    else:
        # graphs of `per` consecutive steps (per divides `steps`), the table
        # copies alternating inside, so that the steps of one replay overlap
        # as eager launches do; one graph per starting copy
        per = next(d for d in (10, 8, 5, 4, 2, 1) if steps % d == 0)
        nc = len(c.steps_by_copy)
        graphs = [graph_of([cl for j in range(per) for cl in c.steps_by_copy[(s0 + j) % nc]]) for s0 in range(nc)]
        step = lambda r: graphs[(r * per) % nc].replay()
        for r in range(max(1, warmup // per)):
            step(r)
        torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    ms = timed_loop(c, step, steps // per) / per
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(world)
    if int(c.err.item()) != 0:
        raise RuntimeError(f"error word {int(c.err.item())} in the timed region")
    return ms, (t0, t1)


def time_e2e(c, steps, graph=False):
    """Same step through the public binding with HOST buffers: each step
    copies its inputs from pinned host memory and reads its results back.
    The step's inputs and outputs share one device buffer (and one pinned
    host mirror) laid out [ids | residuals | error word | lm_head outputs |
    wire message | decoded residuals | embeddings], so a step is one
    host-to-device copy (ids, residuals and the zeroed error word), the
    calls (embed, lm_head, wire encode, wire decode), and two device-to-host
    copies: the embeddings, on a second stream as soon as the gather has
    written them (so they travel while the lm_head streams its table), and
    the error word with the other outputs after the last call.  The step
    ends when both copies have landed (the calls' stream waits for the
    second one), so the next step's gather never overwrites embeddings still
    in flight.  graph=True captures one step — copies and calls, both streams
    — in a CUDA graph and replays it, so the host's per-call launch cost
    leaves the loop."""
    import torch
    lhs = c.lhs
    dev = c.ids.device
    rd_t = torch.bfloat16 if c.w.resid_dtype == wl.BF16 else torch.float32
    relt = 2 if c.w.resid_dtype == wl.BF16 else 4
    H = c.w.hidden
    parts = [("ids", c.n_ids * 4), ("res", c.B * H * relt), ("err", 4)]
    if c.raw:
        parts.append(("raw", c.B * c.w.vocab * 4))
    else:
        parts += [("tid", c.B * c.k * 4), ("tlg", c.B * c.k * 4), ("tpr", c.B * c.k * 4)]
    parts += [("buf", c.wire_bytes), ("dec", c.B * H * 4), ("emb", c.n_ids * H * 4)]
    off, pos = {}, 0
    for name, nb in parts:
        off[name] = pos
        pos = (pos + nb + 255) // 256 * 256
    total = pos
    d_io = torch.empty(total, dtype=torch.uint8, device=dev)
    h_io = torch.empty(total, dtype=torch.uint8).pin_memory()

    def view(t, name, nb, dtype, shape):
        return t[off[name]:off[name] + nb].view(dtype).view(shape)

    # inputs and the zeroed error word, in the host mirror
    view(h_io, "ids", c.n_ids * 4, torch.int32, (c.n_ids,)).copy_(torch.from_numpy(c.ids_host.copy()))
    rh = c.R_host.view(np.int16) if c.R_host.dtype == np.uint16 else c.R_host
    hr = torch.from_numpy(np.ascontiguousarray(rh))
    view(h_io, "res", c.B * H * relt, hr.dtype, (c.B, H)).copy_(hr)
    view(h_io, "err", 4, torch.int32, (1,)).zero_()
    d_ids = view(d_io, "ids", c.n_ids * 4, torch.int32, (c.n_ids,))
    d_res = view(d_io, "res", c.B * H * relt, rd_t, (c.B, H))
    d_err = view(d_io, "err", 4, torch.int32, (1,))
    d_emb = view(d_io, "emb", c.n_ids * H * 4, torch.float32, (c.n_ids, H))
    d_buf = view(d_io, "buf", c.wire_bytes, torch.uint8, (c.wire_bytes,))
    d_dec = view(d_io, "dec", c.B * H * 4, torch.float32, (c.B, H))
    if c.raw:
        d_raw = view(d_io, "raw", c.B * c.w.vocab * 4, torch.float32, (c.B, c.w.vocab))
    else:
        d_tid = view(d_io, "tid", c.B * c.k * 4, torch.int32, (c.B, c.k))
        d_tlg = view(d_io, "tlg", c.B * c.k * 4, torch.float32, (c.B, c.k))
        d_tpr = view(d_io, "tpr", c.B * c.k * 4, torch.float32, (c.B, c.k))
    in_end = off["err"] + 4              # ids, residuals, error word
    out0 = off["err"]                    # error word and the lm_head / wire outputs
    emb0 = off["emb"]                    # the embeddings
    out1 = off["emb"] + c.n_ids * H * 4
    h2d = in_end
    d2h = (emb0 - out0) + (out1 - emb0)

    ncopy = len(c.tables)
    side = torch.cuda.Stream(device=dev)
    ev_emb = torch.cuda.Event()
    ev_back = torch.cuda.Event()

    def one(i):
        tab, lmt = c.tables[i % ncopy], c.lm_tables[i % ncopy]
        main = torch.cuda.current_stream(dev)
        d_io[:in_end].copy_(h_io[:in_end], non_blocking=True)
        lhs.lhs_embed(tab, d_ids, c.scale, out=d_emb, err=d_err)
        if c.n_ids:
            ev_emb.record(main)
            with torch.cuda.stream(side):
                side.wait_event(ev_emb)
                h_io[emb0:out1].copy_(d_io[emb0:out1], non_blocking=True)
                ev_back.record(side)
        if c.raw:
            lhs.lhs_logits(lmt, d_res, out=d_raw, ws=c.ws, err=d_err)
        else:
            lhs.lhs_logits_topk(lmt, d_res, c.k, 1.0, ws=c.ws, ids=d_tid, logits=d_tlg, probs=d_tpr,
                                err=d_err)
        lhs.lhs_wire_encode(c.fmt, d_res, 0, 0, c.k, buf=d_buf, err=d_err)
        lhs.lhs_wire_decode(c.fmt, d_buf, c.B, H, out=d_dec, err=d_err)
        h_io[out0:emb0].copy_(d_io[out0:emb0], non_blocking=True)
        if c.n_ids:
            main.wait_event(ev_back)

    for i in range(6):
        one(i)
    torch.cuda.synchronize()
    step = one
    if graph:
        # one graph per table copy, replayed alternately like the eager calls
        graphs = []
        for j in range(ncopy):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                one(j)
            graphs.append(g)
        torch.cuda.synchronize()

        def step(i):
            graphs[i % ncopy].replay()
        for i in range(4):
            step(i)
        torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(c.stream)
    for i in range(steps):
        step(i)
    e1.record(c.stream)
    e1.synchronize()
    if int(view(h_io, "err", 4, torch.int32, (1,)).item()) != 0:
        raise RuntimeError("error word set in the end-to-end loop")
    return e0.elapsed_time(e1) / steps, h2d, d2h


# ---------------------------------------------------------------------------
# the oracle on host cores (cpu_baseline and --impl reference)
# ---------------------------------------------------------------------------

def oracle_parts(w, T, ids, R, B, k, fmt, budget_s, threads):
    """Time the oracle on a bounded sample of one step: the full embed and
    wire work, and the lm_head over consecutive slices of vocab rows until
    the budget is spent (or every row is done), that time scaled up to the
    full vocabulary.  Returns seconds per step for each part and a
    description of the sample."""
    import oracle as orc
    xv = R if w.resid_dtype == wl.F32 else orc.bf16_to_f32(R)
    t0 = time.perf_counter()
    if w.n_ids:
        orc.embed(T, w.dtype, w.vocab, w.hidden, ids, w.embed_scale)
    t_embed = time.perf_counter() - t0
    t0 = time.perf_counter()
    if B:
        buf, _ = orc.wire_encode(fmt, xv)
        orc.wire_decode(fmt, buf, B, w.hidden)
    t_wire = time.perf_counter() - t0
    rows = min(64, w.vocab)
    t_lm = 0.0
    done = 0
    if B:
        while True:
            t1 = time.perf_counter()
            L = orc.logits(T, w.dtype, w.vocab, w.hidden, xv, v0=done, v1=done + rows, threads=threads)
            for b in range(B):
                orc.topk_f64(L[b], min(k, rows))
            t_lm += time.perf_counter() - t1
            done += rows
            if t_lm + t_embed + t_wire >= budget_s or done >= w.vocab:
                break
            rows = min(rows * 2, 1 << 14, w.vocab - done)
    scale = w.vocab / done if done else 0.0
    sample = (f"1 step: full embed ({w.n_ids} ids) + wire encode/decode of {B} residual(s)"
              + (f"; lm_head over {done} of {w.vocab} vocab rows, time scaled x{scale:.1f}" if done else ""))
    return {"embed_s": t_embed, "wire_s": t_wire, "lm_s": t_lm * scale, "sample": sample}


def oracle_rate(w, T, ids, R, B, k, fmt, budget_s, threads):
    """(residuals/s of the oracle's step, sample description)."""
    p = oracle_parts(w, T, ids, R, B, k, fmt, budget_s, threads)
    return B / (p["embed_s"] + p["wire_s"] + p["lm_s"]), p["sample"]


def cpu_baseline_entry(w, T, ids, R, B, k, fmt, budget_s):
    """The oracle timed single threaded and on every host core.  Workloads
    with an lm_head report residuals/s of the whole step; the gather-only
    workload reports gathered rows/s."""
    cores = os.cpu_count() or 1
    out = {"kind": "oracle", "cores": cores}
    for label, threads in (("single_thread", 1), ("all_cores", cores)):
        p = oracle_parts(w, T, ids, R, B, k, fmt, budget_s, threads)
        t = p["embed_s"] + p["wire_s"] + p["lm_s"]
        if B:
            out[label] = {"value": B / t, "unit": UNIT, "threads": threads}
        else:
            out[label] = {"value": len(ids) / max(p["embed_s"], 1e-9), "unit": "rows/s", "threads": threads}
        out["sample"] = p["sample"]
    out["value"] = out["all_cores"]["value"]
    out["unit"] = out["all_cores"]["unit"]
    return out


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    w = wl.WORKLOADS[args.workload]
    B = args.batch or (w.batches[0] if w.batches else 1)
    k = w.k or 10
    fmt = w.wire[0] if w.wire else wl.WIRE_F16
    T = wl.table_for(w)
    ids = wl.ids_for(w) if w.n_ids else np.zeros(1, np.int32)
    R = wl.residuals_for(w, B)
    threads = os.cpu_count() or 1
    steps = args.steps or 3
    per_step_budget = max(2.0, min(20.0, 150.0 / max(1, steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_rate(w, T, ids, R, B, k, fmt, min(1.0, per_step_budget), threads)
    rates, sample = [], ""
    for _ in range(steps):
        r, sample = oracle_rate(w, T, ids, R, B, k, fmt, per_step_budget, threads)
        rates.append(r)
    value = statistics.median(rates)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * B / value, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, B, k, fmt, w.n_ids or 1, world, args.untied, args.raw_logits),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------------------
# per-workload entries of the `configs` block
# ---------------------------------------------------------------------------

def _free():
    import gc

    import torch
    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def lm_measure(c, key, peak, peak_src, seconds, sampler, records, label=None):
    """The lm_head call of context `c` as a roofline measurement: a CUDA graph
    of GRAPH_CALLS back-to-back calls (table copies alternating) replayed,
    or eager calls when the table is flushed from L2 before every call or
    --eager asks for them."""
    if c.policy == "flush" or EAGER:
        m = measure(c, lambda i: call(c.lm_by_copy[i % len(c.lm_by_copy)]), seconds, sampler)
    else:
        g = graph_of([c.lm_by_copy[i % len(c.lm_by_copy)] for i in range(GRAPH_CALLS)])
        m = measure(c, lambda i: g.replay(), seconds, sampler, calls_per_body=GRAPH_CALLS)
        del g
    launch = (f"a CUDA graph of {GRAPH_CALLS} back-to-back calls, replayed"
              if not (c.policy == "flush" or EAGER) else "eager calls")
    kern = f"{'lhs_logits' if c.raw else 'lhs_logits_topk'} call ({c.lm_launches} kernels)"
    e = roofline_entry(key, kern, m, lm_bytes(c.w, c.B, c.k, c.raw), peak, peak_src, records)
    e["launch"] = launch
    e["batch"], e["k"] = c.B, c.k
    e["residuals_per_s"] = c.B / (m["avg_us"] * 1e-6)
    return e


def config_tiny(dev, peak, peak_src, seconds, sampler, records, cpu_budget):
    """C1: parity + latency case (8 MiB f32 table, flushed out of L2)."""
    c = setup("tiny", None, dev)
    w = c.w
    ent = {"workload": w.name, "kind": "latency (the table fits in L2; flushed before every call)",
           "table_bytes": w.table_bytes, "lm_batch": c.B, "k": c.k}
    t0 = time.time()
    ent["step_us"] = latency(c, lambda i: run_step(c, i), 200)
    ent["lm_head_us"] = latency(c, lambda i: call(c.lm_call), 200)
    ent["embed_us"] = latency(c, lambda i: call(c.embed_by_copy[0]), 200)
    import torch
    for fmt, fname in ((wl.WIRE_F16, "f16"), (wl.WIRE_I8, "i8")):
        c.fmt = fmt
        c.wire_bytes = c.lhs.lhs_wire_bytes(fmt, c.B, w.hidden)
        c.wire_buf = torch.empty(c.wire_bytes, dtype=torch.uint8, device=dev)
        enc, dec = wire_calls(c)
        ent[f"wire_{fname}_encode_us"] = latency(c, lambda i: call(enc), 200)
        ent[f"wire_{fname}_decode_us"] = latency(c, lambda i: call(dec), 200)
    ent["clocks"] = sampler.window(t0, time.time())
    if cpu_budget:
        ent["cpu_baseline"] = cpu_baseline_entry(w, c.T_host, c.ids_host, c.R_host, c.B, c.k, wl.WIRE_F16,
                                                 cpu_budget)
    del c
    _free()
    return ent


def config_qwen05b(c, lm_entry, dev, cpu_entry):
    """C2: the headline workload; its lm_head roofline is the line's."""
    w = c.w
    ent = {"workload": w.name, "lm_batch": c.B, "k": c.k, "table_bytes": w.table_bytes,
           "l2": l2_note(c.policy), "roofline": lm_entry}
    ent["embed_us"] = latency(c, lambda i: call(c.embed_by_copy[i % len(c.embed_by_copy)]), 200)
    ent["embed_ids"] = c.n_ids
    ent["embed_distinct"] = int(len(np.unique(c.ids_host)))
    enc, dec = wire_calls(c)
    ent["wire_f16_encode_us"] = latency(c, lambda i: call(enc), 200)
    ent["wire_f16_decode_us"] = latency(c, lambda i: call(dec), 200)
    if cpu_entry:
        ent["cpu_baseline"] = cpu_entry
    return ent


def config_gemma_q8(dev, peak, peak_src, seconds, sampler, records, cpu_budget):
    """C3: Q8_0 gather of 8192 ids (latency), its steady state over 2^20
    ids of the same distribution (bandwidth), and the lm_head on the Q8_0
    table (batch 1, k 10)."""
    import ctypes

    import torch
    c = setup("gemma_q8", 1, dev)
    w = c.w
    L = c.L
    ent = {"workload": w.name, "table_bytes": w.table_bytes, "l2": l2_note(c.policy)}
    ent["embed_us"] = latency(c, lambda i: call(c.embed_by_copy[i % len(c.embed_by_copy)]), 200)
    ent["embed_ids"] = c.n_ids
    distinct = int(len(np.unique(c.ids_host)))
    ent["embed_distinct"] = distinct
    ent["embed_rows_per_s"] = c.n_ids / (ent["embed_us"]["avg_us"] * 1e-6)
    ent["embed_algorithmic_bytes"] = embed_bytes(w, c.n_ids, distinct)
    # steady state: 2^20 ids, Zipf over the same table
    n = 1 << 20
    ids_h = wl.zipf_ids(w.cid, n, w.vocab, w.zipf_s, w.session_vocab)
    ids = up(ids_h, dev)
    out = torch.empty((n, w.hidden), dtype=torch.float32, device=dev)
    dn = int(len(np.unique(ids_h)))
    args = [(L.lhs_embed, (ctypes.byref(t.c), ids.data_ptr(), n, ctypes.c_float(c.scale), out.data_ptr(),
                           c.err.data_ptr(), c.sptr)) for t in c.tables]
    m = measure(c, lambda i: call(args[i % len(args)]), seconds, sampler)
    g = roofline_entry("gemma_q8/gather_steady", "lhs_embed (1 kernel)", m, embed_bytes(w, n, dn), peak,
                       peak_src, records)
    g.update({"ids": n, "distinct": dn, "rows_per_s": n / (m["avg_us"] * 1e-6)})
    ent["gather_steady_state"] = g
    del out
    # the same gather written straight into an i8 wire message
    nb = c.lhs.lhs_wire_bytes(wl.WIRE_I8, n, w.hidden)
    buf = torch.empty(nb, dtype=torch.uint8, device=dev)
    args = [(L.lhs_embed_wire, (ctypes.byref(t.c), ids.data_ptr(), n, ctypes.c_float(c.scale), wl.WIRE_I8,
                                0, 0, 0, buf.data_ptr(), nb, c.err.data_ptr(), c.sptr)) for t in c.tables]
    m = measure(c, lambda i: call(args[i % len(args)]), seconds, sampler)
    g = roofline_entry("gemma_q8/embed_wire_i8_steady", "lhs_embed_wire i8 (1 kernel)", m,
                       n * 4 + dn * w.row_bytes + nb, peak, peak_src, records)
    g.update({"ids": n, "distinct": dn, "values_per_ms": n * w.hidden / (m["avg_us"] * 1e-3)})
    ent["embed_wire_i8_steady_state"] = g
    del buf, ids
    ent["lm_head"] = lm_measure(c, "gemma_q8/lm_head", peak, peak_src, seconds, sampler, records)
    if cpu_budget:
        ent["cpu_baseline"] = cpu_baseline_entry(w, c.T_host, c.ids_host, c.R_host, 0, c.k, wl.WIRE_F16,
                                                 cpu_budget)
    del c
    _free()
    return ent


def config_gemma31b(dev, peak, peak_src, seconds, sampler, records, cpu_budget):
    """C4: lm_head GEMV at batch 1 and 8, k 40, f16 table of 2.82 GB; i8
    wire round trip of the batch."""
    ent = {"workload": "gemma31b"}
    T = None
    for B in (1, 8):
        c = setup("gemma31b", B, dev, T_host=T)
        T = c.T_host
        ent["table_bytes"] = c.w.table_bytes
        ent["l2"] = l2_note(c.policy)
        ent[f"lm_head_b{B}"] = lm_measure(c, f"gemma31b/lm_head_b{B}", peak, peak_src, seconds, sampler,
                                          records)
        enc, dec = wire_calls(c)
        ent[f"wire_i8_encode_b{B}_us"] = latency(c, lambda i: call(enc), 200)
        ent[f"wire_i8_decode_b{B}_us"] = latency(c, lambda i: call(dec), 200)
        if cpu_budget and B == 8:
            ent["cpu_baseline"] = cpu_baseline_entry(c.w, T, c.ids_host, c.R_host, B, c.k, wl.WIRE_I8,
                                                     cpu_budget)
        del c
        _free()
    return ent


def config_batched(dev, peak, tflops, peak_src, seconds, sampler, records, cpu_budget):
    """C5: 256 bf16 residuals against a bf16 table of 2.68 GB on tcgen05,
    k 50; f16 wire encode of the batch."""
    c = setup("batched", 256, dev)
    w = c.w
    ent = {"workload": w.name, "table_bytes": w.table_bytes, "l2": l2_note(c.policy)}
    e = lm_measure(c, "batched/lm_head", peak, peak_src, seconds, sampler, records)
    flops = 2.0 * c.B * w.vocab * w.hidden
    tf = flops / (e["avg_us"] * 1e-6) / 1e12
    e["roofline_tensor"] = {"bound": "tensor", "achieved": tf, "peak": tflops, "unit": "TFLOP/s",
                            "frac": tf / tflops, "peak_source": f"{peak_src} bf16_tflops_sustained",
                            "flops": flops}
    ent["lm_head"] = e
    enc, dec = wire_calls(c)
    ent["wire_f16_encode_us"] = latency(c, lambda i: call(enc), 200)
    ent["wire_f16_decode_us"] = latency(c, lambda i: call(dec), 200)
    if cpu_budget:
        ent["cpu_baseline"] = cpu_baseline_entry(w, c.T_host, c.ids_host, c.R_host, c.B, c.k, wl.WIRE_F16,
                                                 cpu_budget)
    del c
    _free()
    return ent


CODEC_SEQ, CODEC_HIDDEN = 65536, 5376


def config_codec(dev, peak, peak_src, seconds, sampler, records):
    """Wire codecs in steady state: 65,536 positions x 5,376 (f32 in, f16 /
    i8 message; >= 1 GB moved per call), seeded N(0, sigma^2) rows with
    sigma ~ U[0.5, 8]."""
    import ctypes

    import torch

    import embedding_lookup_tied_gb300 as lhs
    S, H = CODEC_SEQ, CODEC_HIDDEN
    c = Ctx()
    c.policy = "stream"
    c.stream = torch.cuda.current_stream(dev)
    c.err = torch.zeros(1, dtype=torch.int32, device=dev)
    x = up(wl.residuals(900, S, H, (0.5, 8.0)), dev)
    dec = torch.empty_like(x)
    L = lhs.lib()
    sp = c.stream.cuda_stream
    ent = {"seq_len": S, "hidden": H, "input": "f32 N(0, sigma^2), sigma ~ U[0.5, 8] per position"}
    for fmt, fname in ((wl.WIRE_F16, "f16"), (wl.WIRE_I8, "i8")):
        nb = lhs.lhs_wire_bytes(fmt, S, H)
        buf = torch.empty(nb, dtype=torch.uint8, device=dev)
        enc = (L.lhs_wire_encode, (fmt, x.data_ptr(), lhs.LHS_F32, S, H, 0, 0, 0, buf.data_ptr(), nb,
                                   c.err.data_ptr(), sp))
        dca = (L.lhs_wire_decode, (fmt, buf.data_ptr(), nb, S, H, dec.data_ptr(), c.err.data_ptr(), sp))
        m = measure(c, lambda i: call(enc), seconds, sampler)
        ent[f"{fname}_encode"] = roofline_entry(f"codec/{fname}_encode", f"lhs_wire_encode {fname} (1 kernel)",
                                                m, S * H * 4 + nb, peak, peak_src, records)
        m = measure(c, lambda i: call(dca), seconds, sampler)
        ent[f"{fname}_decode"] = roofline_entry(f"codec/{fname}_decode", f"lhs_wire_decode {fname} (1 kernel)",
                                                m, nb + S * H * 4, peak, peak_src, records)
        del buf
    del x, dec
    _free()
    return ent


# ---------------------------------------------------------------------------

SWEEP_HIDDEN = (2560, 4096, 5120, 5376)   # ADR-0009 benchmark sizes
SWEEP_SEQ = (1, 32, 256, 65536)


def run_sweep(dev, peak):
    """Steady-state numbers for the steps that take a few microseconds at
    the configs' sizes: the gather over 2^20 Zipf ids of the gemma_q8 and
    qwen05b tables, and f16 / i8 encode and decode over the ADR-0009 sizes.
    Points moving >= 1 GB per call report a bandwidth fraction; the others
    are latency (their bytes sit in L2 between iterations)."""
    import ctypes

    import torch

    import embedding_lookup_tied_gb300 as lhs

    def t_us(fn, n):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            fn()
        e1.record()
        e1.synchronize()
        return e0.elapsed_time(e1) * 1e3 / n

    def emit(kind, cfg, us, nbytes):
        d = {"sweep": kind, "config": cfg, "us_per_call": us, "algorithmic_bytes": nbytes,
             "gbs": nbytes / (us * 1e-6) / 1e9}
        if nbytes >= 1e9:
            d["frac_of_measured_hbm"] = d["gbs"] / peak
        else:
            d["latency_only"] = True
        print(json.dumps(d), flush=True)

    L = lhs.lib()
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    sp = torch.cuda.current_stream(dev).cuda_stream
    n_ids = 1 << 20
    for name in ("gemma_q8", "qwen05b"):
        w = wl.WORKLOADS[name]
        T = wl.table_for(w)
        tab = lhs.lhs_table_init(up(T, dev), w.vocab, w.hidden, w.dtype)
        ids_h = wl.zipf_ids(w.cid, n_ids, w.vocab, w.zipf_s, w.session_vocab)
        ids = up(ids_h, dev)
        out = torch.empty((n_ids, w.hidden), dtype=torch.float32, device=dev)
        distinct = len(np.unique(ids_h))
        args = (ctypes.byref(tab.c), ids.data_ptr(), n_ids, ctypes.c_float(float(w.embed_scale)),
                out.data_ptr(), err.data_ptr(), sp)
        us = t_us(lambda: L.lhs_embed(*args), 10)
        nbytes = embed_bytes(w, n_ids, distinct)
        emit("gather", {"table": name, "ids": n_ids, "distinct": distinct, "hidden": w.hidden}, us, nbytes)
        # the same gather through the distinct ids (each distinct row decoded once)
        dws = torch.empty(lhs.lib().lhs_embed_dedup_workspace(ctypes.byref(tab.c), n_ids), dtype=torch.uint8,
                          device=dev)
        da = (ctypes.byref(tab.c), ids.data_ptr(), n_ids, ctypes.c_float(float(w.embed_scale)), out.data_ptr(),
              dws.data_ptr(), dws.numel(), err.data_ptr(), sp)
        us = t_us(lambda: L.lhs_embed_dedup(*da), 10)
        emit("gather_dedup", {"table": name, "ids": n_ids, "distinct": distinct, "hidden": w.hidden}, us, nbytes)
        del out, dws
        # the gather written straight into f16 / i8 wire messages
        for fmt, fname in ((lhs.LHS_WIRE_F16, "f16"), (lhs.LHS_WIRE_I8, "i8")):
            nb = lhs.lhs_wire_bytes(fmt, n_ids, w.hidden)
            buf = torch.empty(nb, dtype=torch.uint8, device=dev)
            wa = (ctypes.byref(tab.c), ids.data_ptr(), n_ids, ctypes.c_float(float(w.embed_scale)), fmt,
                  0, 0, 0, buf.data_ptr(), nb, err.data_ptr(), sp)
            us = t_us(lambda: L.lhs_embed_wire(*wa), 10)
            emit("embed_wire", {"table": name, "format": fname, "ids": n_ids, "distinct": distinct,
                                "hidden": w.hidden}, us, n_ids * 4 + distinct * w.row_bytes + nb)
            del buf
        del T, tab
        torch.cuda.empty_cache()
    for H in SWEEP_HIDDEN:
        for S in SWEEP_SEQ:
            x = torch.randn((S, H), dtype=torch.float32, device=dev)
            dec = torch.empty_like(x)
            for fmt, fname in ((lhs.LHS_WIRE_F16, "f16"), (lhs.LHS_WIRE_I8, "i8")):
                nb = lhs.lhs_wire_bytes(fmt, S, H)
                buf = torch.empty(nb, dtype=torch.uint8, device=dev)
                ea = (fmt, x.data_ptr(), lhs.LHS_F32, S, H, 0, 0, 0, buf.data_ptr(), nb, err.data_ptr(), sp)
                da = (fmt, buf.data_ptr(), nb, S, H, dec.data_ptr(), err.data_ptr(), sp)
                n = 10 if S == 65536 else 200
                us = t_us(lambda: L.lhs_wire_encode(*ea), n)
                emit("wire_encode", {"format": fname, "seq_len": S, "hidden": H}, us, S * H * 4 + nb)
                us = t_us(lambda: L.lhs_wire_decode(*da), n)
                emit("wire_decode", {"format": fname, "seq_len": S, "hidden": H}, us, nb + S * H * 4)
                del buf
            del x, dec
            torch.cuda.empty_cache()
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"error word {int(err.item())} in the sweep")
    return 0


def wire_agreement(lhs, tab, x, k, fmt):
    """Per-residual top-k agreement of decode(encode(x)) with x on the GPU:
    (ordered-equal flags, same-set flags), numpy bool arrays [B].
    x: f32 CUDA tensor [B, H]."""
    import torch
    ref, _, _, e0 = lhs.lhs_logits_topk(tab, x, k, want_probs=False)
    buf, e1 = lhs.lhs_wire_encode(fmt, x)
    y, e2 = lhs.lhs_wire_decode(fmt, buf, x.shape[0], x.shape[1])
    got, _, _, e3 = lhs.lhs_logits_topk(tab, y, k, want_probs=False)
    torch.cuda.synchronize()
    for e in (e0, e1, e2, e3):
        if int(e.item()) != 0:
            raise RuntimeError(f"error word {int(e.item())}")
    a, b = ref.cpu().numpy(), got.cpu().numpy()
    ordered = np.all(a == b, axis=1)
    same_set = np.array([set(r) == set(g) for r, g in zip(a, b)])
    return ordered, same_set


def run_wire_accuracy(dev):
    """ADR-0009 Validation: f16 wire must keep the top-5 tokens, i8 the top-1,
    measured on synthetic tables and residuals of the C4 and C5 shapes."""
    import torch

    import embedding_lookup_tied_gb300 as lhs
    for name, B in (("gemma31b", 64), ("batched", 256)):
        w = wl.WORKLOADS[name]
        T = wl.table_for(w)
        t = torch.from_numpy(T.view(np.int16)).to(dev)
        del T
        tab = lhs.lhs_table_init(t, w.vocab, w.hidden, w.dtype)
        R = wl.residuals_for(w, B)
        xv = R if w.resid_dtype == wl.F32 else (R.astype(np.uint32) << 16).view(np.float32)  # bf16 -> f32, exact
        x = torch.from_numpy(np.ascontiguousarray(xv)).to(dev)
        for fmt, fname, k in ((lhs.LHS_WIRE_F16, "f16", 5), (lhs.LHS_WIRE_I8, "i8", 1)):
            ordered, same_set = wire_agreement(lhs, tab, x, k, fmt)
            print(json.dumps({"wire_accuracy": fname, "workload": name, "residuals": B, "top_k": k,
                              "agreement_ordered": float(ordered.mean()),
                              "agreement_set": float(same_set.mean()),
                              "data": "synthetic table and residuals"}), flush=True)
        del t, tab
        torch.cuda.empty_cache()
    return 0


def run_profile_case(case, dev, warm=3, calls=2):
    """`warm` then `calls` eager calls of one measurement (the sizes of the
    timed loops), for an ncu launch list; prints what ran."""
    import ctypes

    import torch

    import embedding_lookup_tied_gb300 as lhs
    parts = case.split(":")
    kind = parts[0]
    L = lhs.lib()
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    sp = torch.cuda.current_stream(dev).cuda_stream
    if kind == "lm_head":
        vocab = int(parts[2]) if len(parts) > 2 and parts[2] else None
        batch = int(parts[3]) if len(parts) > 3 else None
        c = setup(parts[1], batch, dev, vocab)
        fn = lambda i: call(c.lm_by_copy[i % len(c.lm_by_copy)])
        what = {"workload": c.w.name, "vocab": c.w.vocab, "batch": c.B, "k": c.k,
                "kernels_per_call": c.lm_launches}
    elif kind in ("gather", "embed_wire_i8"):
        w = wl.WORKLOADS[parts[1]]
        tab = lhs.lhs_table_init(up(wl.table_for(w), dev), w.vocab, w.hidden, w.dtype)
        n_ids = int(parts[2]) if len(parts) > 2 and parts[2] else 1 << 20
        ids = up(wl.zipf_ids(w.cid, n_ids, w.vocab, w.zipf_s, w.session_vocab), dev)
        scale = ctypes.c_float(float(w.embed_scale))
        if kind == "gather":
            out = torch.empty((n_ids, w.hidden), dtype=torch.float32, device=dev)
            args = (ctypes.byref(tab.c), ids.data_ptr(), n_ids, scale, out.data_ptr(), err.data_ptr(), sp)
            fn = lambda i: L.lhs_embed(*args)
        else:
            nb = lhs.lhs_wire_bytes(lhs.LHS_WIRE_I8, n_ids, w.hidden)
            buf = torch.empty(nb, dtype=torch.uint8, device=dev)
            args = (ctypes.byref(tab.c), ids.data_ptr(), n_ids, scale, lhs.LHS_WIRE_I8, 0, 0, 0, buf.data_ptr(),
                    nb, err.data_ptr(), sp)
            fn = lambda i: L.lhs_embed_wire(*args)
        what = {"workload": w.name, "ids": n_ids, "kernels_per_call": 1}
    elif kind == "codec":
        fmt = {"f16": lhs.LHS_WIRE_F16, "i8": lhs.LHS_WIRE_I8}[parts[1]]
        seq, H = (int(parts[3]) if len(parts) > 3 and parts[3] else 65536), 5376
        x = torch.from_numpy(wl.residuals(77, seq, H, (0.5, 8.0))).to(dev)
        nb = lhs.lhs_wire_bytes(fmt, seq, H)
        buf = torch.empty(nb, dtype=torch.uint8, device=dev)
        enc = (x.data_ptr(), lhs.LHS_F32, seq, H, 0, 0, 0, buf.data_ptr(), nb, err.data_ptr(), sp)
        dec_out = torch.empty((seq, H), dtype=torch.float32, device=dev)
        dec = (buf.data_ptr(), nb, seq, H, dec_out.data_ptr(), err.data_ptr(), sp)
        assert L.lhs_wire_encode(fmt, *enc) == 0
        fn = (lambda i: L.lhs_wire_encode(fmt, *enc)) if parts[2] == "encode" else (lambda i: L.lhs_wire_decode(fmt, *dec))
        what = {"format": parts[1], "op": parts[2], "seq_len": seq, "hidden": H, "kernels_per_call": 1}
    else:
        raise SystemExit(f"unknown profile case {case}")
    for i in range(warm + calls):
        rc = fn(i)
        if rc not in (None, 0):
            raise RuntimeError(f"{case}: call returned {rc}")
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"{case}: error word {int(err.item())}")
    print(json.dumps({"profile_case": case, "warm_calls": warm, "calls": calls, **what}), flush=True)
    return 0


def main(argv=None):
    global EAGER
    args = parse_args(argv)
    EAGER = args.eager
    rank, world, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.sweep:
        import torch
        torch.cuda.set_device(local)
        return run_sweep(torch.device("cuda", local), load_peaks()[0])
    if args.profile_case:
        import torch
        torch.cuda.set_device(local)
        return run_profile_case(args.profile_case, torch.device("cuda", local))
    if args.wire_accuracy:
        import torch
        torch.cuda.set_device(local)
        return run_wire_accuracy(torch.device("cuda", local))
    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    peak, tflops, peak_src = load_peaks()
    records = load_traffic_records()
    sampler = ClockSampler(torch.cuda.current_device()).start()
    try:
        c = setup(args.workload, args.batch, dev, args.vocab, args.untied, args.raw_logits)
        steps = args.steps or default_steps(args.workload)
        warmup = max(3, args.warmup)
        ms, step_win = time_device(c, steps, warmup, world)
        ms = max_over_ranks(ms, world, dev)
        default_b = c.w.batches[0] if c.w.batches else 1
        variant = bool(args.vocab or args.raw_logits or args.untied
                       or (args.batch and not (c.w.name == "gemma31b" and args.batch in (1, 8))
                           and args.batch != default_b))
        if variant:
            key = f"{c.w.name}/lm_head_variant"
        elif c.w.name == "gemma31b":
            key = f"gemma31b/lm_head_b{c.B}"
        else:
            key = f"{c.w.name}/lm_head"
        lm = lm_measure(c, key, peak, peak_src, args.roofline_seconds, sampler, records)
        e2e_steps = max(20, min(steps, 2000))
        e2e_graph = not args.e2e_eager
        e2e_ms, h2d, d2h = time_e2e(c, e2e_steps, graph=e2e_graph)
        e2e_ms = max_over_ranks(e2e_ms, world, dev)
        value = world * c.B / (ms / 1e3)
        roof = {k: v for k, v in lm.items() if k not in ("batch", "k", "residuals_per_s")}
        step_clocks = sampler.window(*step_win)
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
            "warmup": warmup, "ms_per_step": ms, "higher_is_better": True,
            "launch": ("eager calls" if (args.eager or c.policy == "flush") else
                       "CUDA graphs of up to 10 consecutive steps (their calls captured once), replayed "
                       "to make exactly `steps` steps"),
            "scaling": "weak", "vs_baseline": None,
            "dtype": {wl.F32: "f32", wl.F16: "f16", wl.BF16: "bf16", wl.Q8_0: "q8_0"}[c.w.dtype]
                     + "-table/f32-accumulate",
            "data": "synthetic",
            "config": workload_config(c.w, c.B, c.k, c.fmt, c.n_ids, world, c.untied, c.raw),
            "hbm_gbs_step": world * step_bytes(c) / (ms / 1e3) / 1e9,
            "embed_rows_per_s": world * c.n_ids / (ms / 1e3),
            "roofline": roof,
            "gpu_launches": c.launches_per_step * steps,
            "e2e": {"value": world * c.B / (e2e_ms / 1e3), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "ms_per_step": e2e_ms,
                    "step": "embed, lm_head top-k, wire encode and wire decode, as in the device step; "
                            "the embeddings copied back on a second stream while the lm_head runs",
                    "launch": ("one CUDA graph per step (the copies and the calls, captured once)" if e2e_graph
                               else "eager calls")},
        }
        if c.gemm:
            flops = 2.0 * c.B * c.w.vocab * c.w.hidden
            tf = flops / (lm["avg_us"] * 1e-6) / 1e12
            line["roofline_tensor"] = {"bound": "tensor", "achieved": tf, "peak": tflops, "unit": "TFLOP/s",
                                       "frac": tf / tflops, "peak_source": f"{peak_src} bf16_tflops_sustained",
                                       "flops": flops}
        cpu_head = None
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            cpu_head = cpu_baseline_entry(c.w, c.T_host, c.ids_host, c.R_host, c.B, c.k, c.fmt, args.cpu_budget_s)
            line["cpu_baseline"] = dict(cpu_head)
        configs = {}
        if not args.no_configs and not variant:
            want = [s.strip() for s in args.configs.split(",") if s.strip()]
            sub = 0.0 if (args.no_cpu_baseline or rank != 0 or world != 1) else args.cpu_budget_s / 3
            if "qwen05b" in want and c.w.name == "qwen05b":
                configs["qwen05b"] = config_qwen05b(c, roof, dev, cpu_head)
            del c
            _free()
            for name in want:
                if name in configs:
                    continue
                if name == "tiny":
                    configs[name] = config_tiny(dev, peak, peak_src, args.roofline_seconds, sampler, records, sub)
                elif name == "qwen05b":
                    cq = setup("qwen05b", None, dev)
                    lq = lm_measure(cq, "qwen05b/lm_head", peak, peak_src, args.roofline_seconds, sampler,
                                    records)
                    configs[name] = config_qwen05b(cq, lq, dev, None)
                    del cq
                    _free()
                elif name == "gemma_q8":
                    configs[name] = config_gemma_q8(dev, peak, peak_src, args.roofline_seconds, sampler,
                                                    records, sub)
                elif name == "gemma31b":
                    configs[name] = config_gemma31b(dev, peak, peak_src, args.roofline_seconds, sampler,
                                                    records, sub)
                elif name == "batched":
                    configs[name] = config_batched(dev, peak, tflops, peak_src, args.roofline_seconds, sampler,
                                                   records, sub)
                elif name == "codec":
                    configs[name] = config_codec(dev, peak, peak_src, args.roofline_seconds, sampler, records)
        all_loops = summarize_clocks(list(sampler.samples))
    finally:
        sampler.stop()
    # the step loop itself is too short for the 200 ms sampler; the line's
    # clock record covers the whole run (every timed loop), and the step
    # loop's own samples are listed beside it
    clocks = dict(all_loops)
    clocks["scope"] = "every sample of the run (all timing loops)"
    clocks["step_loop"] = step_clocks
    clocks["lm_head_loop"] = lm["clocks"]
    line["clocks"] = clocks
    if configs:
        line["configs"] = configs
    if rank == 0:
        print(json.dumps(line))
    barrier(world)
    return 0


if __name__ == "__main__":
    sys.exit(main())
