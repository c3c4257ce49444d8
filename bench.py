#!/usr/bin/env python3
"""Benchmark of the embed / tied lm_head service hot path on GB300.

One step = one pass of the whole hot path over one batch of the workload:
  embed gather of the workload's token ids (x sqrt(hidden)),
  tied lm_head projection with fused top-k (+ probabilities),
  wire encode + decode of the residual batch in the workload's format.
Inputs are seeded synthetic data (workloads/), resident in HBM before the
timed region.  The table is larger than L2, so each step streams it from HBM.

Prints one JSON line.  `value` is lm_head top-k residuals per second for the
whole job (all ranks).  Under torchrun every rank runs its own replica of the
workload (weak scaling; the path needs no exchange between GPUs).

  python bench.py [--workload qwen05b] [--steps K] [--warmup W]
  python bench.py --impl reference      # the CPU oracle, timed on host cores
"""
from __future__ import annotations

import argparse
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


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="lhs", choices=["lhs", "reference"])
    ap.add_argument("--workload", default="qwen05b", choices=sorted(wl.WORKLOADS))
    ap.add_argument("--batch", type=int, default=None, help="lm_head batch (default: workload's first)")
    ap.add_argument("--vocab", type=int, default=None,
                    help="override the workload's vocab rows (small cases for profiling)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    ap.add_argument("--untied", action="store_true",
                    help="lm_head on a second table of the same shape (an untied lm_head)")
    ap.add_argument("--e2e-eager", action="store_true",
                    help="time the end-to-end step as eager calls instead of replaying it as a CUDA graph")
    ap.add_argument("--raw-logits", action="store_true",
                    help="the step's lm_head call returns the full logits (raw-logits mode)")
    ap.add_argument("--wire-accuracy", action="store_true",
                    help="top-k agreement of logits from wire-decoded residuals with the "
                         "originals (f16: top-5, i8: top-1) on the gemma31b and batched workloads")
    ap.add_argument("--sweep", action="store_true",
                    help="steady-state sweep of the sub-10-us steps (gather, wire codecs): one "
                         "JSON line per point instead of the step line")
    return ap.parse_args()


def default_steps(name):
    # keep the device-timed region around 2-4 s (clock sampling needs >1 s)
    return {"tiny": 20000, "qwen05b": 20000, "gemma_q8": 20000, "gemma31b": 4000,
            "batched": 2000}[name]


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
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured", d
    except Exception:
        return FALLBACK_HBM_GBS, "fallback", {}


_REASON_COLS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the timed
    region runs."""

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
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
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, mx, reasons = [], [], set()
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(_REASON_COLS, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# workload setup
# ---------------------------------------------------------------------------

class Ctx:
    pass


def setup(name, batch, device, vocab=None, untied=False, raw=False):
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

    def up(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        return torch.from_numpy(a).to(device)

    c.T_host = wl.table_for(w)
    c.table = lhs.lhs_table_init(up(c.T_host), w.vocab, w.hidden, w.dtype)
    c.untied, c.raw = untied, raw
    if untied:
        # a second table, same shape and distribution, other seed
        c.lm_table = lhs.lhs_table_init(up(wl.make_table(w.dtype, w.vocab, w.hidden, 0.02, cid=w.cid + 50)),
                                        w.vocab, w.hidden, w.dtype)
    else:
        c.lm_table = c.table
    c.ids_host = wl.ids_for(w) if w.n_ids else wl.zipf_ids(w.cid, 1, w.vocab)
    c.R_host = wl.residuals_for(w, c.B)
    c.ids = up(c.ids_host)
    c.resid = up(c.R_host)
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
    # direct C-ABI argument lists (no per-call marshalling in the timed loop)
    import ctypes
    L = lhs.lib()
    tb = ctypes.byref(c.table.c)
    lb = ctypes.byref(c.lm_table.c)
    if raw:
        lm_call = (L.lhs_logits, (lb, c.resid.data_ptr(), rd, c.B, c.raw_out.data_ptr(), c.ws.data_ptr(),
                                  c.ws.numel(), c.err.data_ptr(), c.sptr))
    else:
        lm_call = (L.lhs_logits_topk, (lb, c.resid.data_ptr(), rd, c.B, c.k, ctypes.c_float(1.0),
                                       c.top_ids.data_ptr(), c.top_logits.data_ptr(),
                                       c.top_probs.data_ptr(), c.ws.data_ptr(), c.ws.numel(),
                                       c.err.data_ptr(), c.sptr))
    c.calls = [
        (L.lhs_embed, (tb, c.ids.data_ptr(), c.n_ids, ctypes.c_float(c.scale),
                       c.emb_out.data_ptr(), c.err.data_ptr(), c.sptr)),
        lm_call,
        (L.lhs_wire_encode, (c.fmt, c.resid.data_ptr(), rd, c.B, H, 0, 0, c.k,
                             c.wire_buf.data_ptr(), c.wire_bytes, c.err.data_ptr(), c.sptr)),
        (L.lhs_wire_decode, (c.fmt, c.wire_buf.data_ptr(), c.wire_bytes, c.B, H,
                             c.dec.data_ptr(), c.err.data_ptr(), c.sptr)),
    ]
    c.lm_call = c.calls[1]
    c.flush_l2 = w.table_bytes < 2 * L2_BYTES
    if c.flush_l2:
        c.flush_buf = torch.zeros(2 * L2_BYTES // 4, dtype=torch.int32, device=device)
    # kernels per step: embed 1, the lm_head call as the library reports it
    # for this plan, wire encode 1, decode 1
    lm = lhs.lhs_logits_topk_launches(c.lm_table, c.B, 0 if raw else c.k, rd)
    c.lm_launches = lm
    c.gemm = (w.dtype == wl.BF16 and w.resid_dtype == wl.BF16 and c.B > 8)
    c.launches_per_step = 1 + lm + 1 + 1
    return c


def run_step(c):
    for fn, args in c.calls:
        rc = fn(*args)
        if rc != 0:
            raise RuntimeError(f"{fn.__name__} -> {rc}")


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one lm_head
# call, from the ncu captures summarised under profiles/, with a digest of
# the kernel sources they were taken on: once the sources change, the
# recorded traffic no longer describes the kernel and is reported as null.
TRAFFIC_RECORDS = {
    # workload: (digest of the dominant kernel's sources, DRAM bytes per call, summary)
    "qwen05b": ("d013ab5bc4d85982", 275.64e6, "profiles/gemv_tc_qwen05b.md"),
    "batched": ("c58151cfb28be31f", 2.762e9, "profiles/gemm_tc_batched.md"),
}
# the files each recorded kernel is compiled from: a change to any of them
# voids its record
KERNEL_SOURCES = {
    "qwen05b": ("embedding_lookup_tied_gb300/csrc/lm_head.cu",
                "embedding_lookup_tied_gb300/csrc/lhs_internal.cuh"),
    "batched": ("embedding_lookup_tied_gb300/csrc/gemm_tc.cu",
                "embedding_lookup_tied_gb300/csrc/lm_head.cu",
                "embedding_lookup_tied_gb300/csrc/lhs_internal.cuh"),
}
L2_BYTES = 129 * 1024 * 1024


def kernel_digest(name) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[name]:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(name):
    rec = TRAFFIC_RECORDS.get(name)
    if rec is None:
        return None, "no ncu capture recorded for this workload"
    digest, nbytes, src = rec
    if kernel_digest(name) != digest:
        return None, f"kernel sources changed since the capture in {src}"
    return nbytes, src


def workload_config(w, B, k, fmt, n_ids, world, untied=False, raw=False):
    """The `config` object of the JSON line (both arms)."""
    flush = w.table_bytes < 2 * L2_BYTES
    return {"workload": w.name, "vocab": w.vocab, "hidden": w.hidden,
            "table_dtype": wl.DTYPE_NAMES[w.dtype], "table_bytes": w.table_bytes,
            "embed_ids": n_ids, "lm_batch": B, "k": k,
            "lm_table": "untied (second table, same shape)" if untied else "tied (the embedding table)",
            "lm_output": "raw logits [batch x vocab]" if raw else "top-k ids, logits, probs",
            "wire": {0: "f32", 1: "f16", 2: "i8"}[fmt],
            "l2": ("flushed before every timed iteration (a 258 MB buffer rewritten outside the "
                   "timed events): the table fits in L2" if flush else
                   "no flush: the table is larger than twice the L2 and is streamed every step"),
            "parallelism": f"replicas x{world}"}


def lm_bytes(c):
    """Algorithmic bytes of one lm_head call: every table row once, the
    residuals once, the top-k outputs once."""
    w = c.w
    relt = 4 if w.resid_dtype == wl.F32 else 2
    out = c.B * w.vocab * 4 if c.raw else c.B * c.k * 12
    return w.vocab * w.row_bytes + c.B * w.hidden * relt + out


def step_bytes(c):
    w = c.w
    relt = 4 if w.resid_dtype == wl.F32 else 2
    distinct = len(np.unique(c.ids_host)) if w.n_ids else 0
    embed = c.n_ids * (4 + w.hidden * 4) + distinct * w.row_bytes
    wire = 2 * (c.B * w.hidden * relt) + 2 * c.wire_bytes
    return lm_bytes(c) + embed + wire


# ---------------------------------------------------------------------------
# timing
# ---------------------------------------------------------------------------

def timed_loop(c, body, n):
    """Device time of `body` per iteration.  When the table fits in L2 a
    buffer larger than L2 is overwritten before every iteration, outside the
    timed events, so every iteration starts with the table in HBM."""
    import torch
    if not c.flush_l2:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(c.stream)
        for _ in range(n):
            body()
        e1.record(c.stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / n
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for a, b in ev:
        c.flush_buf.add_(1)
        a.record(c.stream)
        body()
        b.record(c.stream)
    ev[-1][1].synchronize()
    return sum(a.elapsed_time(b) for a, b in ev) / n


def time_device(c, steps, warmup, world):
    import torch
    for _ in range(warmup):
        run_step(c)
    torch.cuda.synchronize()
    if int(c.err.item()) != 0:
        raise RuntimeError(f"error word {int(c.err.item())} during warm-up")
    # lm_head call alone (the dominant kernel), events on its stream
    lm_steps = max(50, steps // 4)
    fn, args = c.lm_call
    for _ in range(5):
        fn(*args)
    torch.cuda.synchronize()
    lm_ms = timed_loop(c, lambda: fn(*args), lm_steps)
    # whole step
    barrier(world)
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    ms = timed_loop(c, lambda: run_step(c), steps)
    torch.cuda.synchronize()
    barrier(world)
    ck = clocks.stop()
    if int(c.err.item()) != 0:
        raise RuntimeError(f"error word {int(c.err.item())} in the timed region")
    return ms, lm_ms, ck


def time_e2e(c, steps, graph=False):
    """Same step through the public binding with HOST buffers: each step
    copies its inputs from pinned host memory and reads its results back.
    The step's inputs and outputs share one device buffer (and one pinned
    host mirror) laid out [ids | residuals | error word | lm_head outputs |
    wire message | embeddings], so a step is one host-to-device copy (ids,
    residuals and the zeroed error word), the calls, and one device-to-host
    copy (the error word and every output), all on the stream of the calls.
    (Copying the embeddings on a second stream, overlapped with the
    lm_head, measured slower: the per-step cross-stream waits cost more.)
    graph=True captures one step — copies and calls — in a CUDA graph and
    replays it, so the host's per-call launch cost leaves the loop."""
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
    parts += [("buf", c.wire_bytes), ("emb", c.n_ids * H * 4)]
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
    if c.raw:
        d_raw = view(d_io, "raw", c.B * c.w.vocab * 4, torch.float32, (c.B, c.w.vocab))
    else:
        d_tid = view(d_io, "tid", c.B * c.k * 4, torch.int32, (c.B, c.k))
        d_tlg = view(d_io, "tlg", c.B * c.k * 4, torch.float32, (c.B, c.k))
        d_tpr = view(d_io, "tpr", c.B * c.k * 4, torch.float32, (c.B, c.k))
    in_end = off["err"] + 4              # ids, residuals, error word
    out0 = off["err"]                    # error word and every output
    out1 = off["emb"] + c.n_ids * H * 4
    h2d = in_end
    d2h = out1 - out0

    def one():
        d_io[:in_end].copy_(h_io[:in_end], non_blocking=True)
        lhs.lhs_embed(c.table, d_ids, c.scale, out=d_emb, err=d_err)
        if c.raw:
            lhs.lhs_logits(c.lm_table, d_res, out=d_raw, ws=c.ws, err=d_err)
        else:
            lhs.lhs_logits_topk(c.lm_table, d_res, c.k, 1.0, ws=c.ws, ids=d_tid, logits=d_tlg, probs=d_tpr,
                                err=d_err)
        lhs.lhs_wire_encode(c.fmt, d_res, 0, 0, c.k, buf=d_buf, err=d_err)
        h_io[out0:out1].copy_(d_io[out0:out1], non_blocking=True)

    for _ in range(5):
        one()
    torch.cuda.synchronize()
    step = one
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            one()
        torch.cuda.synchronize()
        step = g.replay
        for _ in range(3):
            step()
        torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(c.stream)
    for _ in range(steps):
        step()
    e1.record(c.stream)
    e1.synchronize()
    if int(view(h_io, "err", 4, torch.int32, (1,)).item()) != 0:
        raise RuntimeError("error word set in the end-to-end loop")
    return e0.elapsed_time(e1) / steps, h2d, d2h


# ---------------------------------------------------------------------------
# the oracle on host cores (cpu_baseline and --impl reference)
# ---------------------------------------------------------------------------

def oracle_rate(w, T, ids, R, B, k, fmt, budget_s, threads):
    """Time the oracle on a bounded sample of one step: the full embed and
    wire work, and the lm_head over a slice of vocab rows; the lm_head time
    is scaled up to the full vocabulary.  Returns (residuals/s, sample)."""
    import oracle as orc
    xv = R if w.resid_dtype == wl.F32 else orc.bf16_to_f32(R)
    t0 = time.perf_counter()
    if w.n_ids:
        orc.embed(T, w.dtype, w.vocab, w.hidden, ids, w.embed_scale)
    buf, _ = orc.wire_encode(fmt, xv)
    orc.wire_decode(fmt, buf, B, w.hidden)
    t_fixed = time.perf_counter() - t0
    rows = min(64, w.vocab)
    t_lm = 0.0
    done = 0
    while True:
        # consecutive, disjoint slices of the vocabulary, growing until the
        # budget is spent or every row has been done once
        t1 = time.perf_counter()
        L = orc.logits(T, w.dtype, w.vocab, w.hidden, xv, v0=done, v1=done + rows,
                       threads=threads)
        for b in range(B):
            orc.topk_f64(L[b], min(k, rows))
        t_lm += time.perf_counter() - t1
        done += rows
        if t_lm + t_fixed >= budget_s or done >= w.vocab:
            break
        rows = min(rows * 2, 1 << 14, w.vocab - done)
    t_step = t_fixed + t_lm * (w.vocab / done)
    sample = (f"1 step: full embed ({w.n_ids} ids) + wire encode/decode; lm_head over "
              f"{done} of {w.vocab} vocab rows for {B} residual(s), time scaled x{w.vocab / done:.1f}")
    return B / t_step, sample


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

SWEEP_HIDDEN = (2560, 4096, 5120, 5376)   # ADR-0009 benchmark sizes
SWEEP_SEQ = (1, 32, 256, 65536)


def run_sweep(dev, peak):
    """Steady-state numbers for the steps that take a few microseconds at
    the configs' sizes: the gather over 2^20 Zipf ids of the gemma_q8 and
    qwen05b tables, and f16 / i8 encode and decode over the ADR-0009 sizes.
    Points moving >= 1 GB per call report a bandwidth fraction; the others
    are latency (their bytes sit in L2 between iterations)."""
    import torch

    import embedding_lookup_tied_gb300 as lhs

    def up(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        return torch.from_numpy(a).to(dev)

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
    import ctypes
    n_ids = 1 << 20
    for name in ("gemma_q8", "qwen05b"):
        w = wl.WORKLOADS[name]
        T = wl.table_for(w)
        tab = lhs.lhs_table_init(up(T), w.vocab, w.hidden, w.dtype)
        ids_h = wl.zipf_ids(w.cid, n_ids, w.vocab, w.zipf_s, w.session_vocab)
        ids = up(ids_h)
        out = torch.empty((n_ids, w.hidden), dtype=torch.float32, device=dev)
        distinct = len(np.unique(ids_h))
        args = (ctypes.byref(tab.c), ids.data_ptr(), n_ids, ctypes.c_float(float(w.embed_scale)),
                out.data_ptr(), err.data_ptr(), sp)
        us = t_us(lambda: L.lhs_embed(*args), 10)
        nbytes = n_ids * (4 + w.hidden * 4) + distinct * w.row_bytes
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
    """Fractions of residuals whose top-k ids from decode(encode(x)) equal
    those from x: (same ordered ids, same set).  x: f32 CUDA tensor [B, H]."""
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
    ordered = float(np.mean(np.all(a == b, axis=1)))
    same_set = float(np.mean([set(r) == set(g) for r, g in zip(a, b)]))
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
                              "agreement_ordered": ordered, "agreement_set": same_set,
                              "data": "synthetic table and residuals"}), flush=True)
        del t, tab
        torch.cuda.empty_cache()
    return 0


def main():
    args = parse_args()
    rank, world, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.sweep:
        import torch
        torch.cuda.set_device(local)
        return run_sweep(torch.device("cuda", local), load_peaks()[0])
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
    c = setup(args.workload, args.batch, dev, args.vocab, args.untied, args.raw_logits)
    steps = args.steps or default_steps(args.workload)
    ms, lm_ms, clocks = time_device(c, steps, max(3, args.warmup), world)
    ms = max_over_ranks(ms, world, dev)
    e2e_steps = max(20, min(steps // 10, 2000))
    e2e_graph = not args.e2e_eager
    e2e_ms, h2d, d2h = time_e2e(c, e2e_steps, graph=e2e_graph)
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    peak, peak_kind, _ = load_peaks()
    value = world * c.B / (ms / 1e3)
    lmb = lm_bytes(c)
    achieved = lmb / (lm_ms / 1e3) / 1e9
    traffic, traffic_src = (recorded_traffic(c.w.name) if not (args.vocab or args.raw_logits or args.untied)
                            else (None, "no capture recorded for this variant"))
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": {wl.F32: "f32", wl.F16: "f16", wl.BF16: "bf16", wl.Q8_0: "q8_0"}[c.w.dtype]
                 + "-table/f32-accumulate",
        "data": "synthetic",
        "config": workload_config(c.w, c.B, c.k, c.fmt, c.n_ids, world, c.untied, c.raw),
        "hbm_gbs_step": world * step_bytes(c) / (ms / 1e3) / 1e9,
        "embed_rows_per_s": world * c.n_ids / (ms / 1e3),
        "roofline": {"kernel": f"{'lhs_logits' if c.raw else 'lhs_logits_topk'} call ({c.lm_launches} kernels)",
                     "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": f"{peak_kind} hbm_gbs",
                     "traffic": traffic, "traffic_source": traffic_src,
                     "algorithmic_bytes": lmb, "avg_ms": lm_ms},
        "gpu_launches": c.launches_per_step * steps,
        "clocks": clocks,
        "e2e": {"value": world * c.B / (e2e_ms / 1e3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "ms_per_step": e2e_ms,
                "launch": ("one CUDA graph per step (the copies and the calls, captured once)" if e2e_graph
                           else "eager calls")},
    }
    if c.gemm:
        # a dense contraction near the ridge point: its tensor-core fraction too
        _, _, pk = load_peaks()
        flops = 2.0 * c.B * c.w.vocab * c.w.hidden
        tf = flops / (lm_ms / 1e3) / 1e12
        tpk = float(pk.get("bf16_tflops_sustained", pk.get("bf16_tflops", 1700.0)))
        line["roofline_tensor"] = {"bound": "tensor", "achieved": tf, "peak": tpk, "unit": "TFLOP/s",
                                   "frac": tf / tpk,
                                   "peak_source": "measured bf16_tflops_sustained" if pk else "fallback",
                                   "flops": flops}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        r, sample = oracle_rate(c.w, c.T_host, c.ids_host, c.R_host, c.B, c.k, c.fmt,
                                args.cpu_budget_s, threads)
        line["cpu_baseline"] = {"value": r, "unit": UNIT, "cores": threads, "kind": "oracle",
                                "sample": sample}
    if rank == 0:
        print(json.dumps(line))
    barrier(world)
    return 0


if __name__ == "__main__":
    sys.exit(main())
