"""Seeded synthetic inputs for the embed / tied lm_head hot path.

This module only draws numbers and lays them out in the table / id /
residual formats the service reads; it holds none of the service's
arithmetic.  Both sides — the oracle (test infrastructure) and the CUDA
path — consume what it returns, so neither imports the other.

Every draw comes from ``numpy.random.default_rng`` seeded with
``[config_id, purpose(, chunk)]``: purpose 0 = table, 1 = token ids,
2 = residuals, 3 = per-row residual scales.  Large tables are drawn in
fixed-size chunks with their own child seeds, so the result does not depend
on how many threads draw them.

The five workloads mirror the pages' settings (sizes quoted on the pages,
distributions chosen here and stated in the design notes):
  tiny          f32 8192 x 256                       (parity / latency case)
  qwen05b       bf16 151,936 x 896   (HELIX §1, §3: Qwen2.5-0.5B table and a
                                      628-token session touching 109 ids)
  gemma_q8      Q8_0 262,144 x 768   (Port Spec: Q8_0 token_embd, sqrt(768))
  gemma31b      f16 262,144 x 5376   (ADR-0008: Gemma 4 31B lm_head shape)
  batched       bf16 262,144 x 5120  (ADR-0009: hidden 5120, seq_len 256)
"""
from __future__ import annotations

import concurrent.futures as cf
import math
import os
from dataclasses import dataclass, field

import numpy as np

# Table element types as numbered by the service's public header.
F32, F16, BF16, Q8_0 = 0, 1, 2, 3
WIRE_F32, WIRE_F16, WIRE_I8 = 0, 1, 2
DTYPE_NAMES = {F32: "f32", F16: "f16", BF16: "bf16", Q8_0: "q8_0"}

PURPOSE_TABLE, PURPOSE_IDS, PURPOSE_RESID, PURPOSE_SCALES = 0, 1, 2, 3
_CHUNK_ROWS = 1 << 14


@dataclass(frozen=True)
class Workload:
    cid: int                 # seed namespace
    name: str
    dtype: int               # table element type
    vocab: int
    hidden: int
    table_std: float         # N(0, std) entries (f32/f16/bf16 tables)
    n_ids: int               # tokens gathered per step
    id_sessions: int         # the ids are this many sequences of n_ids/id_sessions
    session_vocab: int       # >0: Zipf over a random subset of this many ids
    batches: tuple           # lm_head batch sizes
    resid_dtype: int         # F32 or BF16 residuals
    resid_scale_range: tuple | None  # per-row sigma ~ U[lo, hi]; None -> 1
    k: int                   # top-k
    wire: tuple              # wire formats exercised
    wire_rows: int           # positions per wire message (0 -> lm_head batch)
    zipf_s: float = 1.1
    q8_d_std: float = 0.002
    extra: dict = field(default_factory=dict)

    @property
    def row_bytes(self) -> int:
        if self.dtype == F32:
            return self.hidden * 4
        if self.dtype in (F16, BF16):
            return self.hidden * 2
        return self.hidden // 32 * 34

    @property
    def table_bytes(self) -> int:
        return self.vocab * self.row_bytes

    @property
    def embed_scale(self) -> np.float32:
        """sqrt(hidden) rounded once to binary32 (Port Spec forward graph)."""
        return np.float32(math.sqrt(float(self.hidden)))


WORKLOADS = {
    "tiny": Workload(0, "tiny", F32, 8192, 256, 0.02, 16, 1, 0, (4,), F32, None, 5,
                     (WIRE_F16, WIRE_I8), 0),
    "qwen05b": Workload(1, "qwen05b", BF16, 151936, 896, 0.02, 628, 1, 109, (1,), F32,
                        None, 10, (WIRE_F16,), 0),
    "gemma_q8": Workload(2, "gemma_q8", Q8_0, 262144, 768, 0.0, 8192, 64, 0, (), F32,
                         None, 0, (), 0),
    "gemma31b": Workload(3, "gemma31b", F16, 262144, 5376, 0.02, 0, 1, 0, (1, 8), F32,
                         (0.5, 8.0), 40, (WIRE_I8,), 0),
    "batched": Workload(4, "batched", BF16, 262144, 5120, 0.02, 0, 1, 0, (256,), BF16,
                        (0.5, 8.0), 50, (WIRE_F16,), 0),
}


def rng(cid: int, purpose: int, *more: int) -> np.random.Generator:
    return np.random.default_rng([cid, purpose, *more])


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even) -> uint16
    bit patterns.  Inputs are finite synthetic data."""
    u = np.array(x, np.float32, copy=True).view(np.uint32)
    r = (u >> 16) & 1
    u += np.uint32(0x7FFF)
    u += r
    u >>= 16
    return u.astype(np.uint16)


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _gauss_chunk(cid, ci, rows, hidden, std, dtype):
    g = rng(cid, PURPOSE_TABLE, ci)
    v = g.standard_normal((rows, hidden), dtype=np.float32)
    v *= np.float32(std)
    if dtype == F32:
        return v
    if dtype == F16:
        return v.astype(np.float16).view(np.uint16)
    return f32_to_bf16_bits(v)


def _q8_chunk(cid, ci, rows, hidden, d_std):
    g = rng(cid, PURPOSE_TABLE, ci)
    nb = hidden // 32
    q = g.integers(-127, 128, size=(rows, nb, 32), dtype=np.int16).astype(np.int8)
    d = np.abs(g.standard_normal((rows, nb), dtype=np.float32) * np.float32(d_std))
    d16 = d.astype(np.float16).view(np.uint8).reshape(rows, nb, 2)
    blk = np.empty((rows, nb, 34), np.uint8)
    blk[:, :, 0:2] = d16                  # f16 d, little-endian, first
    blk[:, :, 2:34] = q.view(np.uint8)    # 32 int8 codes
    return blk.reshape(rows, nb * 34)


def make_table(dtype: int, vocab: int, hidden: int, std: float = 0.02, cid: int = 0,
               q8_d_std: float = 0.002, threads: int | None = None) -> np.ndarray:
    """Table in its stored form: f32 -> float32 [V,H]; f16 / bf16 -> uint16 bit
    patterns [V,H]; Q8_0 -> uint8 [V, H/32*34] (blocks of f16 d then 32 int8).

    f32/f16/bf16 entries ~ N(0, std) rounded to the type; Q8_0 codes
    ~ U{-127..127}, d = f16(|N(0, q8_d_std)|).
    """
    if dtype == Q8_0 and hidden % 32:
        raise ValueError("Q8_0 needs hidden % 32 == 0")
    if dtype == F32:
        out = np.empty((vocab, hidden), np.float32)
    elif dtype in (F16, BF16):
        out = np.empty((vocab, hidden), np.uint16)
    else:
        out = np.empty((vocab, hidden // 32 * 34), np.uint8)
    chunks = [(ci, r0, min(vocab, r0 + _CHUNK_ROWS))
              for ci, r0 in enumerate(range(0, vocab, _CHUNK_ROWS))]

    def work(c):
        ci, r0, r1 = c
        if dtype == Q8_0:
            out[r0:r1] = _q8_chunk(cid, ci, r1 - r0, hidden, q8_d_std)
        else:
            out[r0:r1] = _gauss_chunk(cid, ci, r1 - r0, hidden, std, dtype)

    n = threads or _threads()
    if n == 1 or len(chunks) == 1:
        for c in chunks:
            work(c)
    else:
        with cf.ThreadPoolExecutor(n) as ex:
            list(ex.map(work, chunks))
    return out


def zipf_ids(cid: int, n: int, vocab: int, s: float = 1.1, session_vocab: int = 0,
             purpose: int = PURPOSE_IDS) -> np.ndarray:
    """n token ids, rank r drawn with P(r) ~ r^-s.  Ranks map to ids through a
    seeded permutation of the vocabulary (hot ids scattered), or — with
    ``session_vocab`` > 0 — through a uniform draw of that many distinct ids
    (a session that touches few rows, HELIX §2)."""
    g = rng(cid, purpose)
    m = session_vocab if session_vocab > 0 else vocab
    w = np.arange(1, m + 1, dtype=np.float64) ** (-s)
    cdf = np.cumsum(w)
    cdf /= cdf[-1]
    if session_vocab > 0:
        pool = g.choice(vocab, size=session_vocab, replace=False)
    else:
        pool = g.permutation(vocab)
    r = np.searchsorted(cdf, g.random(n), side="right")
    r = np.minimum(r, m - 1)
    return pool[r].astype(np.int32)


def residuals(cid: int, batch: int, hidden: int, scale_range=None,
              dtype: int = F32, std: float = 1.0):
    """Residuals N(0, sigma_b^2): sigma_b = std, or U[lo, hi] per row, in
    their stored form: f32 -> float32 [B,H]; bf16 -> uint16 bit patterns of
    bf16(N(0,1) * sigma_b)."""
    g = rng(cid, PURPOSE_RESID)
    x = g.standard_normal((batch, hidden), dtype=np.float32)
    if scale_range is not None:
        sg = rng(cid, PURPOSE_SCALES).uniform(scale_range[0], scale_range[1],
                                              size=(batch, 1)).astype(np.float32)
        x = x * sg
    else:
        x = x * np.float32(std)
    if dtype == F32:
        return x
    return f32_to_bf16_bits(x)


def table_for(w: Workload, threads: int | None = None) -> np.ndarray:
    return make_table(w.dtype, w.vocab, w.hidden, w.table_std, w.cid, w.q8_d_std,
                      threads)


def ids_for(w: Workload) -> np.ndarray:
    return zipf_ids(w.cid, w.n_ids, w.vocab, w.zipf_s, w.session_vocab)


def residuals_for(w: Workload, batch: int):
    return residuals(w.cid * 100 + batch, batch, w.hidden, w.resid_scale_range,
                     w.resid_dtype)
