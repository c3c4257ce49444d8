"""The oracle: a plain, slow CPU implementation of the embed / tied lm_head
service hot path, written from the pages that define it.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module.  The product path (``embedding_lookup_tied_gb300`` and its CUDA
library) never imports it; the two share no code.

The arithmetic lives in ``lhs_oracle.c`` (plain C, compiled with
``-O2 -ffp-contract=off``, no fast-math).  This module only builds that file
with gcc and marshals numpy arrays into it.

Sources (page title, section) — each function below names the one it follows:
  ADR-0008 "Remote Embeddings and lm_head Service"  (/v1/embed, /v1/logits,
           Error contract, Open Questions 1-2)
  HELIX "Columnar Embedding — Design Proposal" (§3 row-aligned table, §5 lm_head)
  "embedding-inference — Port Specification" (Q8_0 token_embd, forward graph)
  ADR-0009 "Wire Format Evolution: f16 Default + i8 Quantised Residuals"
           (Wire Layout, Trade-offs)

Every reading of a point the pages leave open is stated in ``lhs_oracle.c``
next to the code that takes it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# LHS_ORACLE_SRC names another C source to build the oracle from; only the
# mutation test sets it, to check that the pins fail on planted mistakes.
_SRC = os.environ.get("LHS_ORACLE_SRC") or os.path.join(_HERE, "lhs_oracle.c")
_LIB = (os.path.splitext(_SRC)[0] + ".so" if os.environ.get("LHS_ORACLE_SRC")
        else os.path.join(_HERE, "liblhs_oracle.so"))
_CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-Wall", "-Wextra"]

# Oracle's own numbering of table types, wire formats and error bits.
F32, F16, BF16, Q8_0, FP8_E4M3 = 0, 1, 2, 3, 4
WIRE_F32, WIRE_F16, WIRE_I8 = 0, 1, 2
ERR_BAD_TOKEN, ERR_MALFORMED, ERR_NONFINITE = 1, 2, 4
Q8_BLOCK, Q8_BLOCK_BYTES = 32, 34

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``lhs_oracle.c`` into ``liblhs_oracle.so`` (gcc, host arch)."""
    stale = (not os.path.exists(_LIB)
             or os.path.getmtime(_LIB) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm", "-lpthread"],
                       check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, f32, f64 = (ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                              ctypes.c_double)
        sig = {
            "orc_f16_value": (f64, [ctypes.c_uint16]),
            "orc_bf16_value": (f32, [ctypes.c_uint16]),
            "orc_f16_from_f32_sat": (ctypes.c_uint16, [f32]),
            "orc_f16_value_array": (None, [P, i64, P]),
            "orc_f16_from_f32_sat_array": (None, [P, i64, P]),
            "orc_row_bytes": (i64, [ctypes.c_int, i32]),
            "orc_embed": (ctypes.c_int, [P, ctypes.c_int, i64, i32, i64, P, i64,
                                         f32, P, P]),
            "orc_decode_rows": (None, [P, ctypes.c_int, i32, i64, i64, i64, P]),
            "orc_decode_bf16_array": (None, [P, i64, P]),
            "orc_decode_f16_array": (None, [P, i64, P]),
            "orc_logits": (ctypes.c_int, [P, ctypes.c_int, i64, i32, i64, P, i32,
                                          i64, i64, P, P, ctypes.c_int]),
            "orc_topk_f32": (ctypes.c_int, [P, i64, i32, P, P]),
            "orc_topk_f64": (ctypes.c_int, [P, i64, i32, P, P]),
            "orc_softmax_probs": (ctypes.c_int, [P, i64, f64, P, i32, P]),
            "orc_wire_bytes": (i64, [ctypes.c_int, i32, i32]),
            "orc_wire_encode": (ctypes.c_int, [ctypes.c_int, P, i32, i32,
                                               ctypes.c_uint32, ctypes.c_uint32,
                                               ctypes.c_uint32, P, P]),
            "orc_wire_decode": (ctypes.c_int, [ctypes.c_int, P, i64, i32, i32, P, P]),
            "orc_wire_response_bytes": (i64, [ctypes.c_int, i32, i32]),
            "orc_wire_encode_response": (ctypes.c_int, [ctypes.c_int, P, i32, i32, ctypes.c_uint32,
                                                        ctypes.c_float, P, P]),
            "orc_wire_decode_response": (ctypes.c_int, [ctypes.c_int, P, i64, i32, i32, P, P]),
            "orc_fp8_e4m3_value": (f64, [ctypes.c_uint8]),
            "orc_mixed_row_bytes": (i64, [ctypes.c_int, i32]),
            "orc_embed_mixed": (None, [P, i64, P, P, i64, i32, P, i64, f32, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# binary16 / bfloat16
# --------------------------------------------------------------------------

def f16_value(bits) -> np.ndarray:
    """IEEE 754 binary16 bit patterns -> exact values (float64)."""
    b = _c(np.atleast_1d(bits), np.uint16)
    out = np.empty(b.shape, np.float64)
    _load().orc_f16_value_array(_ptr(b), b.size, _ptr(out))
    return out


def bf16_to_f32(bits) -> np.ndarray:
    """bfloat16 bit patterns -> float32 values."""
    b = _c(np.atleast_1d(bits), np.uint16)
    out = np.empty(b.shape, np.float32)
    _load().orc_decode_bf16_array(_ptr(b), b.size, _ptr(out))
    return out


def f16_to_f32(bits) -> np.ndarray:
    """binary16 bit patterns -> float32 values (exact widening)."""
    b = _c(np.atleast_1d(bits), np.uint16)
    out = np.empty(b.shape, np.float32)
    _load().orc_decode_f16_array(_ptr(b), b.size, _ptr(out))
    return out


def f16_from_f32_sat(x) -> np.ndarray:
    """float32 -> binary16 bits, round-half-even, finite overflow -> +-65504
    (ADR-0009 Trade-offs: clamp-to-max), NaN -> 0x7E00."""
    a = _c(np.atleast_1d(x), np.float32)
    out = np.empty(a.shape, np.uint16)
    _load().orc_f16_from_f32_sat_array(_ptr(a), a.size, _ptr(out))
    return out


# --------------------------------------------------------------------------
# table layout and gather (HELIX §3; ADR-0008 /v1/embed; Port Spec forward graph)
# --------------------------------------------------------------------------

def row_bytes(dtype: int, hidden: int) -> int:
    """Bytes per table row: hidden*itemsize, Q8_0: hidden/32 blocks of 34 B."""
    return int(_load().orc_row_bytes(dtype, hidden))


def embed(table: np.ndarray, dtype: int, vocab: int, hidden: int, ids,
          scale: float):
    """out[t] = element(T[ids[t]]) * scale (binary32); bad ids -> zero row and
    the BAD_TOKEN bit.  ``table`` is the raw table bytes (any dtype view)."""
    tb = np.ascontiguousarray(table).view(np.uint8).reshape(-1)
    ids = _c(ids, np.int32)
    rb = row_bytes(dtype, hidden)
    if rb < 0 or tb.size < vocab * rb:
        raise ValueError("table too small for vocab x row_bytes")
    out = np.empty((ids.size, hidden), np.float32)
    err = ctypes.c_int32(0)
    rc = _load().orc_embed(_ptr(tb), dtype, vocab, hidden, rb, _ptr(ids),
                           ids.size, ctypes.c_float(np.float32(scale)), _ptr(out),
                           ctypes.byref(err))
    if rc:
        raise ValueError(f"orc_embed rc={rc}")
    return out, int(err.value)


def fp8_e4m3_value(codes) -> np.ndarray:
    """Exact values (float64) of OCP FP8 E4M3 codes."""
    c = _c(codes, np.uint8)
    L = _load()
    return np.array([L.orc_fp8_e4m3_value(int(v)) for v in c.reshape(-1)], np.float64).reshape(c.shape)


def mixed_row_bytes(dtype: int, hidden: int) -> int:
    return int(_load().orc_mixed_row_bytes(dtype, hidden))


def embed_mixed(data: np.ndarray, row_offset, row_dtype, vocab: int, hidden: int, ids,
                scale: float):
    """Gather from a table whose rows carry their own element type (HELIX §3
    sidecar): row r decoded as row_dtype[r] from data[row_offset[r]:]."""
    db = np.ascontiguousarray(data).view(np.uint8).reshape(-1)
    off = _c(row_offset, np.int64)
    dts = _c(row_dtype, np.uint8)
    ids = _c(ids, np.int32)
    if off.size < vocab or dts.size < vocab:
        raise ValueError("sidecar shorter than vocab")
    out = np.empty((ids.size, hidden), np.float32)
    err = ctypes.c_int32(0)
    _load().orc_embed_mixed(_ptr(db), db.size, _ptr(off), _ptr(dts), vocab, hidden, _ptr(ids), ids.size,
                            ctypes.c_float(np.float32(scale)), _ptr(out), ctypes.byref(err))
    return out, int(err.value)


def unique_ids(ids, vocab: int):
    """HELIX Appendix B "tokenize, dedupe, fetch": the distinct valid ids in
    ascending order, each position's index into them (-1 for an id outside
    [0, vocab)) and the BAD_TOKEN bit if there was one."""
    ids = np.asarray(ids, np.int64).reshape(-1)
    ok = (ids >= 0) & (ids < vocab)
    uniq, inv = np.unique(ids[ok], return_inverse=True)
    inverse = np.full(ids.size, -1, np.int32)
    inverse[ok] = inv.astype(np.int32)
    return uniq.astype(np.int32), inverse, (1 if not ok.all() else 0)


def decode_rows(table: np.ndarray, dtype: int, hidden: int, row0: int,
                nrows: int) -> np.ndarray:
    """Rows [row0, row0+nrows) of a table as float32 values."""
    tb = np.ascontiguousarray(table).view(np.uint8).reshape(-1)
    rb = row_bytes(dtype, hidden)
    if tb.size < (row0 + nrows) * rb:
        raise ValueError("rows out of range")
    out = np.empty((nrows, hidden), np.float32)
    _load().orc_decode_rows(_ptr(tb), dtype, hidden, rb, row0, nrows, _ptr(out))
    return out


# --------------------------------------------------------------------------
# lm_head (ADR-0008 /v1/logits; HELIX §5) and top-k / prob
# --------------------------------------------------------------------------

def logits(table: np.ndarray, dtype: int, vocab: int, hidden: int, x,
           v0: int = 0, v1: int | None = None, threads: int = 1,
           with_sumabs: bool = False):
    """logit[b][v] = sum_j T[v][j]*x[b][j] in binary64 for v in [v0, v1).

    ``x`` holds the residual VALUES as float32 [B, hidden] (decode bf16
    residuals with :func:`bf16_to_f32` first).  Returns float64 [B, v1-v0]
    (and sum_j |T[v][j]*x[b][j]| when ``with_sumabs``).
    """
    tb = np.ascontiguousarray(table).view(np.uint8).reshape(-1)
    x = _c(x, np.float32).reshape(-1, hidden)
    B = x.shape[0]
    v1 = vocab if v1 is None else v1
    rb = row_bytes(dtype, hidden)
    if tb.size < vocab * rb:
        raise ValueError("table too small")
    out = np.empty((B, v1 - v0), np.float64)
    sab = np.empty((B, v1 - v0), np.float64) if with_sumabs else None
    rc = _load().orc_logits(_ptr(tb), dtype, vocab, hidden, rb, _ptr(x), B, v0, v1,
                            _ptr(out), None if sab is None else _ptr(sab),
                            int(threads))
    if rc:
        raise RuntimeError(f"orc_logits rc={rc}")
    if with_sumabs:
        return out, sab
    return out


def topk_f32(logits_row, k: int):
    """Top-k of one float32 logits row: (value desc, id asc), NaN first."""
    lg = _c(logits_row, np.float32).reshape(-1)
    ids = np.empty(k, np.int32)
    vals = np.empty(k, np.float32)
    rc = _load().orc_topk_f32(_ptr(lg), lg.size, k, _ptr(ids), _ptr(vals))
    if rc:
        raise ValueError(f"orc_topk_f32 rc={rc}")
    return ids, vals


def topk_f64(logits_row, k: int):
    """Top-k of one float64 logits row under the same order."""
    lg = _c(logits_row, np.float64).reshape(-1)
    ids = np.empty(k, np.int32)
    vals = np.empty(k, np.float64)
    rc = _load().orc_topk_f64(_ptr(lg), lg.size, k, _ptr(ids), _ptr(vals))
    if rc:
        raise ValueError(f"orc_topk_f64 rc={rc}")
    return ids, vals


def softmax_probs(logits_row, temperature: float, ids) -> np.ndarray:
    """prob(id) = softmax(logits / T) over the full row, in binary64."""
    lg = _c(logits_row, np.float32).reshape(-1)
    ids = _c(ids, np.int32).reshape(-1)
    out = np.empty(ids.size, np.float64)
    rc = _load().orc_softmax_probs(_ptr(lg), lg.size, float(temperature), _ptr(ids),
                                   ids.size, _ptr(out))
    if rc:
        raise ValueError(f"orc_softmax_probs rc={rc}")
    return out


# --------------------------------------------------------------------------
# wire codecs (ADR-0009 Wire Layout)
# --------------------------------------------------------------------------

def wire_bytes(fmt: int, seq_len: int, hidden: int) -> int:
    return int(_load().orc_wire_bytes(fmt, seq_len, hidden))


def wire_encode(fmt: int, x, layer: int = 0, flags: int = 0, top_k: int = 0):
    """Encode float32 [seq_len, hidden] -> (bytes as uint8 array, err bits)."""
    x = _c(x, np.float32)
    if x.ndim != 2:
        raise ValueError("x must be [seq_len, hidden]")
    s, h = x.shape
    buf = np.zeros(wire_bytes(fmt, s, h), np.uint8)
    err = ctypes.c_int32(0)
    rc = _load().orc_wire_encode(fmt, _ptr(x), s, h, layer, flags, top_k, _ptr(buf),
                                 ctypes.byref(err))
    if rc:
        raise ValueError(f"orc_wire_encode rc={rc}")
    return buf, int(err.value)


def wire_response_bytes(fmt: int, seq_len: int, hidden: int) -> int:
    return int(_load().orc_wire_response_bytes(fmt, seq_len, hidden))


def wire_encode_response(fmt: int, x, layer: int = 0, latency_ms: float = 0.0):
    """Encode float32 [seq_len, hidden] as a single-layer response message
    ([layer][seq_len][latency_ms] header) -> (bytes as uint8 array, err bits)."""
    x = _c(x, np.float32)
    if x.ndim != 2:
        raise ValueError("x must be [seq_len, hidden]")
    s, h = x.shape
    buf = np.zeros(wire_response_bytes(fmt, s, h), np.uint8)
    err = ctypes.c_int32(0)
    rc = _load().orc_wire_encode_response(fmt, _ptr(x), s, h, layer, latency_ms, _ptr(buf),
                                          ctypes.byref(err))
    if rc:
        raise ValueError(f"orc_wire_encode_response rc={rc}")
    return buf, int(err.value)


def wire_decode_response(fmt: int, buf, seq_len: int, hidden: int, out=None):
    """Decode a single-layer response -> (float32 [seq_len, hidden], err
    bits).  On a malformed message ``out`` is returned untouched."""
    buf = _c(buf, np.uint8).reshape(-1)
    x = np.zeros((seq_len, hidden), np.float32) if out is None else out
    err = ctypes.c_int32(0)
    rc = _load().orc_wire_decode_response(fmt, _ptr(buf), buf.size, seq_len, hidden, _ptr(x),
                                          ctypes.byref(err))
    if rc:
        raise ValueError(f"orc_wire_decode_response rc={rc}")
    return x, int(err.value)


def wire_decode(fmt: int, buf, seq_len: int, hidden: int, out=None):
    """Decode a message -> (float32 [seq_len, hidden], err bits).  On a
    malformed message ``out`` is returned untouched."""
    buf = _c(buf, np.uint8).reshape(-1)
    x = np.zeros((seq_len, hidden), np.float32) if out is None else out
    err = ctypes.c_int32(0)
    rc = _load().orc_wire_decode(fmt, _ptr(buf), buf.size, seq_len, hidden, _ptr(x),
                                 ctypes.byref(err))
    if rc:
        raise ValueError(f"orc_wire_decode rc={rc}")
    return x, int(err.value)
