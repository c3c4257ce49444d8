"""Python binding of ``liblhs.so``, the GB300 embed / tied lm_head library.

Argument marshalling only: every step runs in the library's CUDA kernels.
The functions carry the C-ABI names (see ``include/lhs.h``) and take torch
CUDA tensors, which supply device memory and the stream.  There is no CPU
path: a missing library, a CPU tensor or a failed call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

LHS_OK = 0
LHS_ERR_INVALID_ARG = -1
LHS_ERR_BUFFER_TOO_SMALL = -2
LHS_ERR_UNSUPPORTED = -3
LHS_ERR_CUDA = -4
LHS_ERRBIT_BAD_TOKEN = 1
LHS_ERRBIT_MALFORMED = 2
LHS_ERRBIT_NONFINITE = 4
LHS_ERRBIT_TIMEOUT = 8
LHS_F32, LHS_F16, LHS_BF16, LHS_Q8_0, LHS_FP8_E4M3 = 0, 1, 2, 3, 4
LHS_WIRE_F32, LHS_WIRE_F16, LHS_WIRE_I8 = 0, 1, 2
LHS_NOALLOC_SCRATCH_BYTES = 4 * 1024 * 1024

LIB_PATH = _build.LIB

# Exported symbols of the C-ABI, in declaration order.
ABI_SYMBOLS = (
    "lhs_table_init", "lhs_table_info", "lhs_embed", "lhs_embed_wire", "lhs_embed_wire_response",
    "lhs_unique_ids_workspace",
    "lhs_unique_ids", "lhs_embed_dedup_workspace", "lhs_embed_dedup", "lhs_embed_mixed",
    "lhs_logits_topk_workspace",
    "lhs_logits_topk_launches", "lhs_logits_topk", "lhs_logits", "lhs_logits_topk_noalloc", "lhs_wire_bytes",
    "lhs_wire_encode",
    "lhs_wire_decode", "lhs_wire_response_bytes", "lhs_wire_encode_response", "lhs_wire_decode_response",
    "lhs_selftest_bounded_wait", "lhs_strerror",
    "lhs_last_cuda_error", "lhs_version",
)


class LhsError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = lib().lhs_strerror(status).decode()
        if status == LHS_ERR_CUDA:
            msg += f" (cudaError {lib().lhs_last_cuda_error()})"
        super().__init__(f"{where}: {msg} [{status}]")


class lhs_table(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("vocab", ctypes.c_int64),
                ("hidden", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("row_bytes", ctypes.c_int64)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library.  Raises if ``liblhs.so`` has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -m embedding_lookup_tied_gb300._build`")
    L = ctypes.CDLL(LIB_PATH)
    P, i32, i64, u32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                            ctypes.c_uint32, ctypes.c_size_t)
    T = ctypes.POINTER(lhs_table)
    sig = {
        "lhs_table_init": (ctypes.c_int, [T, P, i64, i32, i32]),
        "lhs_table_info": (ctypes.c_int, [T, P, P, P, P]),
        "lhs_embed": (ctypes.c_int, [T, P, i64, ctypes.c_float, P, P, P]),
        "lhs_embed_wire": (ctypes.c_int, [T, P, i64, ctypes.c_float, i32, u32, u32, u32, P,
                                          ctypes.c_size_t, P, P]),
        "lhs_embed_wire_response": (ctypes.c_int, [T, P, i64, ctypes.c_float, i32, u32, ctypes.c_float, P,
                                                   sz, P, P]),
        "lhs_unique_ids_workspace": (i64, [i64]),
        "lhs_unique_ids": (ctypes.c_int, [i64, P, i64, P, P, P, P, sz, P, P]),
        "lhs_embed_dedup_workspace": (i64, [T, i64]),
        "lhs_embed_dedup": (ctypes.c_int, [T, P, i64, ctypes.c_float, P, P, sz, P, P]),
        "lhs_embed_mixed": (ctypes.c_int, [P, i64, P, P, i64, i32, P, i64, ctypes.c_float, P, P, P]),
        "lhs_logits_topk_workspace": (ctypes.c_int, [T, i32, i32, i32, P]),
        "lhs_logits_topk_launches": (ctypes.c_int, [T, i32, i32, i32, P]),
        "lhs_logits_topk": (ctypes.c_int, [T, P, i32, i32, i32, ctypes.c_float, P, P, P,
                                           P, sz, P, P]),
        "lhs_logits": (ctypes.c_int, [T, P, i32, i32, P, P, sz, P, P]),
        "lhs_logits_topk_noalloc": (ctypes.c_int, [T, P, i32, i32, i32, ctypes.c_float, P,
                                                   P, P, P, P]),
        "lhs_wire_bytes": (i64, [i32, i32, i32]),
        "lhs_wire_encode": (ctypes.c_int, [i32, P, i32, i32, i32, u32, u32, u32, P, sz,
                                           P, P]),
        "lhs_wire_decode": (ctypes.c_int, [i32, P, sz, i32, i32, P, P, P]),
        "lhs_wire_response_bytes": (i64, [i32, i32, i32]),
        "lhs_wire_encode_response": (ctypes.c_int, [i32, P, i32, i32, i32, u32, ctypes.c_float, P, sz,
                                                    P, P]),
        "lhs_wire_decode_response": (ctypes.c_int, [i32, P, sz, i32, i32, P, P, P]),
        "lhs_selftest_bounded_wait": (ctypes.c_int, [P, i64, P]),
        "lhs_strerror": (ctypes.c_char_p, [ctypes.c_int]),
        "lhs_last_cuda_error": (ctypes.c_int, []),
        "lhs_version": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def _check(rc: int, where: str):
    if rc != LHS_OK:
        raise LhsError(rc, where)


def _dev(t: torch.Tensor, name: str) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _err_word(err, device) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device) if err is None else err


class Table:
    """A device-resident table plus its ``lhs_table`` descriptor.  Keeps the
    tensor alive for as long as the descriptor is used."""

    def __init__(self, tensor: torch.Tensor, vocab: int, hidden: int, dtype: int):
        self.tensor = tensor
        self.c = lhs_table()
        _check(lib().lhs_table_init(ctypes.byref(self.c), _dev(tensor, "table"), vocab,
                                    hidden, dtype), "lhs_table_init")

    @property
    def vocab(self):
        return self.c.vocab

    @property
    def hidden(self):
        return self.c.hidden

    @property
    def dtype(self):
        return self.c.dtype

    @property
    def row_bytes(self):
        return self.c.row_bytes

    @property
    def device(self):
        return self.tensor.device


def lhs_table_init(tensor: torch.Tensor, vocab: int, hidden: int, dtype: int) -> Table:
    return Table(tensor, vocab, hidden, dtype)


def lhs_table_info(table: Table) -> dict:
    v, h, rb, tb = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int64(), ctypes.c_int64()
    _check(lib().lhs_table_info(ctypes.byref(table.c), ctypes.byref(v), ctypes.byref(h),
                                ctypes.byref(rb), ctypes.byref(tb)), "lhs_table_info")
    return {"vocab": v.value, "hidden": h.value, "row_bytes": rb.value,
            "total_bytes": tb.value}


def lhs_embed(table: Table, ids: torch.Tensor, scale: float, out=None, err=None,
              stream=None):
    """Gather rows ``ids`` (int32, CUDA) -> f32 [n, hidden] scaled by ``scale``.
    Returns (out, err word)."""
    n = ids.numel()
    if ids.dtype != torch.int32:
        raise ValueError("ids must be int32")
    if out is None:
        out = torch.empty((n, table.hidden), dtype=torch.float32, device=table.device)
    err = _err_word(err, table.device)
    _check(lib().lhs_embed(ctypes.byref(table.c), _dev(ids, "ids") if n else None, n,
                           float(scale), _dev(out, "out") if n else None,
                           _dev(err, "err"), _stream(stream)), "lhs_embed")
    return out, err


def lhs_embed_wire(table: Table, ids: torch.Tensor, scale: float, fmt: int, layer: int = 0,
                   flags: int = 0, top_k: int = 0, buf=None, err=None, stream=None):
    """Gather rows ``ids`` scaled by ``scale`` straight into a wire message of
    format ``fmt`` (uint8 tensor).  Returns (buf, err word)."""
    n = ids.numel()
    if ids.dtype != torch.int32:
        raise ValueError("ids must be int32")
    nb = lhs_wire_bytes(fmt, n, table.hidden)
    if nb < 0:
        raise ValueError("bad wire format or shape")
    buf = torch.empty(nb, dtype=torch.uint8, device=table.device) if buf is None else buf
    err = _err_word(err, table.device)
    _check(lib().lhs_embed_wire(ctypes.byref(table.c), _dev(ids, "ids") if n else None, n,
                                float(scale), fmt, layer, flags, top_k, _dev(buf, "buf"),
                                buf.numel(), _dev(err, "err"), _stream(stream)), "lhs_embed_wire")
    return buf, err


def lhs_embed_wire_response(table: Table, ids: torch.Tensor, scale: float, fmt: int, layer: int = 0,
                            latency_ms: float = 0.0, buf=None, err=None, stream=None):
    """Gather rows ``ids`` scaled by ``scale`` straight into a single-layer
    response message of format ``fmt``.  Without ``buf`` the message is a
    view 4 bytes into a fresh buffer, so that its payload is 16-byte
    aligned.  Returns (buf, err word)."""
    n = ids.numel()
    if ids.dtype != torch.int32:
        raise ValueError("ids must be int32")
    nb = lhs_wire_response_bytes(fmt, n, table.hidden)
    if nb < 0:
        raise ValueError("bad wire format or shape")
    if buf is None:
        buf = torch.empty(nb + 4, dtype=torch.uint8, device=table.device)[4:]
    err = _err_word(err, table.device)
    _check(lib().lhs_embed_wire_response(ctypes.byref(table.c), _dev(ids, "ids") if n else None, n,
                                         float(scale), fmt, layer, float(latency_ms), _dev(buf, "buf"),
                                         buf.numel(), _dev(err, "err"), _stream(stream)),
           "lhs_embed_wire_response")
    return buf, err


def lhs_unique_ids(ids: torch.Tensor, vocab: int, ws=None, err=None, stream=None, unique=None,
                   inverse=None, count=None):
    """Distinct ids in [0, vocab), ascending, and each position's index into
    them (-1 for a bad id).  Returns (unique, inverse, count tensor, err word);
    unique holds min(n, vocab) entries, the first `count` of them valid."""
    n = ids.numel()
    dev = ids.device
    if ids.dtype != torch.int32:
        raise ValueError("ids must be int32")
    need = lib().lhs_unique_ids_workspace(vocab)
    if need < 0:
        raise ValueError("bad vocab")
    ws = torch.empty(need, dtype=torch.uint8, device=dev) if ws is None else ws
    if unique is None:
        unique = torch.empty(max(1, min(n, vocab)), dtype=torch.int32, device=dev)
    if inverse is None:
        inverse = torch.empty(max(1, n), dtype=torch.int32, device=dev)
    if count is None:
        count = torch.empty(1, dtype=torch.int32, device=dev)
    if unique.numel() < min(n, vocab) or inverse.numel() < n or count.numel() < 1:
        raise ValueError("output tensors too small")
    err = _err_word(err, dev)
    _check(lib().lhs_unique_ids(vocab, _dev(ids, "ids") if n else None, n, _dev(unique, "unique"),
                                _dev(inverse, "inverse"), _dev(count, "count"), _dev(ws, "ws"),
                                ws.numel(), _dev(err, "err"), _stream(stream)), "lhs_unique_ids")
    return unique, inverse[:n], count, err


def lhs_embed_dedup(table: Table, ids: torch.Tensor, scale: float, out=None, ws=None, err=None,
                    stream=None):
    """lhs_embed through the distinct ids (each distinct row decoded once).
    Returns (out, err word)."""
    n = ids.numel()
    if ids.dtype != torch.int32:
        raise ValueError("ids must be int32")
    if out is None:
        out = torch.empty((n, table.hidden), dtype=torch.float32, device=table.device)
    err = _err_word(err, table.device)
    if n == 0:
        return out, err
    need = lib().lhs_embed_dedup_workspace(ctypes.byref(table.c), n)
    ws = torch.empty(need, dtype=torch.uint8, device=table.device) if ws is None else ws
    _check(lib().lhs_embed_dedup(ctypes.byref(table.c), _dev(ids, "ids"), n, float(scale), _dev(out, "out"),
                                 _dev(ws, "ws"), ws.numel(), _dev(err, "err"), _stream(stream)),
           "lhs_embed_dedup")
    return out, err


def lhs_embed_mixed(data: torch.Tensor, row_offset: torch.Tensor, row_dtype: torch.Tensor, vocab: int,
                    hidden: int, ids: torch.Tensor, scale: float, out=None, err=None, stream=None):
    """Gather from a table whose rows carry their own element type (uint8
    data, int64 row offsets, uint8 row types).  Returns (out, err word)."""
    n = ids.numel()
    dev = data.device
    if out is None:
        out = torch.empty((n, hidden), dtype=torch.float32, device=dev)
    err = _err_word(err, dev)
    _check(lib().lhs_embed_mixed(_dev(data, "data"), data.numel() * data.element_size(),
                                 _dev(row_offset, "row_offset"), _dev(row_dtype, "row_dtype"), vocab, hidden,
                                 _dev(ids, "ids") if n else None, n, float(scale),
                                 _dev(out, "out") if n else None, _dev(err, "err"), _stream(stream)),
           "lhs_embed_mixed")
    return out, err


def _resid_dtype(resid: torch.Tensor) -> int:
    if resid.dtype == torch.float32:
        return LHS_F32
    if resid.dtype == torch.bfloat16:
        return LHS_BF16
    raise ValueError("residuals must be float32 or bfloat16")


def lhs_logits_topk_workspace(table: Table, batch: int, k: int, resid_dtype: int) -> int:
    b = ctypes.c_size_t()
    _check(lib().lhs_logits_topk_workspace(ctypes.byref(table.c), batch, k, resid_dtype,
                                           ctypes.byref(b)), "lhs_logits_topk_workspace")
    return b.value


def lhs_logits_topk_launches(table: Table, batch: int, k: int, resid_dtype: int) -> int:
    n = ctypes.c_int32()
    _check(lib().lhs_logits_topk_launches(ctypes.byref(table.c), batch, k, resid_dtype,
                                          ctypes.byref(n)), "lhs_logits_topk_launches")
    return n.value


def lhs_logits_topk(table: Table, resid: torch.Tensor, k: int, temperature: float = 1.0,
                    want_probs: bool = True, ws=None, ids=None, logits=None, probs=None,
                    err=None, stream=None):
    """Top-k of resid @ table.T per residual.  Returns (ids, logits, probs|None,
    err word)."""
    B = resid.shape[0]
    rd = _resid_dtype(resid)
    dev = table.device
    if ws is None:
        ws = torch.empty(lhs_logits_topk_workspace(table, B, k, rd), dtype=torch.uint8,
                         device=dev)
    ids = torch.empty((B, k), dtype=torch.int32, device=dev) if ids is None else ids
    logits = torch.empty((B, k), dtype=torch.float32, device=dev) if logits is None else logits
    if want_probs and probs is None:
        probs = torch.empty((B, k), dtype=torch.float32, device=dev)
    err = _err_word(err, dev)
    _check(lib().lhs_logits_topk(ctypes.byref(table.c), _dev(resid, "resid"), rd, B, k,
                                 float(temperature), _dev(ids, "ids"),
                                 _dev(logits, "logits"),
                                 _dev(probs, "probs") if want_probs else None,
                                 _dev(ws, "ws"), ws.numel() * ws.element_size(),
                                 _dev(err, "err"), _stream(stream)), "lhs_logits_topk")
    return ids, logits, (probs if want_probs else None), err


def lhs_logits(table: Table, resid: torch.Tensor, ws=None, out=None, err=None, stream=None):
    """Raw logits f32 [batch, vocab].  Returns (logits, err word)."""
    B = resid.shape[0]
    rd = _resid_dtype(resid)
    dev = table.device
    if ws is None:
        ws = torch.empty(lhs_logits_topk_workspace(table, B, 0, rd), dtype=torch.uint8,
                         device=dev)
    out = torch.empty((B, table.vocab), dtype=torch.float32, device=dev) if out is None else out
    err = _err_word(err, dev)
    _check(lib().lhs_logits(ctypes.byref(table.c), _dev(resid, "resid"), rd, B,
                            _dev(out, "logits"), _dev(ws, "ws"),
                            ws.numel() * ws.element_size(), _dev(err, "err"),
                            _stream(stream)), "lhs_logits")
    return out, err


def lhs_logits_topk_noalloc(table: Table, resid: torch.Tensor, k: int,
                            temperature: float = 1.0, want_probs: bool = True, ids=None,
                            logits=None, probs=None, err=None, stream=None):
    """lhs_logits_topk with the library's built-in scratch instead of a
    workspace, for callers that cannot allocate device memory on the call
    path.  Returns (ids, logits, probs|None, err word)."""
    B = resid.shape[0]
    dev = table.device
    ids = torch.empty((B, k), dtype=torch.int32, device=dev) if ids is None else ids
    logits = torch.empty((B, k), dtype=torch.float32, device=dev) if logits is None else logits
    if want_probs and probs is None:
        probs = torch.empty((B, k), dtype=torch.float32, device=dev)
    err = _err_word(err, dev)
    _check(lib().lhs_logits_topk_noalloc(ctypes.byref(table.c), _dev(resid, "resid"),
                                         _resid_dtype(resid), B, k, float(temperature),
                                         _dev(ids, "ids"), _dev(logits, "logits"),
                                         _dev(probs, "probs") if want_probs else None,
                                         _dev(err, "err"), _stream(stream)),
           "lhs_logits_topk_noalloc")
    return ids, logits, (probs if want_probs else None), err


def lhs_wire_bytes(fmt: int, seq_len: int, hidden: int) -> int:
    return int(lib().lhs_wire_bytes(fmt, seq_len, hidden))


def lhs_wire_encode(fmt: int, x: torch.Tensor, layer: int = 0, flags: int = 0,
                    top_k: int = 0, buf=None, err=None, stream=None):
    """Encode residuals [seq_len, hidden] (f32 or bf16) into a uint8 message.
    Returns (buf, err word)."""
    s, h = x.shape
    n = lhs_wire_bytes(fmt, s, h)
    if n < 0:
        raise ValueError("bad wire format or shape")
    buf = torch.empty(n, dtype=torch.uint8, device=x.device) if buf is None else buf
    err = _err_word(err, x.device)
    _check(lib().lhs_wire_encode(fmt, _dev(x, "x") if s else None, _resid_dtype(x), s, h,
                                 layer, flags, top_k, _dev(buf, "buf"), buf.numel(),
                                 _dev(err, "err"), _stream(stream)), "lhs_wire_encode")
    return buf, err


def lhs_wire_decode(fmt: int, buf: torch.Tensor, seq_len: int, hidden: int, out=None,
                    err=None, stream=None):
    """Decode a message into f32 [seq_len, hidden].  Returns (x, err word)."""
    if out is None:
        out = torch.empty((seq_len, hidden), dtype=torch.float32, device=buf.device)
    err = _err_word(err, buf.device)
    _check(lib().lhs_wire_decode(fmt, _dev(buf, "buf"), buf.numel(), seq_len, hidden,
                                 _dev(out, "x") if seq_len else None, _dev(err, "err"),
                                 _stream(stream)), "lhs_wire_decode")
    return out, err


def lhs_wire_response_bytes(fmt: int, seq_len: int, hidden: int) -> int:
    return int(lib().lhs_wire_response_bytes(fmt, seq_len, hidden))


def lhs_wire_encode_response(fmt: int, x: torch.Tensor, layer: int = 0, latency_ms: float = 0.0,
                             buf=None, err=None, stream=None):
    """Encode residuals [seq_len, hidden] (f32 or bf16) as a single-layer
    response message ([layer][seq_len][latency_ms] header).  Without ``buf``
    the message is a view 4 bytes into a fresh buffer, so that its payload
    is 16-byte aligned.  Returns (buf, err word)."""
    s, h = x.shape
    n = lhs_wire_response_bytes(fmt, s, h)
    if n < 0:
        raise ValueError("bad wire format or shape")
    if buf is None:
        buf = torch.empty(n + 4, dtype=torch.uint8, device=x.device)[4:]
    err = _err_word(err, x.device)
    _check(lib().lhs_wire_encode_response(fmt, _dev(x, "x") if s else None, _resid_dtype(x), s, h,
                                          layer, float(latency_ms), _dev(buf, "buf"), buf.numel(),
                                          _dev(err, "err"), _stream(stream)), "lhs_wire_encode_response")
    return buf, err


def lhs_wire_decode_response(fmt: int, buf: torch.Tensor, seq_len: int, hidden: int, out=None,
                             err=None, stream=None):
    """Decode a single-layer response message into f32 [seq_len, hidden].
    Returns (x, err word)."""
    if out is None:
        out = torch.empty((seq_len, hidden), dtype=torch.float32, device=buf.device)
    err = _err_word(err, buf.device)
    _check(lib().lhs_wire_decode_response(fmt, _dev(buf, "buf"), buf.numel(), seq_len, hidden,
                                          _dev(out, "x") if seq_len else None, _dev(err, "err"),
                                          _stream(stream)), "lhs_wire_decode_response")
    return out, err


def lhs_selftest_bounded_wait(timeout_ns: int, err=None, device=None, stream=None):
    """Run the never-satisfied bounded wait; returns the err word (TIMEOUT set)."""
    err = _err_word(err, device or torch.device("cuda"))
    _check(lib().lhs_selftest_bounded_wait(_dev(err, "err"), int(timeout_ns),
                                           _stream(stream)), "lhs_selftest_bounded_wait")
    return err


def lhs_version() -> str:
    return lib().lhs_version().decode()
