"""The C-ABI library builds, loads and exports every symbol ``include/lhs.h``
declares; host-side argument checks answer without touching a GPU (CPU only).
"""
import ctypes
import os
import re

import pytest

import embedding_lookup_tied_gb300 as lhs
from embedding_lookup_tied_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    _build.build()
    return lhs.lib()


def _declared():
    with open(os.path.join(ROOT, "include", "lhs.h")) as f:
        text = f.read()
    return re.findall(r"LHS_API\s+[\w\s\*]*?\b(lhs_\w+)\s*\(", text)


def test_header_declares_the_binding_symbols():
    assert tuple(_declared()) == lhs.ABI_SYMBOLS


def test_library_exports_every_declared_symbol(L):
    for name in _declared():
        assert hasattr(L, name), name
        assert ctypes.cast(getattr(L, name), ctypes.c_void_p).value


def test_only_the_abi_is_exported(L):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", lhs.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    text_syms = [l.split()[-1] for l in out.splitlines() if " T " in l]
    assert sorted(text_syms) == sorted(lhs.ABI_SYMBOLS)


def test_version_and_strerror(L):
    assert b"sm_103a" in L.lhs_version()
    for code, msg in ((0, b"ok"), (-1, b"invalid argument"), (-2, b"buffer too small"),
                      (-3, b"unsupported request"), (-4, b"CUDA error"), (7, b"unknown status")):
        assert L.lhs_strerror(code) == msg


def test_wire_bytes_formula(L):
    assert L.lhs_wire_bytes(0, 3, 8) == 16 + 96
    assert L.lhs_wire_bytes(1, 3, 8) == 16 + 48
    assert L.lhs_wire_bytes(2, 3, 8) == 16 + 3 * 16
    assert L.lhs_wire_bytes(2, 256, 5120) == 16 + 256 * 5128
    assert L.lhs_wire_bytes(3, 1, 1) == -1
    assert L.lhs_wire_bytes(0, -1, 8) == -1
    assert L.lhs_wire_bytes(0, 1, 0) == -1


def test_wire_response_bytes_formula(L):
    # the single-layer response: the request's payload after a 12-byte header
    for fmt, s, h in ((0, 3, 8), (1, 3, 8), (2, 3, 8), (2, 256, 5120), (1, 0, 64)):
        assert L.lhs_wire_response_bytes(fmt, s, h) == L.lhs_wire_bytes(fmt, s, h) - 4
    assert L.lhs_wire_response_bytes(2, 3, 8) == 12 + 3 * 16
    assert L.lhs_wire_response_bytes(3, 1, 1) == -1
    assert L.lhs_wire_response_bytes(0, -1, 8) == -1
    assert L.lhs_wire_response_bytes(0, 1, 0) == -1


FAKE = 0x10000  # an aligned address that is never dereferenced by these calls


def test_table_init_and_info_validate(L):
    t = lhs.lhs_table()
    assert L.lhs_table_init(ctypes.byref(t), FAKE, 151936, 896, lhs.LHS_BF16) == 0
    assert t.row_bytes == 1792
    v, h, rb, tb = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int64(), ctypes.c_int64()
    assert L.lhs_table_info(ctypes.byref(t), ctypes.byref(v), ctypes.byref(h),
                            ctypes.byref(rb), ctypes.byref(tb)) == 0
    assert (v.value, h.value, rb.value, tb.value) == (151936, 896, 1792, 151936 * 1792)
    assert L.lhs_table_init(ctypes.byref(t), FAKE, 262144, 768, lhs.LHS_Q8_0) == 0
    assert t.row_bytes == 816
    bad = [(FAKE, 100, 100, lhs.LHS_Q8_0), (FAKE + 8, 10, 16, lhs.LHS_F32),
           (None, 10, 16, lhs.LHS_F32), (FAKE, 0, 16, lhs.LHS_F32),
           (FAKE, 2 ** 31, 16, lhs.LHS_F32), (FAKE, 10, 0, lhs.LHS_F32),
           (FAKE, 10, 16, 7)]
    for args in bad:
        assert L.lhs_table_init(ctypes.byref(t), *args) == lhs.LHS_ERR_INVALID_ARG, args


def test_host_checks_reject_before_any_launch(L):
    t = lhs.lhs_table()
    assert L.lhs_table_init(ctypes.byref(t), FAKE, 1000, 64, lhs.LHS_F16) == 0
    P = FAKE
    # embed: negative n, misaligned output, non-finite scale; n == 0 is a no-op
    assert L.lhs_embed(ctypes.byref(t), P, -1, 1.0, P, P, None) == lhs.LHS_ERR_INVALID_ARG
    assert L.lhs_embed(ctypes.byref(t), P, 4, 1.0, P + 4, P, None) == lhs.LHS_ERR_INVALID_ARG
    assert L.lhs_embed(ctypes.byref(t), P, 4, float("nan"), P, P, None) == lhs.LHS_ERR_INVALID_ARG
    assert L.lhs_embed(ctypes.byref(t), None, 0, 1.0, None, None, None) == lhs.LHS_OK
    # top-k: k out of range, bad temperature, bad residual dtype
    for k, T, rd in ((0, 1.0, 0), (129, 1.0, 0), (1001, 1.0, 0), (5, 0.0, 0),
                     (5, float("inf"), 0), (5, 1.0, lhs.LHS_F16)):
        assert L.lhs_logits_topk(ctypes.byref(t), P, rd, 1, k, T, P, P, None, P, 1 << 20, P,
                                 None) == lhs.LHS_ERR_INVALID_ARG
    assert L.lhs_logits_topk(ctypes.byref(t), P, 0, 0, 5, 1.0, P, P, None, P, 1 << 20, P,
                             None) == lhs.LHS_ERR_INVALID_ARG
    # wire: short buffer, bad dtype, misaligned buffer
    assert L.lhs_wire_encode(1, P, 0, 2, 64, 0, 0, 0, P, 100, P, None) == \
        lhs.LHS_ERR_BUFFER_TOO_SMALL
    assert L.lhs_wire_encode(1, P, 1, 2, 64, 0, 0, 0, P, 1 << 20, P, None) == \
        lhs.LHS_ERR_INVALID_ARG
    assert L.lhs_wire_decode(2, P + 8, 1 << 20, 2, 64, P, P, None) == lhs.LHS_ERR_INVALID_ARG
    assert L.lhs_wire_decode(2, P, 100, 2, 64, P, P, None) == lhs.LHS_ERR_BUFFER_TOO_SMALL
    # response messages: 4-byte alignment is enough for the buffer (a
    # payload 12 bytes in), not less; sizes against the response size
    assert L.lhs_wire_encode_response(1, P, 0, 2, 64, 0, ctypes.c_float(0.5), P + 2, 1 << 20, P,
                                      None) == lhs.LHS_ERR_INVALID_ARG
    assert L.lhs_wire_encode_response(1, P, 0, 2, 64, 0, ctypes.c_float(0.5), P + 4, 12 + 255, P,
                                      None) == lhs.LHS_ERR_BUFFER_TOO_SMALL
    assert L.lhs_wire_encode_response(1, P + 4, 0, 2, 64, 0, ctypes.c_float(0.5), P, 1 << 20, P,
                                      None) == lhs.LHS_ERR_INVALID_ARG
    assert L.lhs_wire_decode_response(2, P + 2, 1 << 20, 2, 64, P, P, None) == lhs.LHS_ERR_INVALID_ARG
    assert L.lhs_wire_decode_response(2, P + 4, 12 + 2 * 72 - 1, 2, 64, P, P, None) == \
        lhs.LHS_ERR_BUFFER_TOO_SMALL
    assert L.lhs_embed_wire_response(ctypes.byref(t), P, 4, ctypes.c_float(1.0), 2, 0, ctypes.c_float(0.0),
                                     P + 2, 1 << 20, P, None) == lhs.LHS_ERR_INVALID_ARG
    assert L.lhs_embed_wire_response(ctypes.byref(t), P, 4, ctypes.c_float(1.0), 2, 0, ctypes.c_float(0.0),
                                     P + 4, 12 + 4 * 72 - 1, P, None) == lhs.LHS_ERR_BUFFER_TOO_SMALL
    assert L.lhs_selftest_bounded_wait(P, -5, None) == lhs.LHS_ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros((2, 8), dtype=torch.float32)
    with pytest.raises(ValueError):
        lhs.lhs_wire_encode(lhs.LHS_WIRE_F16, x)
