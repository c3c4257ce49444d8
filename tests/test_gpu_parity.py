"""GPU parity: the CUDA path through the C-ABI against the oracle.

Bit-exact for the gather, Q8_0 dequant, wire codecs and top-k selection;
lm_head logits within RTOL * sum|T x| of the binary64 oracle; probabilities
within 1e-5 (relative) of the oracle evaluated on the GPU's own logits.
"""
import functools
import math
import struct

import numpy as np
import pytest
import torch

import embedding_lookup_tied_gb300 as lhs
import oracle as orc
import workloads as wl
from gpu_util import (PROB_RTOL, RTOL, canaries_intact, check_topk_against_fp64, guarded,
                      resid_values, same_f32, to_dev, upload_table)

pytestmark = pytest.mark.gpu


# ---------------------------------------------------------------------------
# step 1: gather
# ---------------------------------------------------------------------------

def _embed_case(dtype, V, H, ids, scale, seed=0):
    T = wl.make_table(dtype, V, H, 0.02, cid=100 + seed, threads=4)
    tab = upload_table(T, dtype, V, H)
    ids_d = to_dev(np.asarray(ids, np.int32))
    raw, out, pad = guarded((len(ids), H), torch.float32)
    _, err = lhs.lhs_embed(tab, ids_d, scale, out=out)
    ref, ref_err = orc.embed(T, dtype, V, H, ids, scale)
    got = out.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    assert int(err.item()) == ref_err
    assert canaries_intact(raw, pad)


@pytest.mark.parametrize("dtype,H", [(orc.F32, 256), (orc.F32, 36), (orc.F32, 7),
                                     (orc.F16, 256), (orc.F16, 72), (orc.F16, 13),
                                     (orc.BF16, 896), (orc.BF16, 100),
                                     (orc.Q8_0, 768), (orc.Q8_0, 96), (orc.Q8_0, 32)])
@pytest.mark.parametrize("scaled", [False, True])
def test_embed_parity(dtype, H, scaled):
    V = 1031
    g = np.random.default_rng(H)
    ids = np.concatenate([[0, V - 1, 5, 5], g.integers(0, V, 200), [-1, V, 2 ** 31 - 1, 7]])
    s = np.float32(math.sqrt(H)) if scaled else np.float32(1.0)
    _embed_case(dtype, V, H, ids.astype(np.int32), s, seed=dtype)


@pytest.mark.parametrize("name", ["tiny", "qwen05b", "gemma_q8"])
def test_embed_workloads_full_size(name):
    w = wl.WORKLOADS[name]
    T = wl.table_for(w)
    tab = upload_table(T, w.dtype, w.vocab, w.hidden)
    ids = wl.ids_for(w)
    for s in ([w.embed_scale, np.float32(1.0)] if name == "qwen05b" else [w.embed_scale]):
        out, err = lhs.lhs_embed(tab, to_dev(ids), s)
        ref, ref_err = orc.embed(T, w.dtype, w.vocab, w.hidden, ids, s)
        assert int(err.item()) == ref_err == 0
        assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_embed_empty_and_q8_closed_form():
    V, H = 64, 768
    T = wl.make_table(orc.Q8_0, V, H, cid=7, threads=1)
    tab = upload_table(T, orc.Q8_0, V, H)
    out, err = lhs.lhs_embed(tab, torch.empty(0, dtype=torch.int32, device="cuda"), 1.0)
    assert out.numel() == 0 and int(err.item()) == 0
    # Port Spec forward graph: x = token_embd[ids] * sqrt(768), from the blocks
    ids = np.arange(V, dtype=np.int32)
    s = np.float32(math.sqrt(768.0))
    out, err = lhs.lhs_embed(tab, to_dev(ids), s)
    blk = T.reshape(V, 24, 34)
    d = blk[:, :, 0:2].copy().view(np.float16).astype(np.float64)   # [V,24,1]
    q = blk[:, :, 2:].view(np.int8).astype(np.float64)               # [V,24,32]
    expect = (d * q).reshape(V, H).astype(np.float32) * s
    assert np.array_equal(out.cpu().numpy(), expect)


# ---------------------------------------------------------------------------
# step 4: wire codecs
# ---------------------------------------------------------------------------

def _special(x):
    x = x.copy()
    flat = x.reshape(-1)
    vals = [np.nan, np.inf, -np.inf, 1e6, -65519.99, 65520.0, 65504.0, 3e-8, -0.0, 0.0,
            6.1e-5, 2 ** -25, 1 + 2 ** -11]
    for i, v in enumerate(vals):
        if i * 7 < flat.size:
            flat[i * 7] = v
    return x


@pytest.mark.parametrize("shape", [(4, 256), (1, 896), (8, 5376), (3, 100), (2, 9), (0, 64), (2, 8200),
                                   (40, 1024), (3000, 2048), (1500, 5376), (300, 6144)])
@pytest.mark.parametrize("xdt", [orc.F32, orc.BF16])
@pytest.mark.parametrize("fmt", [orc.WIRE_F32, orc.WIRE_F16, orc.WIRE_I8])
def test_wire_parity(shape, xdt, fmt):
    s, h = shape
    g = np.random.default_rng(s * 1000 + h)
    x = (g.standard_normal(shape).astype(np.float32) *
         g.uniform(0.5, 8, (s, 1)).astype(np.float32))
    if fmt != orc.WIRE_I8:
        x = _special(x)
    elif s >= 3:
        x[1] = 0.0                     # all-zero position
        x[2, min(3, h - 1)] = np.inf   # non-finite position
    if xdt == orc.BF16:
        xs = wl.f32_to_bf16_bits(np.nan_to_num(x, nan=0.0, posinf=3e38, neginf=-3e38))
        xv = orc.bf16_to_f32(xs).reshape(shape)
        xd = to_dev(xs).view(torch.bfloat16).reshape(shape)
    else:
        xv = x
        xd = to_dev(x)
    ref_buf, ref_err = orc.wire_encode(fmt, xv, layer=9, flags=3, top_k=5)
    raw, buf, pad = guarded((ref_buf.size,), torch.uint8)
    _, err = lhs.lhs_wire_encode(fmt, xd, 9, 3, 5, buf=buf)
    got = buf.cpu().numpy()
    assert np.array_equal(got, ref_buf)
    assert int(err.item()) == ref_err
    assert canaries_intact(raw, pad)
    # decode what the GPU encoded
    ref_x, ref_derr = orc.wire_decode(fmt, ref_buf, s, h)
    y, derr = lhs.lhs_wire_decode(fmt, buf, s, h)
    assert same_f32(y.cpu().numpy(), ref_x)
    assert int(derr.item()) == ref_derr == 0


@pytest.mark.parametrize("off", [4, 0], ids=["payload16", "payload12"])
@pytest.mark.parametrize("shape", [(4, 256), (1, 896), (3, 100), (2, 9), (0, 64), (40, 1024),
                                   (300, 2048), (200, 5376)])
@pytest.mark.parametrize("xdt", [orc.F32, orc.BF16])
@pytest.mark.parametrize("fmt", [orc.WIRE_F32, orc.WIRE_F16, orc.WIRE_I8])
def test_wire_response_parity(shape, xdt, fmt, off):
    # single-layer response messages (ADR-0009 Wire Layout): a buffer 4 bytes
    # past a 16-byte boundary puts the payload on one (vector kernels), a
    # 16-byte-aligned buffer leaves it 12 bytes past one (element-wise ones)
    s, h = shape
    g = np.random.default_rng(7 + s * 1000 + h)
    x = (g.standard_normal(shape).astype(np.float32) *
         g.uniform(0.5, 8, (s, 1)).astype(np.float32))
    if fmt != orc.WIRE_I8:
        x = _special(x)
    elif s >= 3:
        x[1] = 0.0
        x[2, min(3, h - 1)] = np.inf
    if xdt == orc.BF16:
        xs = wl.f32_to_bf16_bits(np.nan_to_num(x, nan=0.0, posinf=3e38, neginf=-3e38))
        xv = orc.bf16_to_f32(xs).reshape(shape)
        xd = to_dev(xs).view(torch.bfloat16).reshape(shape)
    else:
        xv = x
        xd = to_dev(x)
    ref_buf, ref_err = orc.wire_encode_response(fmt, xv, layer=9, latency_ms=2.5)
    assert lhs.lhs_wire_response_bytes(fmt, s, h) == ref_buf.size
    pad, n = 256, ref_buf.size
    raw = torch.full((n + 2 * pad + off,), 0x5A, dtype=torch.uint8, device="cuda")
    buf = raw[pad + off:pad + off + n]
    _, err = lhs.lhs_wire_encode_response(fmt, xd, 9, 2.5, buf=buf)
    assert np.array_equal(buf.cpu().numpy(), ref_buf)
    assert int(err.item()) == ref_err
    r = raw.cpu().numpy()
    assert np.all(r[:pad + off] == 0x5A) and np.all(r[pad + off + n:] == 0x5A)
    ref_x, ref_derr = orc.wire_decode_response(fmt, ref_buf, s, h)
    y, derr = lhs.lhs_wire_decode_response(fmt, buf, s, h)
    assert same_f32(y.cpu().numpy(), ref_x)
    assert int(derr.item()) == ref_derr == 0
    if s:
        # a header seq_len other than the caller's: flagged, output untouched
        bad = buf.clone() if off == 0 else torch.empty(n + 4, dtype=torch.uint8, device="cuda")[4:]
        bad.copy_(buf)
        bad[4:8] = torch.from_numpy(np.frombuffer(struct.pack("<I", s + 1), np.uint8).copy()).cuda()
        out = torch.full((s, h), 7.0, dtype=torch.float32, device="cuda")
        _, derr = lhs.lhs_wire_decode_response(fmt, bad, s, h, out=out)
        assert int(derr.item()) == orc.ERR_MALFORMED
        assert bool(torch.all(out == 7.0))


# ---------------------------------------------------------------------------
# steps 1+4 fused: embed straight into a wire message
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,H", [(orc.F32, 256), (orc.F16, 96), (orc.BF16, 64), (orc.Q8_0, 128),
                                     (orc.F32, 36), (orc.BF16, 7), (orc.F16, 5376), (orc.Q8_0, 6656)])
@pytest.mark.parametrize("fmt", [orc.WIRE_F32, orc.WIRE_F16, orc.WIRE_I8])
def test_embed_wire_matches_embed_then_encode(dtype, H, fmt):
    V = 700
    T = wl.make_table(dtype, V, H, 0.02, cid=600 + H, threads=4)
    ids = np.concatenate([[0, V - 1, -1, V, 5, 5],
                          wl.zipf_ids(600 + H, 37, V)]).astype(np.int32)
    scale = float(np.float32(np.sqrt(np.float64(H))))
    tab = upload_table(T, dtype, V, H)
    x_ref, e_ref = orc.embed(T, dtype, V, H, ids, scale)
    ref_buf, e2 = orc.wire_encode(fmt, x_ref, layer=7, flags=2, top_k=9)
    raw, buf, pad = guarded((ref_buf.size,), torch.uint8)
    _, err = lhs.lhs_embed_wire(tab, to_dev(ids), scale, fmt, 7, 2, 9, buf=buf)
    assert np.array_equal(buf.cpu().numpy(), ref_buf)
    assert int(err.item()) == (e_ref | e2)
    assert canaries_intact(raw, pad)


@pytest.mark.parametrize("off", [4, 0], ids=["payload16", "payload12"])
@pytest.mark.parametrize("dtype,H", [(orc.F32, 256), (orc.F16, 96), (orc.BF16, 64), (orc.Q8_0, 128),
                                     (orc.Q8_0, 768), (orc.BF16, 7), (orc.F16, 5376)])
@pytest.mark.parametrize("fmt", [orc.WIRE_F32, orc.WIRE_F16, orc.WIRE_I8])
def test_embed_wire_response_matches_embed_then_encode(dtype, H, fmt, off):
    # the embed reply as a single-layer response message (ADR-0009 Wire
    # Layout), byte for byte the oracle's encode of the oracle's rows
    V = 700
    T = wl.make_table(dtype, V, H, 0.02, cid=650 + H, threads=4)
    ids = np.concatenate([[0, V - 1, -1, V, 5, 5],
                          wl.zipf_ids(650 + H, 37, V)]).astype(np.int32)
    scale = float(np.float32(np.sqrt(np.float64(H))))
    tab = upload_table(T, dtype, V, H)
    x_ref, e_ref = orc.embed(T, dtype, V, H, ids, scale)
    ref_buf, e2 = orc.wire_encode_response(fmt, x_ref, layer=7, latency_ms=0.1)
    assert lhs.lhs_wire_response_bytes(fmt, len(ids), H) == ref_buf.size
    pad, n = 256, ref_buf.size
    raw = torch.full((n + 2 * pad + off,), 0x5A, dtype=torch.uint8, device="cuda")
    buf = raw[pad + off:pad + off + n]
    _, err = lhs.lhs_embed_wire_response(tab, to_dev(ids), scale, fmt, 7, 0.1, buf=buf)
    assert np.array_equal(buf.cpu().numpy(), ref_buf)
    assert int(err.item()) == (e_ref | e2)
    r = raw.cpu().numpy()
    assert np.all(r[:pad + off] == 0x5A) and np.all(r[pad + off + n:] == 0x5A)


def test_embed_wire_empty_and_nonfinite_rows():
    V, H = 64, 64
    T = wl.make_table(orc.F16, V, H, 0.02, cid=610, threads=1)
    T[3, 5] = 0x7C00                       # +inf in row 3
    T[4, :] = 0x7BFF                       # 65504 everywhere in row 4: f16 stays finite
    tab = upload_table(T, orc.F16, V, H)
    for fmt in (orc.WIRE_F32, orc.WIRE_F16, orc.WIRE_I8):
        buf, err = lhs.lhs_embed_wire(tab, torch.empty(0, dtype=torch.int32, device="cuda"), 1.0, fmt,
                                      1, 2, 3)
        ref, _ = orc.wire_encode(fmt, np.zeros((0, H), np.float32), layer=1, flags=2, top_k=3)
        assert np.array_equal(buf.cpu().numpy(), ref) and int(err.item()) == 0
        ids = np.array([3, 4, 1], np.int32)
        x_ref, e_ref = orc.embed(T, orc.F16, V, H, ids, 2.0)    # row 4 x 2 overflows f16 on the wire
        ref, e2 = orc.wire_encode(fmt, x_ref)
        buf, err = lhs.lhs_embed_wire(tab, to_dev(ids), 2.0, fmt)
        assert np.array_equal(buf.cpu().numpy(), ref)
        assert int(err.item()) == (e_ref | e2)


@pytest.mark.parametrize("H", [128, 768, 832])
def test_embed_wire_q8_nonfinite_scales_and_odd_counts(H):
    # Q8_0 rows whose block scale d is inf or NaN, values that overflow
    # under a large scale, bad ids, and an odd number of tokens (the i8 path
    # quantises two tokens per warp)
    V = 300
    T = wl.make_table(orc.Q8_0, V, H, cid=620 + H, threads=1)
    rb = H // 32 * 34
    T = T.reshape(V, rb).copy()
    T[3, 34 * 1:34 * 1 + 2] = np.frombuffer(np.uint16(0x7C00).tobytes(), np.uint8)   # d = +inf
    T[5, 34 * 2:34 * 2 + 2] = np.frombuffer(np.uint16(0x7E00).tobytes(), np.uint8)   # d = NaN
    T[7, 34 * 0:34 * 0 + 2] = np.frombuffer(np.uint16(0x7BFF).tobytes(), np.uint8)   # d = 65504
    tab = upload_table(T, orc.Q8_0, V, H)
    ids = np.concatenate([[3, 5, 7, -2, V + 1, 0], wl.zipf_ids(630 + H, 31, V)]).astype(np.int32)
    assert len(ids) % 2 == 1
    for scale in (float(np.float32(np.sqrt(np.float64(H)))), 3e33):
        x_ref, e_ref = orc.embed(T, orc.Q8_0, V, H, ids, scale)
        ref_buf, e2 = orc.wire_encode(orc.WIRE_I8, x_ref, layer=1, flags=0, top_k=0)
        buf, err = lhs.lhs_embed_wire(tab, to_dev(ids), scale, orc.WIRE_I8, 1, 0, 0)
        assert np.array_equal(buf.cpu().numpy(), ref_buf), scale
        assert int(err.item()) == (e_ref | e2), scale


def test_embed_wire_full_size_gemma_q8():
    w = wl.WORKLOADS["gemma_q8"]
    T = wl.table_for(w)
    tab = upload_table(T, w.dtype, w.vocab, w.hidden)
    ids = wl.ids_for(w)
    x_ref, _ = orc.embed(T, w.dtype, w.vocab, w.hidden, ids, float(w.embed_scale))
    for fmt in (orc.WIRE_F16, orc.WIRE_I8):
        ref, e2 = orc.wire_encode(fmt, x_ref, layer=0, flags=0, top_k=0)
        buf, err = lhs.lhs_embed_wire(tab, to_dev(ids), float(w.embed_scale), fmt)
        assert np.array_equal(buf.cpu().numpy(), ref)
        assert int(err.item()) == e2


@pytest.mark.parametrize("H", [1024, 2048])   # one warp per position; rows staged per CTA
@pytest.mark.parametrize("xdt", [orc.F32, orc.BF16])
def test_i8_codes_at_rounding_boundaries(xdt, H):
    # quotients x / scale at, just below and just above every half-integer:
    # the encoder's product-with-reciprocal shortcut must fall back to the
    # correctly rounded divide exactly where rounding could differ
    rows = []
    for m in (1.0, 3.0, 1e-3, 7.5e-39):      # last: a subnormal scale
        scale = np.float32(np.float32(m) / np.float32(127.0))
        k = np.arange(-127, 127, dtype=np.float32)
        base = ((k + np.float32(0.5)) * scale).astype(np.float32)
        vals = np.concatenate([base, np.nextafter(base, np.float32(np.inf)),
                               np.nextafter(base, np.float32(-np.inf)), [np.float32(m)]])
        row = np.zeros(H, np.float32)
        row[:vals.size] = vals[:H]
        row[H - 1] = np.float32(m)
        rows.append(row)
    x = np.stack(rows)
    if xdt == orc.BF16:
        xs = wl.f32_to_bf16_bits(x)
        xv = orc.bf16_to_f32(xs).reshape(x.shape)
        xd = to_dev(xs).view(torch.bfloat16).reshape(x.shape)
    else:
        xv, xd = x, to_dev(x)
    ref, ref_err = orc.wire_encode(orc.WIRE_I8, xv)
    buf, err = lhs.lhs_wire_encode(orc.WIRE_I8, xd)
    assert np.array_equal(buf.cpu().numpy(), ref)
    assert int(err.item()) == ref_err


@pytest.mark.parametrize("H", [896, 4096])
def test_i8_nonfinite_rows_many_positions(H):
    # inf / NaN rows among 700 positions: those get scale 0 and zero codes
    # and raise the flag; the rows around them are unaffected
    g = np.random.default_rng(H)
    x = (g.standard_normal((700, H)) * g.uniform(0.1, 9.0, (700, 1))).astype(np.float32)
    x[3, 7] = np.inf
    x[400, H - 1] = np.nan
    x[699, 0] = -np.inf
    ref, ref_err = orc.wire_encode(orc.WIRE_I8, x)
    buf, err = lhs.lhs_wire_encode(orc.WIRE_I8, to_dev(x))
    assert np.array_equal(buf.cpu().numpy(), ref)
    assert int(err.item()) == ref_err == lhs.LHS_ERRBIT_NONFINITE


def _decided_topk(L64, dev, k):
    """fp64 top-k ids per residual, and whether a GPU whose logits lie
    within dev[b] of L64[b] (every vocab row) must return the same ordered
    top-k: every gap between consecutive values among the k+1 largest
    exceeds 2 dev[b]."""
    ids = np.empty((L64.shape[0], k), np.int32)
    decided = np.empty(L64.shape[0], bool)
    for b in range(L64.shape[0]):
        i, v = orc.topk_f64(L64[b], k + 1)
        ids[b] = i[:k]
        decided[b] = bool(np.all(v[:-1] - v[1:] > 2.0 * dev[b]))
    return ids, decided


# ADR-0009 Validation: top-5 agreement of logits from f16-decoded residuals
# with the originals, top-1 for i8.  The shapes of the 31B decode and of the
# batched workload (hidden, table type, residual distribution) on 16,384
# vocab rows, so that the oracle's binary64 logits of every residual finish
# in seconds.
WIRE_ACC_CASES = [("gemma31b", 64, 710), ("batched", 128, 720)]


@pytest.mark.parametrize("name,B,cid", WIRE_ACC_CASES, ids=[c[0] for c in WIRE_ACC_CASES])
def test_wire_accuracy_topk_agreement_matches_oracle(name, B, cid):
    import os

    import bench
    w = wl.WORKLOADS[name]
    V, H = 16384, w.hidden
    T = wl.make_table(w.dtype, V, H, 0.02, cid=cid, threads=8)
    tab = upload_table(T, w.dtype, V, H)
    R = wl.residuals(cid + 1, B, H, w.resid_scale_range, w.resid_dtype)
    xv = np.ascontiguousarray(resid_values(R, w.resid_dtype))   # the residual values, f32
    x = to_dev(xv)
    rtol = RTOL[w.dtype]
    threads = os.cpu_count() or 1
    L64, S64 = orc.logits(T, w.dtype, V, H, xv, threads=threads, with_sumabs=True)
    raw, e = lhs.lhs_logits(tab, x)
    assert int(e.item()) == 0
    dev_x = np.abs(raw.cpu().numpy().astype(np.float64) - L64)
    assert np.all(dev_x <= rtol * S64 + 1e-30)
    for fmt, k in ((orc.WIRE_F16, 5), (orc.WIRE_I8, 1)):
        # oracle: its own codec round trip, binary64 logits of both
        buf, e = orc.wire_encode(fmt, xv)
        assert e == 0
        xh, e = orc.wire_decode(fmt, buf, B, H)
        assert e == 0
        Lh64, Sh64 = orc.logits(T, w.dtype, V, H, xh, threads=threads, with_sumabs=True)
        # the GPU's logits of the same decoded residuals (its codec is
        # byte-exact against the oracle's, checked here too)
        gbuf, e1 = lhs.lhs_wire_encode(fmt, x)
        gxh, e2 = lhs.lhs_wire_decode(fmt, gbuf, B, H)
        assert int(e1.item()) == 0 and int(e2.item()) == 0
        assert np.array_equal(gxh.cpu().numpy().view(np.uint32), xh.view(np.uint32))
        rawh, e = lhs.lhs_logits(tab, gxh)
        assert int(e.item()) == 0
        dev_h = np.abs(rawh.cpu().numpy().astype(np.float64) - Lh64)
        assert np.all(dev_h <= rtol * Sh64 + 1e-30)
        ref_ids, dec_ref = _decided_topk(L64, dev_x.max(axis=1), k)
        got_ids, dec_got = _decided_topk(Lh64, dev_h.max(axis=1), k)
        oracle_agree = np.all(ref_ids == got_ids, axis=1)
        decided = dec_ref & dec_got
        # the GPU's verdict (its fused top-k of x and of the decoded x)
        gpu_agree, _ = bench.wire_agreement(lhs, tab, x, k, fmt)
        # where the GPU's logit error cannot reorder the binary64 top-k, the
        # verdicts must be equal
        assert decided.mean() >= 0.95, (fmt, decided.mean())
        bad = np.flatnonzero(gpu_agree[decided] != oracle_agree[decided])
        assert bad.size == 0, (fmt, bad)
        # the page expects identical top-5 for f16 and top-1 for i8; on
        # Gaussian tables (top logits closer together than a trained
        # model's) the oracle's own verdicts bound what the codecs keep
        if fmt == orc.WIRE_F16:
            assert oracle_agree.mean() >= 0.95
        else:
            assert oracle_agree.mean() >= 0.85


def test_wire_decode_malformed():
    x = np.ones((3, 64), np.float32)
    for fmt in (orc.WIRE_F32, orc.WIRE_F16, orc.WIRE_I8):
        buf, _ = lhs.lhs_wire_encode(fmt, to_dev(x))
        out = torch.full((2, 64), 7.0, device="cuda")
        _, err = lhs.lhs_wire_decode(fmt, buf, 2, 64, out=out)   # header says 3
        assert int(err.item()) == lhs.LHS_ERRBIT_MALFORMED
        assert torch.all(out == 7.0)
    buf, _ = lhs.lhs_wire_encode(orc.WIRE_I8, to_dev(x))
    bad = buf.cpu().numpy().copy()
    bad[16 + 72 + 4:16 + 72 + 8] = np.frombuffer(np.float32(0.5).tobytes(), np.uint8)
    out = torch.full((3, 64), 7.0, device="cuda")
    _, err = lhs.lhs_wire_decode(orc.WIRE_I8, to_dev(bad), 3, 64, out=out)
    ref, ref_err = orc.wire_decode(orc.WIRE_I8, bad, 3, 64, out=np.full((3, 64), 7.0, np.float32))
    assert int(err.item()) == ref_err == lhs.LHS_ERRBIT_MALFORMED
    assert np.array_equal(out.cpu().numpy(), ref)


# ---------------------------------------------------------------------------
# steps 2+3: lm_head + top-k
# ---------------------------------------------------------------------------

LM_CASES = [
    # dtype, V, H, B, k, resid dtype        (tensor-core path unless noted)
    (orc.F16, 1000, 256, 3, 5, orc.F32),
    (orc.BF16, 8191, 96, 8, 40, orc.F32),     # ragged vocab, hidden % 64 != 0
    (orc.BF16, 1500, 64, 11, 7, orc.BF16),    # two batch passes, bf16 residuals
    (orc.F16, 300, 128, 1, 128, orc.F32),     # k = kMax
    (orc.BF16, 5000, 128, 2, 128, orc.F32),   # k = kMax over every SM: lists deeper than staged
    (orc.BF16, 20000, 64, 8, 50, orc.F32),    # one full pass, 8 residuals
    (orc.F16, 20000, 64, 12, 50, orc.F32),    # two passes
    (orc.F16, 3000, 2048, 3, 10, orc.F32),    # 3 residuals: only their rows (+ a zero row) resident
    (orc.F16, 3000, 2048, 4, 10, orc.F32),    # 16 operand rows too large to keep resident: prep + TMA tiles
    (orc.BF16, 2000, 1504, 2, 7, orc.BF16),   # compact resident operand, hidden % 64 != 0
    (orc.BF16, 2000, 1272, 5, 7, orc.BF16),   # largest 16-row resident operand, hidden % 64 != 0
    (orc.BF16, 128, 64, 2, 1, orc.F32),       # one block, k = 1
    (orc.F32, 1000, 256, 4, 5, orc.F32),      # bulk-stream CUDA-core path (1 KB rows)
    (orc.Q8_0, 700, 128, 2, 10, orc.F32),     # CUDA-core path (136-byte rows)
    (orc.Q8_0, 5000, 768, 3, 10, orc.F32),    # Q8_0 tensor-core path, 816-byte rows, ragged last block
    (orc.Q8_0, 2100, 256, 11, 7, orc.BF16),   # Q8_0 tensor-core path: passes of 8 and 3 (two and
                                              # one column groups), bf16 residuals
    (orc.Q8_0, 40000, 512, 8, 50, orc.F32),   # Q8_0 tensor-core path, several blocks on every SM
    (orc.Q8_0, 3001, 2560, 5, 16, orc.F32),   # Q8_0 tensor-core path, 10 stages per block, ragged
    (orc.Q8_0, 100, 256, 3, 20, orc.F32),     # vocab < 128 -> CUDA-core path
    (orc.F32, 3001, 64, 8, 64, orc.F32),      # bulk-stream path, 256-byte rows, ragged vocab
    (orc.F32, 900, 36, 2, 5, orc.F32),        # hidden % 8 != 0: CUDA-core path
    (orc.F16, 1000, 72, 2, 6, orc.F32),       # hidden % 64 != 0, tensor-core path
    (orc.F16, 1000, 68, 2, 6, orc.F32),       # hidden % 8 != 0 -> CUDA-core path
    (orc.BF16, 100, 64, 3, 100, orc.F32),     # vocab < 128 -> CUDA-core path, k = V
    (orc.BF16, 100000, 64, 8, 50, orc.F32),   # several 128-row blocks on every SM
    (orc.F16, 90001, 128, 3, 10, orc.BF16),   # the same with a ragged last block, bf16 residuals
]


def _lm_inputs(dtype, V, H, B, rdt, seed):
    T = wl.make_table(dtype, V, H, 0.02, cid=200 + seed, threads=4)
    R = wl.residuals(300 + seed, B, H, (0.5, 8.0), rdt)
    return T, R


def _resid_dev(R, rdt):
    d = to_dev(R)
    return d.view(torch.bfloat16) if rdt == orc.BF16 else d


@pytest.mark.parametrize("case", LM_CASES,
                         ids=[f"{wl.DTYPE_NAMES[c[0]]}-V{c[1]}-H{c[2]}-B{c[3]}-k{c[4]}"
                              for c in LM_CASES])
def test_lm_head_parity(case):
    dtype, V, H, B, k, rdt = case
    T, R = _lm_inputs(dtype, V, H, B, rdt, seed=LM_CASES.index(case))
    tab = upload_table(T, dtype, V, H)
    rd = _resid_dev(R, rdt)
    xv = resid_values(R, rdt)
    L64, S64 = orc.logits(T, dtype, V, H, xv, threads=8, with_sumabs=True)
    rtol = RTOL[dtype]
    # raw logits: within the dot-product tolerance of binary64
    raw, err = lhs.lhs_logits(tab, rd)
    assert int(err.item()) == 0
    Lg = raw.cpu().numpy()
    assert np.all(np.abs(Lg.astype(np.float64) - L64) <= rtol * S64 + 1e-30)
    # fused top-k: bit-exact against the oracle's top-k of the GPU's own logits
    raw_ids, out_ids, pad_i = guarded((B, k), torch.int32)
    raw_v, out_v, pad_v = guarded((B, k), torch.float32)
    ids, vals, probs, err = lhs.lhs_logits_topk(tab, rd, k, temperature=0.7, ids=out_ids,
                                                logits=out_v)
    assert int(err.item()) == 0
    assert canaries_intact(raw_ids, pad_i) and canaries_intact(raw_v, pad_v)
    ids, vals, probs = ids.cpu().numpy(), vals.cpu().numpy(), probs.cpu().numpy()
    for b in range(B):
        rid, rv = orc.topk_f32(Lg[b], k)
        assert np.array_equal(ids[b], rid), b
        assert np.array_equal(vals[b].view(np.uint32), rv.view(np.uint32)), b
        rp = orc.softmax_probs(Lg[b], 0.7, rid)
        assert np.all(np.abs(probs[b] - rp) <= PROB_RTOL * rp), b
        check_topk_against_fp64(ids[b], vals[b], L64[b], S64[b], k, rtol)


def test_q8_lm_head_residual_range():
    # The Q8_0 tensor-core path scales each residual by a power of two and
    # splits it into two levels of f16 halves: residuals far outside the f16
    # range, deep in the f32 subnormals, or with values 2^33 apart stay within
    # the f32-table tolerance -- also on rows whose code at the outlier is 0,
    # where the logit comes from the small values alone.
    V, H, k = 3000, 768, 12
    T = wl.make_table(orc.Q8_0, V, H, 0.02, cid=290, threads=4)
    tab = upload_table(T, orc.Q8_0, V, H)
    code17 = T.view(np.uint8).reshape(V, -1)[:, 2 + 17].view(np.int8)
    assert np.count_nonzero(code17 == 0) >= 3
    base = wl.residuals(291, 6, H)
    X = np.empty_like(base)
    X[0] = base[0] * np.float32(1e-30)
    X[1] = base[1] * np.float32(1e30)
    X[2] = base[2]
    X[2, 17] = np.float32(1e10)            # one value 2^33 above the rest
    X[3] = base[3] * np.float32(1e-41)     # f32 subnormals
    X[4] = 0.0
    X[5] = base[5] * np.float32(70000.0)   # beyond the f16 range
    L64, S64 = orc.logits(T, orc.Q8_0, V, H, X, threads=8, with_sumabs=True)
    raw, err = lhs.lhs_logits(tab, to_dev(X))
    assert int(err.item()) == 0
    Lg = raw.cpu().numpy()
    assert np.all(np.isfinite(Lg))
    assert np.all(np.abs(Lg.astype(np.float64) - L64) <= RTOL[orc.Q8_0] * S64 + 1e-300)
    assert np.all(Lg[4] == 0.0)
    ids, vals, _, err = lhs.lhs_logits_topk(tab, to_dev(X), k)
    assert int(err.item()) == 0
    for b in range(X.shape[0]):
        rid, rv = orc.topk_f32(Lg[b], k)
        assert np.array_equal(ids.cpu().numpy()[b], rid), b
        assert np.array_equal(vals.cpu().numpy()[b].view(np.uint32), rv.view(np.uint32)), b


def test_q8_lm_head_nonfinite_residuals():
    # inf / NaN residual values: every logit is what binary64 gives (+-inf, or
    # NaN where an inf meets a zero code or inf meets -inf)
    V, H = 1000, 256
    T = wl.make_table(orc.Q8_0, V, H, 0.02, cid=292, threads=4)
    tab = upload_table(T, orc.Q8_0, V, H)
    X = wl.residuals(293, 3, H)
    X[0, 5] = np.inf
    X[1, 7] = np.nan
    X[2, 3] = -np.inf
    X[2, 200] = np.inf
    L64 = orc.logits(T, orc.Q8_0, V, H, X, threads=8)
    raw, err = lhs.lhs_logits(tab, to_dev(X))
    assert int(err.item()) == 0
    Lg = raw.cpu().numpy().astype(np.float64)
    assert np.array_equal(np.isnan(Lg), np.isnan(L64))
    fin = ~np.isnan(L64)
    assert np.array_equal(Lg[fin], L64[fin])   # +-inf on both sides
    assert np.isnan(L64[1]).all() and (~np.isnan(L64[0])).any()


@pytest.mark.parametrize("lm_dtype", [orc.BF16, orc.Q8_0, orc.F32])
def test_untied_lm_head_on_embedded_rows(lm_dtype):
    # untied: rows gathered from one table, projected on another
    V, H, k = 3000, 128, 8
    E = wl.make_table(orc.F16, V, H, 0.02, cid=280, threads=4)
    T = wl.make_table(lm_dtype, V, H, 0.02, cid=281, threads=4)
    et, lt = upload_table(E, orc.F16, V, H), upload_table(T, lm_dtype, V, H)
    ids = wl.zipf_ids(282, 5, V)
    x, err = lhs.lhs_embed(et, to_dev(ids), 11.0)
    assert int(err.item()) == 0
    xv, _ = orc.embed(E, orc.F16, V, H, ids, 11.0)
    assert same_f32(x.cpu().numpy(), xv)
    L64, S64 = orc.logits(T, lm_dtype, V, H, xv, threads=8, with_sumabs=True)
    top, vals, _, err = lhs.lhs_logits_topk(lt, x, k)
    assert int(err.item()) == 0
    raw, _ = lhs.lhs_logits(lt, x)
    Lg = raw.cpu().numpy()
    assert np.all(np.abs(Lg.astype(np.float64) - L64) <= RTOL[lm_dtype] * S64 + 1e-30)
    for b in range(len(ids)):
        rid, rv = orc.topk_f32(Lg[b], k)
        assert np.array_equal(top.cpu().numpy()[b], rid)


def test_launch_count_follows_the_plan():
    V = 5000
    T = wl.make_table(orc.BF16, V, 128, 0.02, cid=250, threads=4)
    tab = upload_table(T, orc.BF16, V, 128)
    n = functools.partial(lhs.lhs_logits_topk_launches, tab)
    # hidden 128: the residual operand stays in shared memory, one launch per pass
    assert n(1, 10, lhs.LHS_F32) == 2                      # GEMV + merge
    assert n(8, 128, lhs.LHS_BF16) == 2
    assert n(9, 10, lhs.LHS_F32) == 3                      # two passes + merge
    assert n(3, 0, lhs.LHS_F32) == 1                       # raw logits: no merge
    # hidden 4096: up to 3 residuals keep only their rows resident; from 4 on
    # the operand tiles are streamed by TMA after a prep kernel
    T4 = wl.make_table(orc.F16, 512, 4096, 0.02, cid=252, threads=4)
    tab4 = upload_table(T4, orc.F16, 512, 4096)
    assert lhs.lhs_logits_topk_launches(tab4, 1, 10, lhs.LHS_F32) == 2
    assert lhs.lhs_logits_topk_launches(tab4, 4, 10, lhs.LHS_F32) == 3
    assert n(64, 10, lhs.LHS_BF16) in (2, 3)               # (counter reset +) GEMM + merge
    assert n(64, 0, lhs.LHS_BF16) == 1
    Tq = wl.make_table(orc.Q8_0, 1000, 512, 0.02, cid=253, threads=4)
    tabq = upload_table(Tq, orc.Q8_0, 1000, 512)
    assert lhs.lhs_logits_topk_launches(tabq, 1, 10, lhs.LHS_F32) == 2    # Q8_0 GEMV + merge
    assert lhs.lhs_logits_topk_launches(tabq, 12, 10, lhs.LHS_BF16) == 3  # two passes + merge
    T32 = wl.make_table(orc.F32, 1000, 64, 0.02, cid=251, threads=4)
    tab32 = upload_table(T32, orc.F32, 1000, 64)
    assert lhs.lhs_logits_topk_launches(tab32, 4, 5, lhs.LHS_F32) == 2   # GEMV + merge


def test_repeated_calls_share_a_workspace():
    # consecutive calls on one workspace, alternating between two tables:
    # nothing a call leaves in the workspace may leak into the next
    V, H, k = 6000, 128, 10
    tabs, Xs = [], []
    for i, (dt, v) in enumerate(((orc.BF16, V), (orc.F16, V // 2 + 37))):
        T = wl.make_table(dt, v, H, 0.02, cid=270 + i, threads=4)
        tabs.append(upload_table(T, dt, v, H))
    X = to_dev(wl.residuals(272, 3, H))
    ws = torch.empty(max(lhs.lhs_logits_topk_workspace(t, 3, k, lhs.LHS_F32) for t in tabs),
                     dtype=torch.uint8, device="cuda")
    ref = [lhs.lhs_logits_topk(t, X, k)[0].cpu().numpy() for t in tabs]
    for rep in range(5):
        for t, r in zip(tabs, ref):
            ids, _, _, err = lhs.lhs_logits_topk(t, X, k, ws=ws)
            assert int(err.item()) == 0
            assert np.array_equal(ids.cpu().numpy(), r), rep


@pytest.mark.parametrize("fill", [0x00, 0xA5, 0xFF])
def test_calls_on_a_dirty_workspace(fill):
    # the caller's workspace holds arbitrary bytes on entry: any fill, and
    # the previous calls' leftovers, give the same result as a fresh call,
    # raw logits included
    V, H, B, k = 98000, 96, 2, 16
    T = wl.make_table(orc.BF16, V, H, 0.02, cid=291, threads=4)
    tab = upload_table(T, orc.BF16, V, H)
    X = to_dev(wl.residuals(292, B, H))
    need = max(lhs.lhs_logits_topk_workspace(tab, B, k, lhs.LHS_F32),
               lhs.lhs_logits_topk_workspace(tab, B, 0, lhs.LHS_F32))
    ws = torch.full((need,), fill, dtype=torch.uint8, device="cuda")
    raw, err = lhs.lhs_logits(tab, X, ws=ws)
    assert int(err.item()) == 0
    Lg = raw.cpu().numpy()
    L64, S64 = orc.logits(T, orc.BF16, V, H, wl.residuals(292, B, H), threads=8, with_sumabs=True)
    assert np.all(np.abs(Lg.astype(np.float64) - L64) <= RTOL[orc.BF16] * S64 + 1e-30)
    for rep in range(4):
        ids, vals, _, err = lhs.lhs_logits_topk(tab, X, k, ws=ws)
        assert int(err.item()) == 0
        for b in range(B):
            rid, rv = orc.topk_f32(Lg[b], k)
            assert np.array_equal(ids.cpu().numpy()[b], rid), (rep, b)
            assert np.array_equal(vals.cpu().numpy()[b].view(np.uint32), rv.view(np.uint32)), (rep, b)
        raw2, err = lhs.lhs_logits(tab, X, ws=ws)
        assert int(err.item()) == 0
        assert np.array_equal(raw2.cpu().numpy().view(np.uint32), Lg.view(np.uint32)), rep


@pytest.mark.parametrize("fill", [0x00, 0xA5, 0xFF])
def test_batched_gemm_on_a_dirty_workspace(fill):
    # the one-pass GEMM keeps arrival counters, the sample and the bounds in
    # the workspace: whatever it holds on entry (counters already past their
    # targets, stale samples), every call gives the top-k of its own logits
    V, H, B, k = 40000, 128, 20, 12   # two tiles per CTA pair or more: sampled bound
    T = wl.make_table(orc.BF16, V, H, 0.02, cid=293, threads=4)
    tab = upload_table(T, orc.BF16, V, H)
    R = wl.residuals(294, B, H, (0.5, 8.0), orc.BF16)
    rd = _resid_dev(R, orc.BF16)
    need = lhs.lhs_logits_topk_workspace(tab, B, k, lhs.LHS_BF16)
    ws = torch.full((need,), fill, dtype=torch.uint8, device="cuda")
    raw, err = lhs.lhs_logits(tab, rd)
    assert int(err.item()) == 0
    Lg = raw.cpu().numpy()
    for rep in range(3):
        ids, vals, _, err = lhs.lhs_logits_topk(tab, rd, k, ws=ws)
        assert int(err.item()) == 0
        ids, vals = ids.cpu().numpy(), vals.cpu().numpy()
        for b in range(B):
            rid, rv = orc.topk_f32(Lg[b], k)
            assert np.array_equal(ids[b], rid), (rep, b)
            assert np.array_equal(vals[b].view(np.uint32), rv.view(np.uint32)), (rep, b)


GEMM_CASES = [
    # bf16 table, bf16 residuals, batch > 8: tcgen05 GEMM path
    # V, H, B, k
    (5000, 512, 37, 20),      # ragged last vocab tile; second CTA of each pair idle
    (1000, 96, 200, 64),      # hidden % 64 != 0; three stages
    (700, 64, 256, 128),      # k = 128, two stages; both residual halves
    (3000, 256, 130, 5),      # one residual in the second half
    (40000, 128, 150, 20),    # >= 2 tiles per cluster: first-tile sample and its bounds
    (39000, 64, 256, 128),    # sample with k = 128 (256-entry buffers)
    (5000, 64, 300, 10),      # beyond one cluster's 256 residuals: two passes
    (40000, 64, 513, 50),     # three passes, each with its sample
    (40000, 64, 9, 1),        # smallest batch on the GEMM, k = 1, sampled bound
    (45000, 256, 129, 3),     # one residual in the second CTA of each pair, sampled bound
]


@pytest.mark.parametrize("case", GEMM_CASES, ids=[f"V{c[0]}-H{c[1]}-B{c[2]}-k{c[3]}"
                                                  for c in GEMM_CASES])
def test_gemm_lm_head_parity(case):
    V, H, B, k = case
    T = wl.make_table(orc.BF16, V, H, 0.02, cid=400 + V, threads=4)
    R = wl.residuals(500 + B, B, H, (0.5, 8.0), orc.BF16)
    tab = upload_table(T, orc.BF16, V, H)
    rd = _resid_dev(R, orc.BF16)
    xv = resid_values(R, orc.BF16)
    L64, S64 = orc.logits(T, orc.BF16, V, H, xv, threads=8, with_sumabs=True)
    raw, err = lhs.lhs_logits(tab, rd)
    assert int(err.item()) == 0
    Lg = raw.cpu().numpy()
    assert np.all(np.abs(Lg.astype(np.float64) - L64) <= RTOL[orc.BF16] * S64 + 1e-30)
    ids, vals, probs, err = lhs.lhs_logits_topk(tab, rd, k, temperature=1.3)
    assert int(err.item()) == 0
    ids, vals, probs = ids.cpu().numpy(), vals.cpu().numpy(), probs.cpu().numpy()
    for b in range(B):
        rid, rv = orc.topk_f32(Lg[b], k)
        assert np.array_equal(ids[b], rid), b
        assert np.array_equal(vals[b].view(np.uint32), rv.view(np.uint32)), b
        rp = orc.softmax_probs(Lg[b], 1.3, rid)
        assert np.all(np.abs(probs[b] - rp) <= PROB_RTOL * rp), b
    for b in (0, B // 2, B - 1):
        check_topk_against_fp64(ids[b], vals[b], L64[b], S64[b], k, RTOL[orc.BF16])


@pytest.mark.parametrize("dtype", [orc.F16, orc.BF16, orc.F32])
def test_lm_head_one_hot_and_integer_tables_exact(dtype):
    V, H = 777, 128
    T = wl.make_table(dtype, V, H, 0.02, cid=55, threads=2)
    tab = upload_table(T, dtype, V, H)
    cols = orc.decode_rows(T, dtype, H, 0, V)
    X = np.zeros((3, H), np.float32)
    X[0, 0] = 1.0
    X[1, 77] = 1.0
    X[2, H - 1] = 1.0
    raw, _ = lhs.lhs_logits(tab, to_dev(X))
    got = raw.cpu().numpy()
    for b, j in enumerate((0, 77, H - 1)):
        assert np.array_equal(got[b], cols[:, j])
    # integer-valued table and residuals: every partial sum is exact
    g = np.random.default_rng(1)
    Ti = g.integers(-2, 3, (V, H))
    Xi = g.integers(-8, 9, (5, H)).astype(np.float32)
    if dtype == orc.F32:
        Ts = Ti.astype(np.float32)
    elif dtype == orc.F16:
        Ts = Ti.astype(np.float16).view(np.uint16)
    else:
        Ts = wl.f32_to_bf16_bits(Ti.astype(np.float32))
    tab = upload_table(Ts, dtype, V, H)
    raw, _ = lhs.lhs_logits(tab, to_dev(Xi))
    assert np.array_equal(raw.cpu().numpy(), (Xi.astype(np.int64) @ Ti.T).astype(np.float32))


@pytest.mark.parametrize("dtype", [orc.BF16, orc.F32])
def test_topk_planted_ties_break_by_id(dtype):
    V, H, k = 2000, 64, 20
    base = wl.make_table(dtype, 40, H, 0.02, cid=9, threads=1)
    T = base[np.arange(V) % 40]          # every row repeated 50 times
    tab = upload_table(T, dtype, V, H)
    X = wl.residuals(9, 2, H)
    ids, vals, _, _ = lhs.lhs_logits_topk(tab, to_dev(X), k)
    raw, _ = lhs.lhs_logits(tab, to_dev(X))
    Lg = raw.cpu().numpy()
    for b in range(2):
        rid, rv = orc.topk_f32(Lg[b], k)
        assert np.array_equal(ids.cpu().numpy()[b], rid)
        # the winners are one row repeated: ids ascend within the tie
        top = ids.cpu().numpy()[b]
        same = Lg[b][top] == Lg[b][top[0]]
        assert np.all(np.diff(top[same]) > 0)


@pytest.mark.parametrize("V", [40000, 80000])
def test_gemm_topk_planted_ties_break_by_id(V):
    # tcgen05 path with 40 distinct rows repeated: the top logit repeats
    # V / 40 times, so every candidate of the merge falls in one bin
    # (1000 ranked directly; 2000 sent to the radix select)
    H, B, k = 64, 24, 50
    base = wl.make_table(orc.BF16, 40, H, 0.02, cid=19, threads=1)
    T = base[np.arange(V) % 40]
    tab = upload_table(T, orc.BF16, V, H)
    R = wl.residuals(19, B, H, (0.5, 8.0), orc.BF16)
    rd = _resid_dev(R, orc.BF16)
    ids, vals, probs, err = lhs.lhs_logits_topk(tab, rd, k)
    assert int(err.item()) == 0
    raw, _ = lhs.lhs_logits(tab, rd)
    Lg = raw.cpu().numpy()
    ids, vals, probs = ids.cpu().numpy(), vals.cpu().numpy(), probs.cpu().numpy()
    for b in range(B):
        rid, rv = orc.topk_f32(Lg[b], k)
        assert np.array_equal(ids[b], rid), b
        assert np.array_equal(vals[b].view(np.uint32), rv.view(np.uint32)), b
        rp = orc.softmax_probs(Lg[b], 1.0, rid)
        assert np.all(np.abs(probs[b] - rp) <= PROB_RTOL * rp), b


def _topk_matches_own_logits(tab, X, k, temperature=1.0):
    ids, vals, probs, err = lhs.lhs_logits_topk(tab, X, k, temperature=temperature)
    assert int(err.item()) == 0
    raw, _ = lhs.lhs_logits(tab, X)
    Lg = raw.cpu().numpy()
    ids, vals, probs = ids.cpu().numpy(), vals.cpu().numpy(), probs.cpu().numpy()
    for b in range(Lg.shape[0]):
        rid, rv = orc.topk_f32(Lg[b], k)
        assert np.array_equal(ids[b], rid), b
        assert np.array_equal(vals[b].view(np.uint32), rv.view(np.uint32)), b
        rp = orc.softmax_probs(Lg[b], temperature, rid)
        assert np.all(np.abs(probs[b] - rp) <= PROB_RTOL * rp), b


def test_topk_clustered_in_one_cta_range():
    # the 64 largest logits sit in the first rows, i.e. in one or two CTAs'
    # row ranges: the merge cannot bound them from a few entries per list
    V, H, k = 5000, 64, 40
    T = wl.make_table(orc.BF16, V, H, 0.02, cid=260, threads=4)
    col0 = (1.0 + np.arange(64, dtype=np.float32) / 128.0)
    T[:64, 0] = wl.f32_to_bf16_bits(col0)
    tab = upload_table(T, orc.BF16, V, H)
    X = wl.residuals(261, 2, H)
    X[:, 0] = 4.0
    _topk_matches_own_logits(tab, to_dev(X), k, temperature=0.9)


def test_topk_many_keys_above_the_merge_bound():
    # 32-row CTA ranges, each with 4 high logits and k = 5: every CTA's k-th
    # key is a low one, so the bound admits all 4 x G high keys (a top-k
    # GEMV runs one CTA per SM but one, which it leaves to the merge)
    G = torch.cuda.get_device_properties(0).multi_processor_count - 1
    V, H, k = 32 * G, 64, 5
    T = wl.make_table(orc.BF16, V, H, 0.02, cid=264, threads=4)
    rows = np.arange(V)
    hi = rows % 32 < 4
    col0 = np.where(hi, 2.0 + rows / V, 0.01).astype(np.float32)
    T[:, 0] = wl.f32_to_bf16_bits(col0)
    tab = upload_table(T, orc.BF16, V, H)
    X = wl.residuals(265, 2, H)
    X[:, 0] = 8.0
    _topk_matches_own_logits(tab, to_dev(X), k, temperature=1.1)


def test_topk_when_some_cta_lists_are_short():
    # 129 rows over 9 CTAs, the last with a single row: k = 128 needs nearly
    # every row and the sampled list prefixes hold padding
    V, H, k = 129, 64, 128
    T = wl.make_table(orc.BF16, V, H, 0.02, cid=262, threads=1)
    tab = upload_table(T, orc.BF16, V, H)
    X = wl.residuals(263, 3, H)
    _topk_matches_own_logits(tab, to_dev(X), k)


def test_f16_table_residual_out_of_range_flags_nonfinite():
    V, H = 256, 64
    T = wl.make_table(orc.F16, V, H, cid=3, threads=1)
    tab = upload_table(T, orc.F16, V, H)
    X = np.zeros((1, H), np.float32)
    X[0, 5] = 70000.0
    _, _, _, err = lhs.lhs_logits_topk(tab, to_dev(X), 3)
    assert int(err.item()) & lhs.LHS_ERRBIT_NONFINITE


@functools.lru_cache(maxsize=1)
def _workload_table(name):
    w = wl.WORKLOADS[name]
    T = wl.table_for(w)
    return T, upload_table(T, w.dtype, w.vocab, w.hidden)


@pytest.mark.parametrize("name,batch", [("tiny", 4), ("qwen05b", 1), ("gemma31b", 1),
                                        ("gemma31b", 8), ("batched", 256)])
def test_lm_head_workloads_full_size(name, batch):
    w = wl.WORKLOADS[name]
    T, tab = _workload_table(name)
    R = wl.residuals_for(w, batch)
    rd = _resid_dev(R, w.resid_dtype)
    xv = resid_values(R, w.resid_dtype)
    ids, vals, probs, err = lhs.lhs_logits_topk(tab, rd, w.k)
    raw, rerr = lhs.lhs_logits(tab, rd)
    assert int(err.item()) == 0 and int(rerr.item()) == 0
    ids, vals, probs = ids.cpu().numpy(), vals.cpu().numpy(), probs.cpu().numpy()
    # every residual's top-k against the oracle's selection over the GPU's
    # own logits; a sample of them against binary64 logits, row by row
    sample = list(range(batch)) if batch <= 8 else [0, 1, 77, 128, 200, 255]
    raw_h = raw.cpu().numpy()
    for b in range(batch):
        Lg = raw_h[b]
        rid, rv = orc.topk_f32(Lg, w.k)
        assert np.array_equal(ids[b], rid), b
        assert np.array_equal(vals[b].view(np.uint32), rv.view(np.uint32)), b
        rp = orc.softmax_probs(Lg, 1.0, rid)
        assert np.all(np.abs(probs[b] - rp) <= PROB_RTOL * rp), b
    for b in sample[:4]:
        L64, S64 = orc.logits(T, w.dtype, w.vocab, w.hidden, xv[b:b + 1], threads=16,
                              with_sumabs=True)
        Lg = raw_h[b].astype(np.float64)
        assert np.all(np.abs(Lg - L64[0]) <= RTOL[w.dtype] * S64[0] + 1e-30), b
        check_topk_against_fp64(ids[b], vals[b], L64[0], S64[0], w.k, RTOL[w.dtype])


# ---------------------------------------------------------------------------
# bounded waits
# ---------------------------------------------------------------------------

def test_bounded_wait_gives_up_and_context_survives():
    err = lhs.lhs_selftest_bounded_wait(50_000_000)
    torch.cuda.synchronize()
    assert int(err.item()) == lhs.LHS_ERRBIT_TIMEOUT
    # the context is still usable
    V, H = 256, 64
    T = wl.make_table(orc.F16, V, H, cid=1, threads=1)
    tab = upload_table(T, orc.F16, V, H)
    out, e2 = lhs.lhs_embed(tab, to_dev(np.array([3, 4], np.int32)), 1.0)
    ref, _ = orc.embed(T, orc.F16, V, H, np.array([3, 4], np.int32), 1.0)
    assert int(e2.item()) == 0 and np.array_equal(out.cpu().numpy(), ref)


# ---------------------------------------------------------------------------
# dedup-then-gather and mixed-precision rows
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n,vocab", [(0, 50), (1, 50), (300, 40), (5000, 262144), (70000, 3000)])
def test_unique_ids_parity(n, vocab):
    g = np.random.default_rng(n + vocab)
    ids = wl.zipf_ids(n % 97, n, vocab) if n else np.zeros(0, np.int32)
    if n > 10:
        ids[g.integers(0, n, 5)] = np.array([-1, vocab, vocab + 7, -1000, 2 ** 31 - 1], np.int32)
    uniq, inv, cnt, err = lhs.lhs_unique_ids(to_dev(ids) if n else torch.empty(0, dtype=torch.int32,
                                                                               device="cuda"), vocab)
    ru, ri, rbad = orc.unique_ids(ids, vocab)
    c = int(cnt.item())
    assert c == ru.size
    assert np.array_equal(uniq.cpu().numpy()[:c], ru)
    assert np.array_equal(inv.cpu().numpy(), ri)
    assert int(err.item()) == rbad


@pytest.mark.parametrize("dtype,H", [(orc.F32, 256), (orc.BF16, 896), (orc.Q8_0, 768), (orc.F16, 36)])
def test_embed_dedup_equals_embed(dtype, H):
    V = 5000
    T = wl.make_table(dtype, V, H, 0.02, cid=800 + H, threads=4)
    tab = upload_table(T, dtype, V, H)
    ids = wl.zipf_ids(801, 3000, V)
    ids[[5, 77]] = [-1, V]
    ids_d = to_dev(ids)
    out, err = lhs.lhs_embed_dedup(tab, ids_d, 27.712812)
    ref, rerr = orc.embed(T, dtype, V, H, ids, 27.712812)
    assert same_f32(out.cpu().numpy(), ref) and int(err.item()) == rerr
    plain, _ = lhs.lhs_embed(tab, ids_d, 27.712812)
    assert torch.equal(plain.view(torch.int32), out.view(torch.int32))


def test_embed_dedup_full_size_gemma_q8():
    w = wl.WORKLOADS["gemma_q8"]
    T = wl.table_for(w)
    tab = upload_table(T, w.dtype, w.vocab, w.hidden)
    ids = wl.ids_for(w)
    out, err = lhs.lhs_embed_dedup(tab, to_dev(ids), float(w.embed_scale))
    ref, rerr = orc.embed(T, w.dtype, w.vocab, w.hidden, ids, float(w.embed_scale))
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    assert int(err.item()) == rerr


def _random_mixed_table(vocab, hidden, seed):
    """Rows of random values stored in random row types (every type present),
    16-byte aligned; returns (data, offsets, types)."""
    g = np.random.default_rng(seed)
    types = g.integers(0, 5, vocab).astype(np.uint8)
    types[:5] = np.arange(5)
    if hidden % 32:
        types[types == orc.Q8_0] = orc.F32           # Q8_0 rows need hidden % 32 == 0
    chunks, offs, off = [], [], 0
    for r in range(vocab):
        dt = int(types[r])
        x = (g.standard_normal(hidden) * 0.05).astype(np.float32)
        if dt == orc.F32:
            b = x.tobytes()
        elif dt == orc.F16:
            b = x.astype(np.float16).tobytes()
        elif dt == orc.BF16:
            b = wl.f32_to_bf16_bits(x).tobytes()
        elif dt == orc.Q8_0:
            q = g.integers(-127, 128, hidden).astype(np.int8).reshape(-1, 32)
            d = np.abs(g.standard_normal(q.shape[0]) * 0.002).astype(np.float16)
            b = b"".join(d[i:i + 1].tobytes() + q[i].tobytes() for i in range(q.shape[0]))
        else:
            c = g.integers(0, 256, hidden).astype(np.uint8)
            c[(c & 0x7F) == 0x7F] = 0x3C                  # no NaN codes in the data
            b = c.tobytes()
        b += bytes((-len(b)) % 16)
        offs.append(off)
        chunks.append(b)
        off += len(b)
    return np.frombuffer(b"".join(chunks), np.uint8).copy(), np.array(offs, np.int64), types


@pytest.mark.parametrize("H", [64, 72, 256])
def test_embed_mixed_parity(H):
    V = 600
    data, offs, types = _random_mixed_table(V, H, seed=H)
    ids = wl.zipf_ids(H, 400, V)
    ids[[0, 1, 2, 3, 4]] = [0, 1, 2, 3, 4]
    ids[[7, 9]] = [-5, V]
    # malformed sidecar entries: unknown type, misaligned f32, past the end
    bad_types = types.copy()
    bad_offs = offs.copy()
    bad_types[10] = 9
    bad_types[11], bad_offs[11] = orc.F32, offs[11] + 2
    bad_offs[12] = data.size
    ids[[20, 21, 22]] = [10, 11, 12]
    ref, rerr = orc.embed_mixed(data, bad_offs, bad_types, V, H, ids, 1.5)
    out, err = lhs.lhs_embed_mixed(to_dev(data), to_dev(bad_offs), to_dev(bad_types), V, H, to_dev(ids), 1.5)
    assert same_f32(out.cpu().numpy(), ref)
    assert int(err.item()) == rerr == (orc.ERR_BAD_TOKEN | orc.ERR_MALFORMED)
