"""Pins of the oracle to facts other than itself (CPU only).

Each check compares the oracle with what the pages print, a closed form, an
invariant, brute force on a tiny case, or an independent library routine
(numpy's own IEEE conversions and BLAS), chosen so that a dropped term, a
wrong sign, index or operand order in the oracle fails at least one of them.
"""
import json
import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle as orc
import workloads as wl


def _golden(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# binary16 / bfloat16
# ---------------------------------------------------------------------------

def test_f16_decode_all_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = orc.f16_value(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signs of zeros
    assert math.copysign(1.0, ours[0x8000]) == -1.0


@pytest.mark.parametrize("bits,value", [
    (0x3C00, 1.0), (0xC000, -2.0), (0x7BFF, 65504.0), (0x0400, 2.0 ** -14),
    (0x0001, 2.0 ** -24), (0x03FF, 1023 * 2.0 ** -24), (0x3555, 0.333251953125),
    (0x7C00, math.inf), (0xFC00, -math.inf)])
def test_f16_decode_hand_values(bits, value):
    assert orc.f16_value([bits])[0] == value


@pytest.mark.parametrize("bits,value", [
    (0x3F80, 1.0), (0xC000, -2.0), (0x4049, 3.140625), (0x0001, 2.0 ** -133),
    (0x7F80, math.inf), (0x0080, 2.0 ** -126), (0x3E80, 0.25)])
def test_bf16_decode_hand_values(bits, value):
    assert float(orc.bf16_to_f32([bits])[0]) == value


def test_f16_encode_round_trips_every_finite_f16():
    # ADR-0009 Context: f16 round trip is lossless for f16-representable values
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    exp = (bits >> 10) & 0x1F
    finite = bits[exp != 31]
    assert finite.size == 63488
    vals = finite.view(np.float16).astype(np.float32)
    assert np.array_equal(orc.f16_from_f32_sat(vals), finite)


def test_f16_encode_matches_numpy_rounding_in_range():
    g = np.random.default_rng(123)
    # log-uniform magnitudes across the normal and subnormal f16 range
    mag = np.exp2(g.uniform(-27, 15.99, 400000)).astype(np.float32)
    x = (mag * np.where(g.random(mag.size) < 0.5, -1, 1)).astype(np.float32)
    # exact ties: midpoints between adjacent f16 values
    h = g.integers(0, 0x7BFE, 20000).astype(np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).astype(np.uint16).view(np.float16).astype(np.float64)
    ties = ((lo + hi) / 2).astype(np.float32)
    x = np.concatenate([x, ties, -ties])
    ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(orc.f16_from_f32_sat(x), ref)


def test_f16_encode_saturates_finite_overflow(golden_dir):
    # ADR-0009 Trade-offs: clamp-to-max, not NaN/inf for finite values
    ex = _golden(golden_dir, "wire_worked_examples.json")["f16"]
    got = orc.f16_from_f32_sat(np.array(ex["x"], np.float32))
    assert [int(b) for b in got] == [int(b, 16) for b in ex["bits"]]
    cases = {65519.99: 0x7BFF, 65520.0: 0x7BFF, 1e30: 0x7BFF, -65520.0: 0xFBFF,
             float(np.finfo(np.float32).max): 0x7BFF}
    for v, b in cases.items():
        assert int(orc.f16_from_f32_sat(np.float32(v))[0]) == b, v
    assert int(orc.f16_from_f32_sat(np.float32(np.inf))[0]) == 0x7C00
    assert int(orc.f16_from_f32_sat(np.float32(-np.inf))[0]) == 0xFC00
    assert int(orc.f16_from_f32_sat(np.float32(np.nan))[0]) == 0x7E00
    assert int(orc.f16_from_f32_sat(np.float32(-0.0))[0]) == 0x8000
    # half-way cases, ties to even
    assert int(orc.f16_from_f32_sat(np.float32(1 + 2 ** -11))[0]) == 0x3C00
    assert int(orc.f16_from_f32_sat(np.float32(1 + 3 * 2 ** -11))[0]) == 0x3C02
    assert int(orc.f16_from_f32_sat(np.float32(2 ** -25))[0]) == 0x0000
    assert int(orc.f16_from_f32_sat(np.float32(3 * 2 ** -25))[0]) == 0x0002


# ---------------------------------------------------------------------------
# table layout (HELIX §3) and the page's sizes
# ---------------------------------------------------------------------------

def test_row_bytes_and_sizes_match_pages(golden_dir):
    g = _golden(golden_dir, "page_figures.json")
    V, H = g["qwen05b_vocab"]["value"], g["qwen05b_hidden"]["value"]
    assert orc.row_bytes(orc.F32, H) == g["qwen05b_row_bytes_fp32"]["value"]
    assert orc.row_bytes(orc.BF16, H) == g["qwen05b_row_bytes_bf16"]["value"]
    assert orc.row_bytes(orc.F16, H) == g["qwen05b_row_bytes_bf16"]["value"]
    assert round(V * orc.row_bytes(orc.F32, H) / 2 ** 20, 2) == \
        g["qwen05b_table_mib_fp32"]["value"]
    assert g["qwen05b_session_rows"]["value"] * orc.row_bytes(orc.F32, H) / 1024 == \
        g["qwen05b_session_kib_fp32"]["value"]
    assert orc.row_bytes(orc.F32, 5376) == g["gemma31b_embed_row_bytes_f32"]["value"]
    assert orc.row_bytes(orc.F32, 2560) == g["gemma3_4b_row_bytes_f32"]["value"]
    gv = g["gemma3_4b_vocab"]["value"]
    assert round(gv * orc.row_bytes(orc.F16, 2560) / 1e9, 2) == \
        g["gemma3_4b_table_gb_f16"]["value"]
    assert round(gv * orc.row_bytes(orc.F32, 2560) / 1e9, 2) == \
        g["gemma3_4b_table_gb_f32"]["value"]
    # Q8_0: hidden/32 blocks of (f16 scale + 32 codes)
    assert g["q8_block_values"]["value"] == orc.Q8_BLOCK
    assert orc.row_bytes(orc.Q8_0, g["gemma_embedding_hidden"]["value"]) == 24 * 34
    assert orc.row_bytes(orc.Q8_0, 100) == -1


def _fingerprint_f32(V, H):
    """Entry (i, j) has a bit pattern that is a hash of (i, j), kept finite."""
    i = np.arange(V, dtype=np.uint64)[:, None]
    j = np.arange(H, dtype=np.uint64)[None, :]
    h = (i * np.uint64(0x9E3779B1) + j * np.uint64(0x85EBCA77) + np.uint64(12345))
    h = (h ^ (h >> np.uint64(15))) * np.uint64(0x2C1B3C6D)
    h = (h ^ (h >> np.uint64(12))) & np.uint64(0xFFFFFFFF)
    b = h.astype(np.uint32)
    # clear the top exponent bit to stay finite (exponent <= 127)
    b &= np.uint32(0xBFFFFFFF)
    return b.view(np.float32)


def test_embed_rows_are_at_i_times_row_bytes_f32():
    V, H = 1031, 96
    T = _fingerprint_f32(V, H)
    ids = np.array([0, V - 1, 5, 5, 517, 1, V - 2], np.int32)
    out, err = orc.embed(T, orc.F32, V, H, ids, 1.0)
    assert err == 0
    assert np.array_equal(out.view(np.uint32), T[ids].view(np.uint32))


@pytest.mark.parametrize("dtype", [orc.F16, orc.BF16])
def test_embed_rows_16bit(dtype):
    V, H = 777, 64
    bits = _fingerprint_f32(V, H).view(np.uint32)
    if dtype == orc.F16:
        b16 = (bits & np.uint32(0xBBFF)).astype(np.uint16)   # finite f16
        expect = b16.view(np.float16).astype(np.float32)
    else:
        b16 = (bits >> 16).astype(np.uint16)
        expect = (b16.astype(np.uint32) << 16).view(np.float32)
    ids = np.array([V - 1, 0, 300, 300, 2], np.int32)
    out, err = orc.embed(b16, dtype, V, H, ids, 1.0)
    assert err == 0
    assert np.array_equal(out.view(np.uint32), expect[ids].view(np.uint32))


def test_embed_scale_is_one_binary32_multiply():
    V, H = 64, 32
    T = np.random.default_rng(5).standard_normal((V, H)).astype(np.float32)
    s = np.float32(math.sqrt(32.0))
    ids = np.arange(V, dtype=np.int32)[::-1].copy()
    out, _ = orc.embed(T, orc.F32, V, H, ids, s)
    assert np.array_equal(out, T[ids] * s)


def _pack_q8(d_bits, q):
    """Test's own packing of a Q8_0 table: rows of blocks (f16 d LE, 32 int8)."""
    V, nb = d_bits.shape
    out = bytearray()
    for r in range(V):
        for b in range(nb):
            out += struct.pack("<H", int(d_bits[r, b]))
            out += struct.pack("<32b", *[int(v) for v in q[r, b]])
    return np.frombuffer(bytes(out), np.uint8).reshape(V, nb * 34)


def test_embed_q8_0_closed_form(golden_dir):
    # Port Spec forward graph: x = token_embd[ids] * sqrt(768), q8_0 dequant
    g = _golden(golden_dir, "page_figures.json")
    H = g["gemma_embedding_hidden"]["value"]
    V, nb = 37, H // 32
    r = np.arange(V)[:, None]
    b = np.arange(nb)[None, :]
    d = ((1 + (r % 7) / 8.0) * np.exp2(-(3 + (b % 5)))).astype(np.float16)
    lanes = np.arange(32)[None, None, :]
    q = (((r[:, :, None] * 31 + b[:, :, None] * 7 + lanes * 3) % 255) - 127).astype(np.int8)
    table = _pack_q8(d.view(np.uint16), q)
    s = np.float32(math.sqrt(768.0))
    assert s.view(np.uint32) == 0x41DDB3D7
    ids = np.array([0, V - 1, 11, 11, 3], np.int32)
    out, err = orc.embed(table, orc.Q8_0, V, H, ids, s)
    assert err == 0
    # value = d * q exactly, then one binary32 multiply by sqrt(768)
    val = (d.astype(np.float64)[:, :, None] * q.astype(np.float64)).reshape(V, H)
    expect = val.astype(np.float32)[ids] * s
    assert np.array_equal(out, expect)


def test_embed_bad_ids_zero_row_and_error_bit():
    V, H = 50, 32
    T = _fingerprint_f32(V, H)
    ids = np.array([3, -1, V, 2 ** 31 - 1, 4], np.int32)
    out, err = orc.embed(T, orc.F32, V, H, ids, 1.0)
    assert err == orc.ERR_BAD_TOKEN
    assert np.all(out[1:4] == 0)
    assert np.array_equal(out[0].view(np.uint32), T[3].view(np.uint32))
    assert np.array_equal(out[4].view(np.uint32), T[4].view(np.uint32))


# ---------------------------------------------------------------------------
# lm_head (ADR-0008 /v1/logits: residual @ lm_head.T)
# ---------------------------------------------------------------------------

def _any_table(dtype, V, H, seed=0):
    return wl.make_table(dtype, V, H, 0.02, cid=seed, threads=1)


@pytest.mark.parametrize("dtype", [orc.F32, orc.F16, orc.BF16, orc.Q8_0])
def test_logits_one_hot_residual_returns_column(dtype):
    V, H = 300, 64
    T = _any_table(dtype, V, H, seed=dtype)
    cols = orc.decode_rows(T, dtype, H, 0, V)
    for j in (0, 17, H - 1):
        x = np.zeros((1, H), np.float32)
        x[0, j] = 1.0
        L = orc.logits(T, dtype, V, H, x)
        assert np.array_equal(L[0], cols[:, j].astype(np.float64))


def test_logits_integer_table_is_exact():
    V, H, B = 257, 96, 3
    g = np.random.default_rng(9)
    Ti = g.integers(-2, 3, (V, H))
    Xi = g.integers(-8, 9, (B, H))
    T16 = Ti.astype(np.float16).view(np.uint16)
    L = orc.logits(T16, orc.F16, V, H, Xi.astype(np.float32))
    assert np.array_equal(L, (Xi @ Ti.T).astype(np.float64))


def test_logits_match_blas_and_are_transposed_correctly():
    V, H, B = 401, 80, 4
    g = np.random.default_rng(10)
    T = g.standard_normal((V, H)).astype(np.float32)
    X = g.standard_normal((B, H)).astype(np.float32)
    L, S = orc.logits(T, orc.F32, V, H, X, with_sumabs=True)
    ref = X.astype(np.float64) @ T.astype(np.float64).T
    assert np.all(np.abs(L - ref) <= 1e-13 * S)
    assert np.allclose(S, np.abs(X.astype(np.float64)) @ np.abs(T.astype(np.float64)).T,
                       rtol=1e-13)
    # sub-ranges and thread counts give identical numbers
    part = orc.logits(T, orc.F32, V, H, X, v0=100, v1=250)
    assert np.array_equal(part, L[:, 100:250])
    assert np.array_equal(orc.logits(T, orc.F32, V, H, X, threads=4), L)


# ---------------------------------------------------------------------------
# top-k and prob
# ---------------------------------------------------------------------------

def _lexsort_topk(vals, k):
    v = np.asarray(vals, np.float64)
    key_nan = np.isnan(v)
    vv = np.where(key_nan, 0.0, v) + 0.0      # -0 -> +0
    order = np.lexsort((np.arange(v.size), -vv, ~key_nan))
    return order[:k]


@pytest.mark.parametrize("seed", range(6))
def test_topk_brute_force_with_planted_ties(seed):
    g = np.random.default_rng(seed)
    V = int(g.integers(1, 65))
    vals = g.choice(np.array([-1.5, -0.0, 0.0, 0.25, 2.0, 7.0], np.float32), V)
    for k in range(0, V + 1):
        ids, got = orc.topk_f32(vals, k)
        ref = _lexsort_topk(vals, k)
        assert np.array_equal(ids, ref)
        assert np.array_equal(got.view(np.uint32), vals[ref].view(np.uint32))
        ids64, _ = orc.topk_f64(vals.astype(np.float64), k)
        assert np.array_equal(ids64, ref)


def test_topk_nan_ranks_first_and_random_matches_sort():
    v = np.array([1.0, np.nan, 3.0, np.nan, -np.inf, np.inf], np.float32)
    ids, _ = orc.topk_f32(v, 6)
    assert list(ids) == [1, 3, 5, 2, 0, 4]
    x = np.random.default_rng(3).standard_normal(5000).astype(np.float32)
    ids, vals = orc.topk_f32(x, 50)
    assert np.array_equal(ids, np.argsort(-x, kind="stable")[:50])


def test_softmax_probs_invariants():
    g = np.random.default_rng(4)
    L = g.standard_normal(1000).astype(np.float32) * 3
    allids = np.arange(1000, dtype=np.int32)
    for T in (0.5, 1.0, 2.0):
        p = orc.softmax_probs(L, T, allids)
        assert abs(p.sum() - 1.0) < 1e-12
        assert np.all(p > 0)
    assert np.allclose(orc.softmax_probs(np.zeros(64, np.float32), 1.0, [5, 9]), 1 / 64,
                       rtol=0, atol=1e-15)
    two = orc.softmax_probs(np.array([0.0, 1.0], np.float32), 1.0, [1, 0])
    assert abs(two[0] - math.e / (1 + math.e)) < 1e-15
    # temperature divides the logits: T=2 on 2L equals T=1 on L
    a = orc.softmax_probs(L * 2, 2.0, allids[:20])
    b = orc.softmax_probs(L, 1.0, allids[:20])
    assert np.allclose(a, b, rtol=1e-13, atol=0)
    # probabilities are ordered like the logits
    ids, _ = orc.topk_f32(L, 10)
    p = orc.softmax_probs(L, 1.0, ids)
    assert np.all(np.diff(p) <= 0)


# ---------------------------------------------------------------------------
# wire codecs (ADR-0009 Wire Layout)
# ---------------------------------------------------------------------------

def test_wire_sizes_match_pages(golden_dir):
    g = _golden(golden_dir, "page_figures.json")
    hdr = g["wire_header_bytes"]["value"]
    per = g["wire_bytes_per_value"]["value"]
    assert orc.wire_bytes(orc.WIRE_F32, 1, 5120) - hdr == \
        g["wire_f32_residual_5120_bytes"]["value"]
    for s, h in ((1, 2560), (32, 4096), (256, 5120)):
        assert orc.wire_bytes(orc.WIRE_F32, s, h) == hdr + per["f32"] * s * h
        assert orc.wire_bytes(orc.WIRE_F16, s, h) == hdr + per["f16"] * s * h
        assert orc.wire_bytes(orc.WIRE_I8, s, h) == \
            hdr + per["i8"] * s * h + g["wire_i8_position_overhead_bytes"]["value"] * s
    over = orc.wire_bytes(orc.WIRE_I8, 256, 5120) - hdr - 256 * 5120
    assert over == g["wire_i8_overhead_seq256_bytes"]["value"]
    assert 256 * 5120 / 2 ** 20 == g["wire_i8_payload_seq256_h5120_mib"]["value"]


def test_wire_header_layout_and_f32_identity():
    x = np.random.default_rng(1).standard_normal((3, 8)).astype(np.float32)
    buf, err = orc.wire_encode(orc.WIRE_F32, x, layer=7, flags=0xABCD, top_k=40)
    assert err == 0
    assert struct.unpack("<4I", buf[:16].tobytes()) == (7, 3, 0xABCD, 40)
    assert buf[16:].tobytes() == x.astype("<f4").tobytes()
    y, err = orc.wire_decode(orc.WIRE_F32, buf, 3, 8)
    assert err == 0 and np.array_equal(y.view(np.uint32), x.view(np.uint32))


def test_wire_f16_layout_and_lossless_round_trip():
    g = np.random.default_rng(2)
    x = g.standard_normal((5, 64)).astype(np.float32) * 30
    buf, err = orc.wire_encode(orc.WIRE_F16, x, layer=1, flags=2, top_k=3)
    assert err == 0 and buf.size == 16 + 5 * 64 * 2
    assert struct.unpack("<4I", buf[:16].tobytes()) == (1, 5, 2, 3)
    assert np.array_equal(np.frombuffer(buf[16:].tobytes(), "<u2"),
                          x.astype(np.float16).view(np.uint16).reshape(-1))
    # f16-representable values survive the round trip exactly
    xr = x.astype(np.float16).astype(np.float32)
    b2, _ = orc.wire_encode(orc.WIRE_F16, xr)
    y, err = orc.wire_decode(orc.WIRE_F16, b2, 5, 64)
    assert err == 0 and np.array_equal(y, xr)


def test_wire_i8_worked_example(golden_dir):
    ex = _golden(golden_dir, "wire_worked_examples.json")["i8"]
    x = np.array(ex["x"], np.float32)
    buf, err = orc.wire_encode(orc.WIRE_I8, x, ex["layer"], ex["flags"], ex["top_k"])
    assert err == 0
    s, h = x.shape
    assert struct.unpack("<4I", buf[:16].tobytes()) == (ex["layer"], s, ex["flags"],
                                                       ex["top_k"])
    for p in range(s):
        off = 16 + p * (8 + h)
        scale_bits, zp_bits = struct.unpack("<II", buf[off:off + 8].tobytes())
        assert scale_bits == int(ex["scale_bits"][p], 16)
        assert zp_bits == 0
        assert list(buf[off + 8: off + 8 + h].view(np.int8)) == ex["q"][p]
    y, err = orc.wire_decode(orc.WIRE_I8, buf, s, h)
    assert err == 0
    got = [[int(v) for v in row] for row in y.view(np.uint32)]
    want = [[int(b, 16) for b in row] for row in ex["decoded_bits"]]
    assert got == want


def _exact_rne(fr: Fraction) -> int:
    fl = math.floor(fr)
    d = fr - fl
    if d > Fraction(1, 2):
        return fl + 1
    if d < Fraction(1, 2):
        return fl
    return fl if fl % 2 == 0 else fl + 1


def test_wire_i8_formula_bound_and_max_code():
    g = np.random.default_rng(6)
    sig = g.uniform(0.5, 8, size=(16, 1)).astype(np.float32)
    x = (g.standard_normal((16, 200)).astype(np.float32) * sig)
    x[3] = 0.0                                   # all-zero position
    x[5, 7] = -np.abs(x[5]).max() * 2            # negative max
    buf, err = orc.wire_encode(orc.WIRE_I8, x)
    assert err == 0
    y, err = orc.wire_decode(orc.WIRE_I8, buf, 16, 200)
    assert err == 0
    for p in range(16):
        off = 16 + p * 208
        scale = np.frombuffer(buf[off:off + 4].tobytes(), "<f4")[0]
        q = buf[off + 8:off + 208].view(np.int8).astype(np.int64)
        m = np.abs(x[p]).max()
        assert scale == np.float32(m) / np.float32(127)     # binary32 division
        if m == 0:
            assert scale == 0 and np.all(q == 0) and np.all(y[p] == 0)
            continue
        # the position max maps to +-127
        jm = int(np.argmax(np.abs(x[p])))
        assert abs(q[jm]) == 127 and np.sign(q[jm]) == np.sign(x[p, jm])
        # q = rne(binary32(x / scale)), checked with exact rationals
        for j in range(0, 200, 13):
            quot = np.float32(x[p, j]) / np.float32(scale)
            assert q[j] == max(-127, min(127, _exact_rne(Fraction(float(quot)))))
        # decode is q * scale in binary32, and the error bound of the page
        assert np.array_equal(y[p], q.astype(np.float32) * scale)
        err_abs = np.abs(y[p].astype(np.float64) - x[p].astype(np.float64))
        bound = float(scale) / 2 * (1 + 2 ** -20) + np.abs(y[p]) * 2 ** -23
        assert np.all(err_abs <= bound)


def test_wire_i8_nonfinite_and_malformed():
    x = np.ones((3, 16), np.float32)
    x[1, 4] = np.inf
    buf, err = orc.wire_encode(orc.WIRE_I8, x)
    assert err == orc.ERR_NONFINITE
    off = 16 + 1 * 24
    assert buf[off:off + 24].tobytes() == bytes(24)
    # header seq_len must match the caller's seq_len
    canary = np.full((2, 16), 7.0, np.float32)
    y, err = orc.wire_decode(orc.WIRE_I8, buf, 2, 16, out=canary.copy())
    assert err == orc.ERR_MALFORMED and np.all(y == 7.0)
    # a non-zero zero_point is not the symmetric format: that position is
    # flagged and left untouched, the other positions decode
    good, _ = orc.wire_encode(orc.WIRE_I8, np.ones((2, 16), np.float32))
    bad = good.copy()
    bad[16 + 24 + 4:16 + 24 + 8] = np.frombuffer(struct.pack("<f", 0.5), np.uint8)
    y, err = orc.wire_decode(orc.WIRE_I8, bad, 2, 16, out=canary.copy())
    assert err == orc.ERR_MALFORMED and np.all(y[1] == 7.0) and np.all(y[0] == 1.0)
    y, err = orc.wire_decode(orc.WIRE_F16, orc.wire_encode(orc.WIRE_F16, x)[0], 2, 16,
                             out=canary.copy())
    assert err == orc.ERR_MALFORMED and np.all(y == 7.0)
    with pytest.raises(ValueError):       # buffer shorter than the message
        orc.wire_decode(orc.WIRE_F16, orc.wire_encode(orc.WIRE_F16, x)[0], 4, 16)


def test_wire_response_header_and_payloads():
    # ADR-0009 Wire Layout, "Single-layer response": [layer u32][seq_len u32]
    # [latency_ms f32] (little-endian), then the request's payload
    g = np.random.default_rng(11)
    x = g.standard_normal((3, 8)).astype(np.float32) * 3
    assert orc.wire_response_bytes(orc.WIRE_F32, 3, 8) == 12 + 3 * 8 * 4
    assert orc.wire_response_bytes(orc.WIRE_F16, 3, 8) == 12 + 3 * 8 * 2
    assert orc.wire_response_bytes(orc.WIRE_I8, 3, 8) == 12 + 3 * (8 + 8)
    buf, err = orc.wire_encode_response(orc.WIRE_F32, x, layer=9, latency_ms=2.1)
    assert err == 0 and buf.size == 12 + 96
    assert buf[:12].tobytes() == struct.pack("<IIf", 9, 3, 2.1)
    assert buf[12:].tobytes() == x.astype("<f4").tobytes()
    y, err = orc.wire_decode_response(orc.WIRE_F32, buf, 3, 8)
    assert err == 0 and np.array_equal(y.view(np.uint32), x.view(np.uint32))
    buf, err = orc.wire_encode_response(orc.WIRE_F16, x, layer=4, latency_ms=0.1)
    assert err == 0 and buf[:12].tobytes() == struct.pack("<IIf", 4, 3, 0.1)
    assert np.array_equal(np.frombuffer(buf[12:].tobytes(), "<u2"),
                          x.astype(np.float16).view(np.uint16).reshape(-1))
    y, err = orc.wire_decode_response(orc.WIRE_F16, buf, 3, 8)
    assert err == 0 and np.array_equal(y, x.astype(np.float16).astype(np.float32))


def test_wire_response_i8_worked_example(golden_dir):
    ex = _golden(golden_dir, "wire_worked_examples.json")["i8"]
    x = np.array(ex["x"], np.float32)
    s, h = x.shape
    buf, err = orc.wire_encode_response(orc.WIRE_I8, x, layer=ex["layer"], latency_ms=1.5)
    assert err == 0 and buf.size == 12 + s * (8 + h)
    assert buf[:12].tobytes() == struct.pack("<IIf", ex["layer"], s, 1.5)
    for p in range(s):
        off = 12 + p * (8 + h)
        scale_bits, zp_bits = struct.unpack("<II", buf[off:off + 8].tobytes())
        assert scale_bits == int(ex["scale_bits"][p], 16) and zp_bits == 0
        assert list(buf[off + 8: off + 8 + h].view(np.int8)) == ex["q"][p]
    y, err = orc.wire_decode_response(orc.WIRE_I8, buf, s, h)
    assert err == 0
    assert [[int(v) for v in row] for row in y.view(np.uint32)] == \
        [[int(b, 16) for b in row] for row in ex["decoded_bits"]]


def test_wire_response_malformed():
    x = np.ones((2, 16), np.float32)
    canary = np.full((2, 16), 7.0, np.float32)
    buf, _ = orc.wire_encode_response(orc.WIRE_I8, x, layer=1, latency_ms=0.5)
    # the header's seq_len (its second word) must match the caller's
    bad = buf.copy()
    bad[4:8] = np.frombuffer(struct.pack("<I", 3), np.uint8)
    y, err = orc.wire_decode_response(orc.WIRE_I8, bad, 2, 16, out=canary.copy())
    assert err == orc.ERR_MALFORMED and np.all(y == 7.0)
    # a non-zero zero_point: that position flagged and left untouched
    bad = buf.copy()
    bad[12 + 24 + 4:12 + 24 + 8] = np.frombuffer(struct.pack("<f", 0.5), np.uint8)
    y, err = orc.wire_decode_response(orc.WIRE_I8, bad, 2, 16, out=canary.copy())
    assert err == orc.ERR_MALFORMED and np.all(y[1] == 7.0) and np.all(y[0] == 1.0)
    with pytest.raises(ValueError):       # buffer shorter than the message
        orc.wire_decode_response(orc.WIRE_F16, orc.wire_encode_response(orc.WIRE_F16, x)[0], 4, 16)


# ---------------------------------------------------------------------------
# Mixed-precision rows (HELIX §3 sidecar) and dedup (HELIX Appendix B)
# ---------------------------------------------------------------------------

def test_fp8_e4m3_published_values():
    # OCP 8-bit floating point, E4M3: bias 7, no infinities, S.1111.111 NaN,
    # largest finite 448, smallest normal 2^-6, smallest subnormal 2^-9
    v = orc.fp8_e4m3_value(np.arange(256, dtype=np.uint8))
    assert v[0x38] == 1.0 and v[0xB8] == -1.0
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0
    assert v[0x08] == 2.0 ** -6 and v[0x01] == 2.0 ** -9
    assert v[0x00] == 0.0 and math.copysign(1.0, v[0x80]) == -1.0
    nan = np.isnan(v)
    assert sorted(np.nonzero(nan)[0].tolist()) == [0x7F, 0xFF]
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0)                       # codes order like values
    assert np.array_equal(v[0x80:0xFF], -v[:0x7F])         # sign bit only flips the sign
    # within each binade the eight codes are evenly spaced by 2^(e-10)
    for e in range(1, 16):
        codes = [(e << 3) | m for m in range(8) if (e << 3) | m <= 0x7E]
        step = np.diff(v[codes])
        assert np.all(step == 2.0 ** (e - 10))


def _mixed_table(values, dtypes):
    """Rows of `values` (k * 2^-3, |k| <= 15: exact in every row type) stored
    each in its own type; returns (data, offsets)."""
    vocab, hidden = values.shape
    chunks, offsets, off = [], [], 0
    for r in range(vocab):
        x = values[r].astype(np.float32)
        dt = int(dtypes[r])
        if dt == orc.F32:
            b = x.tobytes()
        elif dt == orc.F16:
            b = x.astype(np.float16).tobytes()
        elif dt == orc.BF16:
            b = (x.view(np.uint32) >> 16).astype(np.uint16).tobytes()
        elif dt == orc.Q8_0:
            q = np.rint(x * 8).astype(np.int8).reshape(-1, 32)
            d = np.float16(0.125).tobytes()
            b = b"".join(d + blk.tobytes() for blk in q)
        else:   # fp8 e4m3: pick the code whose exact value equals x
            table = orc.fp8_e4m3_value(np.arange(0x7F, dtype=np.uint8))
            codes = []
            for val in x:
                c = int(np.nonzero(table == abs(val))[0][0])
                codes.append(c | (0x80 if val < 0 else 0))
            b = bytes(codes)
        b += bytes((-len(b)) % 16)        # 16-byte row alignment in the data
        offsets.append(off)
        chunks.append(b)
        off += len(b)
    return np.frombuffer(b"".join(chunks), np.uint8), np.array(offsets, np.int64)


def test_mixed_rows_match_the_homogeneous_gather():
    g = np.random.default_rng(5)
    vocab, hidden = 40, 64
    values = (g.integers(-15, 16, (vocab, hidden)) * 0.125).astype(np.float32)
    dtypes = np.array([r % 5 for r in range(vocab)], np.uint8)   # every row type
    data, offs = _mixed_table(values, dtypes)
    ids = np.array([0, 1, 2, 3, 4, 39, 17, 17, -1, 40], np.int32)
    got, err = orc.embed_mixed(data, offs, dtypes, vocab, hidden, ids, 3.0)
    ref, ref_err = orc.embed(values, orc.F32, vocab, hidden, ids, 3.0)
    assert np.array_equal(got, ref) and err == ref_err == orc.ERR_BAD_TOKEN
    # an unknown row type: zero row, MALFORMED
    bad = dtypes.copy()
    bad[7] = 9
    got, err = orc.embed_mixed(data, offs, bad, vocab, hidden, [7, 6], 1.0)
    assert np.all(got[0] == 0.0) and np.array_equal(got[1], values[6]) and err == orc.ERR_MALFORMED


def test_unique_ids_against_brute_force():
    g = np.random.default_rng(9)
    for n, vocab in ((0, 10), (1, 10), (50, 7), (300, 1000)):
        ids = g.integers(-3, vocab + 3, n).astype(np.int32)
        uniq, inv, bad = orc.unique_ids(ids, vocab)
        valid = [int(i) for i in ids if 0 <= i < vocab]
        assert uniq.tolist() == sorted(set(valid))
        for i, x in enumerate(ids):
            if 0 <= x < vocab:
                assert uniq[inv[i]] == x
            else:
                assert inv[i] == -1
        assert bad == (1 if len(valid) < n else 0)
