"""The pins catch plausible mistakes in the oracle.

Each mutant below is a copy of ``oracle/lhs_oracle.c`` with one planted
mistake: a dropped term, a wrong sign, index or constant, a transposed
operand, a wrong rounding or order rule.  The pin suite
(``tests/test_oracle_pins.py``) runs against the oracle built from each copy
(in a child process, the oracle pointed at it through ``LHS_ORACLE_SRC``)
and must fail; the unchanged source must pass.  A mutant the pins let
through would mean a function whose pins do not fix what it computes.

The mistakes are planted in the oracle on the CPU only; nothing here touches
the CUDA library.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(REPO, "oracle", "lhs_oracle.c")

# (name, text in the source, replacement, occurrences replaced)
MUTANTS = [
    # binary16 / bfloat16 / fp8 decoding
    ("f16 subnormal scale", "v = ldexp((double)m, -24);", "v = ldexp((double)m, -25);", 1),
    ("f16 exponent bias", "v = ldexp((double)(1024 + m), e - 25);", "v = ldexp((double)(1024 + m), e - 24);", 1),
    ("f16 sign dropped",
     "v = ldexp((double)(1024 + m), e - 25);   /* (1 + m/1024) * 2^(e-15) */\n    }\n    return sign ? -v : v;",
     "v = ldexp((double)(1024 + m), e - 25);   /* (1 + m/1024) * 2^(e-15) */\n    }\n    return v;", 1),
    ("bf16 shift", "uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b << 15;", 1),
    ("fp8 exponent bias", "v = ldexp((double)(8 + m), e - 10);", "v = ldexp((double)(8 + m), e - 11);", 1),
    ("fp8 NaN rule", "if (e == 15 && m == 7) {", "if (e == 15) {", 1),
    # f32 -> binary16 encoding
    ("f16 ties away from zero", "return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;", "return fl + 1.0;", 1),
    ("f16 saturation threshold", "if (a >= 65520.0) return sign | 0x7BFF;", "if (a > 65520.0) return sign | 0x7BFF;", 1),
    ("f16 NaN pattern", "if (isnan(x)) return 0x7E00;", "if (isnan(x)) return 0x7FFF;", 1),
    ("f16 fraction width", "quantum = ldexp(1.0, (E - 1) - 10);", "quantum = ldexp(1.0, (E - 1) - 9);", 1),
    # table layout and Q8_0
    ("q8 block bytes", "return (int64_t)(hidden / ORC_Q8_BLOCK) * ORC_Q8_BLOCK_BYTES;",
     "return (int64_t)(hidden / ORC_Q8_BLOCK) * (ORC_Q8_BLOCK_BYTES + 2);", 1),
    ("q8 scale dropped", "return (float)(d * (double)q);", "return (float)q;", 1),
    ("q8 code offset", "int q = (int)(int8_t)blk[2 + (j % ORC_Q8_BLOCK)];",
     "int q = (int)(int8_t)blk[1 + (j % ORC_Q8_BLOCK)];", 1),
    ("q8 codes unsigned", "int q = (int)(int8_t)blk[2 + (j % ORC_Q8_BLOCK)];",
     "int q = (int)blk[2 + (j % ORC_Q8_BLOCK)];", 1),
    ("f16 row stride", "case ORC_F16: return (float)orc_f16_value(orc_load_u16le(row + 2 * (size_t)j));",
     "case ORC_F16: return (float)orc_f16_value(orc_load_u16le(row + 2 * (size_t)(j ^ 1)));", 1),
    # embed gather + scale
    ("embed scale dropped", "float e = orc_row_element(row, dtype, j);\n                o[j] = e * scale;",
     "float e = orc_row_element(row, dtype, j);\n                o[j] = e;", 1),
    ("embed id bound", "float *o = out + t * (int64_t)hidden;\n        if (id < 0 || id >= vocab) {",
     "float *o = out + t * (int64_t)hidden;\n        if (id < 0 || id > vocab - 1 || id == vocab - 1) {", 1),
    ("embed error bit", "            *err_bits |= ORC_ERR_BAD_TOKEN;\n            continue;\n        }\n        {",
     "            continue;\n        }\n        {", 1),
    ("mixed row type", "float e = dt == ORC_FP8_E4M3 ? (float)orc_fp8_e4m3_value(row[j]) : orc_row_element(row, dt, j);",
     "float e = dt == ORC_FP8_E4M3 ? (float)orc_fp8_e4m3_value(row[j]) : orc_row_element(row, ORC_F16, j);", 1),
    # lm_head projection
    ("logits last term dropped", "for (j = 0; j < jb->hidden; ++j) {\n                double p",
     "for (j = 0; j < jb->hidden - 1; ++j) {\n                double p", 1),
    ("logits row reversed", "rowf[j] = orc_row_element(row, jb->dtype, j);",
     "rowf[j] = orc_row_element(row, jb->dtype, jb->hidden - 1 - j);", 1),
    ("logits output transposed", "jb->out[(int64_t)b * jb->ld + (v - jb->base)] = acc;",
     "jb->out[(v - jb->base) * jb->batch + b] = acc;", 1),
    ("logits product sign", "double p = (double)rowf[j] * (double)xb[j];",
     "double p = (double)rowf[j] * (double)xb[j] * (j == 0 ? -1.0 : 1.0);", 1),
    # top-k order
    ("topk ties by larger id", "if (a < b) return 0;\n    return ia < ib;", "if (a < b) return 0;\n    return ia > ib;", 1),
    ("topk NaN last", "        return an;\n", "        return bn;\n", 1),
    ("topk ascending", "if (a > b) return 1;\n    if (a < b) return 0;", "if (a < b) return 1;\n    if (a > b) return 0;", 1),
    # softmax prob
    ("softmax temperature multiplies", "- M) / temperature)", "- M) * temperature)", 2),
    ("softmax over the top-k only", "for (v = 0; v < V; ++v) S += exp(((double)logits[v] - M) / temperature);",
     "for (v = 0; v < k; ++v) S += exp(((double)logits[ids[v]] - M) / temperature);", 1),
    # wire codecs
    ("wire header order", "orc_store_u32le(buf + 4, (uint32_t)seq_len);\n    orc_store_u32le(buf + 8, flags);",
     "orc_store_u32le(buf + 8, (uint32_t)seq_len);\n    orc_store_u32le(buf + 4, flags);", 1),
    ("wire f16 byte order", "buf[16 + 2 * j] = (uint8_t)(h & 0xff);\n            buf[16 + 2 * j + 1] = (uint8_t)(h >> 8);",
     "buf[16 + 2 * j] = (uint8_t)(h >> 8);\n            buf[16 + 2 * j + 1] = (uint8_t)(h & 0xff);", 1),
    ("i8 scale denominator", "scale = m / 127.0f;", "scale = m / 128.0f;", 1),
    ("i8 truncating rounding", "float r = orc_rne_f32(y);", "float r = truncf(y);", 1),
    ("i8 rounding ties away", "return (fmodf(fl, 2.0f) == 0.0f) ? fl : fl + 1.0f;", "return fl + 1.0f;", 1),
    ("i8 codes unsigned on decode", "float q = (float)(int8_t)pos[8 + j];", "float q = (float)pos[8 + j];", 1),
    ("i8 zero point unchecked", "if (zp != 0.0f) {", "if (zp != zp) {", 1),
    ("i8 non-finite kept", "if (!isfinite(x[j])) nonfinite = 1;", "if (isnan(x[j])) nonfinite = 1;", 1),
    ("wire response header order", "orc_store_u32le(buf + 4, (uint32_t)seq_len);\n        orc_store_u32le(buf + 8, orc_bits_from_f32(latency_ms));",
     "orc_store_u32le(buf + 8, (uint32_t)seq_len);\n        orc_store_u32le(buf + 4, orc_bits_from_f32(latency_ms));", 1),
    ("wire response latency as an integer", "orc_store_u32le(buf + 8, orc_bits_from_f32(latency_ms));",
     "orc_store_u32le(buf + 8, (uint32_t)latency_ms);", 1),
    ("wire seq_len unchecked", "if (orc_load_u32le(buf + 4) != (uint32_t)seq_len) {",
     "if (orc_load_u32le(buf + 4) != orc_load_u32le(buf + 4)) {", 1),
    ("wire i8 position stride", "orc_i8_encode_position(x + p * hidden, hidden,\n                                   buf + 16 + p * (8 + (int64_t)hidden), err_bits);",
     "orc_i8_encode_position(x + p * hidden, hidden,\n                                   buf + 16 + p * (4 + (int64_t)hidden), err_bits);", 1),
]


def _run_pins(src_path):
    env = dict(os.environ, LHS_ORACLE_SRC=src_path, PYTHONDONTWRITEBYTECODE="1")
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(REPO, "tests", "test_oracle_pins.py"),
                        "-x", "-q", "-p", "no:cacheprovider"],
                       cwd=REPO, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-2000:]


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    base = open(SRC).read()
    d = tmp_path_factory.mktemp("mutants")
    jobs = {}
    ctl = d / "control.c"
    ctl.write_text(base)
    jobs["(unchanged)"] = str(ctl)
    for i, (name, old, new, count) in enumerate(MUTANTS):
        assert base.count(old) == count, f"mutant {name!r}: its anchor occurs {base.count(old)} times, not {count}"
        path = d / f"mutant_{i:02d}.c"
        path.write_text(base.replace(old, new))
        jobs[name] = str(path)
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        futs = {name: ex.submit(_run_pins, path) for name, path in jobs.items()}
        return {name: f.result() for name, f in futs.items()}


def test_unchanged_oracle_passes_the_pins(outcomes):
    rc, out = outcomes["(unchanged)"]
    assert rc == 0, out


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(outcomes, name):
    rc, out = outcomes[name]
    # exit code 1: the suite ran and a pin failed (not a crash or a build error)
    assert rc == 1, f"mutant {name!r} exit {rc}:\n{out}"
    assert "CalledProcessError" not in out, f"mutant {name!r} did not build:\n{out}"
