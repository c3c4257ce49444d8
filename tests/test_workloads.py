"""The seeded input generators follow the stated recipe.

``workloads/`` feeds both the oracle and the CUDA path, so what it draws is
checked here on its own: determinism, the layouts the service reads, and the
distributions the design notes state (N(0, 0.02) tables, Q8_0 codes in
[-127, 127] with non-negative f16 scales, Zipf(1.1) ids, per-row residual
scales).  CPU only, small sizes.
"""
import numpy as np
import pytest
import torch

import workloads as wl


def test_tables_do_not_depend_on_the_thread_count():
    V = 2 * (1 << 14) + 123                 # three chunks, the last ragged
    for dt in (wl.F32, wl.F16, wl.BF16, wl.Q8_0):
        a = wl.make_table(dt, V, 64, 0.02, cid=7, threads=1)
        b = wl.make_table(dt, V, 64, 0.02, cid=7, threads=4)
        assert np.array_equal(a, b)
        c = wl.make_table(dt, V, 64, 0.02, cid=8, threads=4)
        assert not np.array_equal(a, c)     # another config draws other numbers


def test_gaussian_tables_have_the_stated_spread():
    T = wl.make_table(wl.F32, 4096, 256, 0.02, cid=11, threads=2)
    assert T.dtype == np.float32 and T.shape == (4096, 256)
    assert abs(float(T.mean())) < 2e-4
    assert abs(float(T.std()) / 0.02 - 1.0) < 0.01


def test_16bit_tables_are_the_f32_draw_rounded():
    f32 = wl.make_table(wl.F32, 1000, 96, 0.02, cid=12, threads=1)
    f16 = wl.make_table(wl.F16, 1000, 96, 0.02, cid=12, threads=1)
    bf16 = wl.make_table(wl.BF16, 1000, 96, 0.02, cid=12, threads=1)
    assert np.array_equal(f16, f32.astype(np.float16).view(np.uint16))
    # bfloat16 rounding (nearest, ties to even) as torch converts it
    ref = torch.from_numpy(f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bf16, ref)


def test_bf16_rounding_ties_to_even():
    # 1 + 2^-8 lies halfway between two bf16 neighbours: rounds to the even one
    x = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8)], np.float32)
    assert wl.f32_to_bf16_bits(x).tolist() == [0x3F80, 0x3F82, 0xBF80]


def test_q8_0_blocks_scale_first_codes_in_range():
    V, H = 500, 128
    T = wl.make_table(wl.Q8_0, V, H, cid=13, q8_d_std=0.002, threads=1)
    assert T.dtype == np.uint8 and T.shape == (V, H // 32 * 34)
    blk = T.reshape(V, H // 32, 34)
    d = blk[:, :, 0:2].copy().view(np.float16).astype(np.float64)
    q = blk[:, :, 2:].view(np.int8).astype(np.int64)
    assert np.all(d >= 0.0) and 0.001 < float(d.mean()) < 0.002   # E|N(0, 0.002)| = 0.0016
    assert q.min() == -127 and q.max() == 127                       # never -128
    with pytest.raises(ValueError):
        wl.make_table(wl.Q8_0, 10, 48)


def test_zipf_ids_follow_the_rank_law():
    n, V = 400_000, 50_000
    ids = wl.zipf_ids(21, n, V, s=1.1)
    assert ids.dtype == np.int32 and ids.min() >= 0 and ids.max() < V
    cnt = np.sort(np.bincount(ids, minlength=V))[::-1].astype(np.float64)
    # frequency of rank r ~ r^-1.1: ranks 1 and 2 differ by 2^1.1, ranks 1 and 10 by 10^1.1
    assert abs(cnt[0] / cnt[1] / 2 ** 1.1 - 1.0) < 0.05
    assert abs(cnt[0] / cnt[9] / 10 ** 1.1 - 1.0) < 0.1
    assert np.array_equal(ids, wl.zipf_ids(21, n, V, s=1.1))


def test_session_ids_touch_few_rows():
    w = wl.WORKLOADS["qwen05b"]
    ids = wl.ids_for(w)
    assert ids.size == 628 and ids.min() >= 0 and ids.max() < w.vocab
    assert np.unique(ids).size <= 109


def test_residual_rows_scaled_within_the_range():
    x = wl.residuals(31, 64, 4096, (0.5, 8.0), wl.F32)
    sd = x.std(axis=1)
    assert sd.min() > 0.5 * 0.95 and sd.max() < 8.0 * 1.05
    assert sd.max() / sd.min() > 4.0              # the rows really differ
    xb = wl.residuals(31, 64, 4096, (0.5, 8.0), wl.BF16)
    assert np.array_equal(xb, wl.f32_to_bf16_bits(x))
    one = wl.residuals(32, 4, 8192, None, wl.F32)
    assert abs(float(one.std()) - 1.0) < 0.02


def test_workload_sizes_match_the_stated_tables():
    w = wl.WORKLOADS
    assert w["qwen05b"].table_bytes == 151936 * 896 * 2
    assert w["gemma_q8"].row_bytes == 768 // 32 * 34
    assert w["gemma31b"].table_bytes == 262144 * 5376 * 2
    assert w["batched"].table_bytes == 262144 * 5120 * 2
    assert w["tiny"].table_bytes == 8192 * 256 * 4
    assert w["gemma_q8"].embed_scale == np.float32(np.sqrt(768.0))
