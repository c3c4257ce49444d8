"""The allocation-free top-k entry point, lhs_logits_topk_noalloc.

It exists for callers that cannot allocate device memory where they need
top-k tokens (an application that owns the whole device memory budget, a
latency-critical loop that must not synchronise on cudaMalloc); its scratch
is a fixed array inside the library.  These tests call it through the C-ABI
and check it against the workspace entry point, lhs_logits_topk, on two
calls in a row with different inputs, so stale scratch contents from the
first call would show in the second.  This file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import embedding_lookup_tied_gb300 as lhs
import workloads as wl

pytestmark = pytest.mark.gpu

PROB_RTOL = 1e-5


def _dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def _noalloc(table, resid, k, temperature):
    """Direct C-ABI call of lhs_logits_topk_noalloc."""
    B = resid.shape[0]
    rd = lhs.LHS_F32 if resid.dtype == torch.float32 else lhs.LHS_BF16
    ids = torch.full((B, k), -7, dtype=torch.int32, device="cuda")
    logits = torch.full((B, k), -7.0, dtype=torch.float32, device="cuda")
    probs = torch.full((B, k), -7.0, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lhs.lib().lhs_logits_topk_noalloc(
        ctypes.byref(table.c), resid.data_ptr(), rd, B, k, ctypes.c_float(temperature),
        ids.data_ptr(), logits.data_ptr(), probs.data_ptr(), err.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert rc == lhs.LHS_OK, rc
    return ids, logits, probs, err


def test_noalloc_matches_workspace_call_twice_in_a_row():
    cases = [
        # call 1: tensor-core path (bf16 table), 3 residuals, k 12
        (wl.BF16, 20000, 512, 3, 12, 1.0, 31),
        # call 2: CUDA-core path (f32 table), 8 residuals, k 40, other inputs
        (wl.F32, 9000, 256, 8, 40, 0.8, 32),
    ]
    for dtype, V, H, B, k, T, seed in cases:
        table_np = wl.make_table(dtype, V, H, 0.02, cid=seed, threads=4)
        table = lhs.lhs_table_init(_dev(table_np), V, H, dtype)
        resid = _dev(wl.residuals(seed, B, H, (0.5, 8.0)))
        ref_ids, ref_logits, ref_probs, ref_err = lhs.lhs_logits_topk(table, resid, k, T)
        ids, logits, probs, err = _noalloc(table, resid, k, T)
        torch.cuda.synchronize()
        assert int(err.item()) == int(ref_err.item()) == 0
        assert torch.equal(ids, ref_ids)
        assert torch.equal(logits, ref_logits)
        rp = ref_probs.double()
        assert torch.all((probs.double() - rp).abs() <= PROB_RTOL * rp)


def test_noalloc_rejects_requests_beyond_its_scratch():
    V, H = 262144, 64
    table = lhs.lhs_table_init(torch.zeros((V, H), dtype=torch.bfloat16, device="cuda"), V, H,
                               lhs.LHS_BF16)
    B, k = 64, 128            # partial lists alone: SMs x 64 x 128 x 8 bytes > 4 MiB
    need = lhs.lhs_logits_topk_workspace(table, B, k, lhs.LHS_F32)
    assert need > lhs.LHS_NOALLOC_SCRATCH_BYTES
    resid = torch.zeros((B, H), dtype=torch.float32, device="cuda")
    out = torch.empty((B, k), dtype=torch.int32, device="cuda")
    vals = torch.empty((B, k), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lhs.lib().lhs_logits_topk_noalloc(
        ctypes.byref(table.c), resid.data_ptr(), lhs.LHS_F32, B, k, ctypes.c_float(1.0),
        out.data_ptr(), vals.data_ptr(), None, err.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert rc == lhs.LHS_ERR_BUFFER_TOO_SMALL
