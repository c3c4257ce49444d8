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


def _resid(seed, B, H, dtype):
    r = wl.residuals(seed, B, H, (0.5, 8.0), dtype)
    t = _dev(r)
    return t.view(torch.bfloat16) if dtype == wl.BF16 else t


def test_noalloc_matches_workspace_call_three_in_a_row():
    # The same kernels on the same inputs: the results must be identical to
    # the workspace call's, bit for bit, whatever the array held before.
    cases = [
        # call 1: tensor-core GEMV (bf16 table), 3 residuals, k 12
        (wl.BF16, 20000, 512, 3, 12, 1.0, 31, wl.F32),
        # call 2: CUDA-core GEMV (f32 table), 8 residuals, k 40, other inputs
        (wl.F32, 9000, 256, 8, 40, 0.8, 32, wl.F32),
        # call 3: tcgen05 GEMM (bf16 table, 16 bf16 residuals), k 8, a vocab
        # of two tiles per cluster or more: the first-tile sample, its bounds
        # and the arrival counters live in the array too
        (wl.BF16, 40000, 256, 16, 8, 1.3, 33, wl.BF16),
    ]
    for dtype, V, H, B, k, T, seed, rdt in cases:
        table_np = wl.make_table(dtype, V, H, 0.02, cid=seed, threads=4)
        table = lhs.lhs_table_init(_dev(table_np), V, H, dtype)
        resid = _resid(seed, B, H, rdt)
        assert lhs.lhs_logits_topk_workspace(table, B, k, lhs.LHS_F32 if rdt == wl.F32 else lhs.LHS_BF16) \
            <= lhs.LHS_NOALLOC_SCRATCH_BYTES
        ref_ids, ref_logits, ref_probs, ref_err = lhs.lhs_logits_topk(table, resid, k, T)
        ids, logits, probs, err = _noalloc(table, resid, k, T)
        torch.cuda.synchronize()
        assert int(err.item()) == int(ref_err.item()) == 0
        assert torch.equal(ids, ref_ids)
        assert torch.equal(logits, ref_logits)
        assert torch.equal(probs, ref_probs)


@pytest.mark.parametrize("case", ["gemv", "gemm_full_batch"])
def test_noalloc_rejects_requests_beyond_its_scratch(case):
    if case == "gemv":
        V, H, B, k, rdt = 262144, 64, 64, 128, lhs.LHS_F32   # partial lists alone > 4 MiB
    else:
        V, H, B, k, rdt = 100000, 64, 256, 8, lhs.LHS_BF16   # candidate buffers of 256 residuals > 4 MiB
    table = lhs.lhs_table_init(torch.zeros((V, H), dtype=torch.bfloat16, device="cuda"), V, H,
                               lhs.LHS_BF16)
    need = lhs.lhs_logits_topk_workspace(table, B, k, rdt)
    assert need > lhs.LHS_NOALLOC_SCRATCH_BYTES
    tdt = torch.float32 if rdt == lhs.LHS_F32 else torch.bfloat16
    resid = torch.zeros((B, H), dtype=tdt, device="cuda")
    # sentinels: a rejected call enqueues nothing, so none of them may change
    out = torch.full((B, k), -7, dtype=torch.int32, device="cuda")
    vals = torch.full((B, k), -7.0, dtype=torch.float32, device="cuda")
    probs = torch.full((B, k), -7.0, dtype=torch.float32, device="cuda")
    err = torch.full((1,), 0x3C, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    rc = lhs.lib().lhs_logits_topk_noalloc(
        ctypes.byref(table.c), resid.data_ptr(), rdt, B, k, ctypes.c_float(1.0),
        out.data_ptr(), vals.data_ptr(), probs.data_ptr(), err.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == lhs.LHS_ERR_BUFFER_TOO_SMALL
    assert torch.all(out == -7) and torch.all(vals == -7.0) and torch.all(probs == -7.0)
    assert int(err.item()) == 0x3C
