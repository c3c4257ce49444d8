"""Chains of library calls on one stream, each consuming what the previous
call wrote.  Every kernel is launched as a programmatic dependent: it may
start before its predecessor finishes and must not read the predecessor's
output before its wait.  Each case refills the consumed buffer with junk
(0xFF bytes) before the chain, so a read that slipped ahead of the wait
shows as a wrong result or a spurious error bit.  The chains run many times
because the race, when there is one, depends on timing.
"""
import numpy as np
import pytest
import torch

import embedding_lookup_tied_gb300 as lhs
import oracle as orc
import workloads as wl
from gpu_util import to_dev, upload_table

pytestmark = pytest.mark.gpu

REPS = 200


def _table(dtype, V, H, cid):
    T = wl.make_table(dtype, V, H, 0.02, cid=cid, threads=8)
    return T, upload_table(T, dtype, V, H)


def test_lm_head_then_encode_then_decode():
    # the decode reads the header and payload the encode has just written
    V, H = 151936, 896
    _, tab = _table(orc.BF16, V, H, 40)
    x = to_dev(wl.residuals(41, 1, H))
    ref_buf, _ = orc.wire_encode(orc.WIRE_F16, x.cpu().numpy())
    ref_y, _ = orc.wire_decode(orc.WIRE_F16, ref_buf, 1, H)
    nb = lhs.lhs_wire_bytes(orc.WIRE_F16, 1, H)
    buf = torch.empty(nb, dtype=torch.uint8, device="cuda")
    y = torch.empty((1, H), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(lhs.lhs_logits_topk_workspace(tab, 1, 10, lhs.LHS_F32), dtype=torch.uint8,
                     device="cuda")
    bad = 0
    for _ in range(REPS):
        buf.fill_(0xFF)
        y.fill_(float("nan"))
        err.zero_()
        torch.cuda.synchronize()
        lhs.lhs_logits_topk(tab, x, 10, ws=ws, err=err)
        lhs.lhs_wire_encode(orc.WIRE_F16, x, 0, 0, 10, buf=buf, err=err)
        lhs.lhs_wire_decode(orc.WIRE_F16, buf, 1, H, out=y, err=err)
        torch.cuda.synchronize()
        bad += int(err.item()) != 0 or not np.array_equal(y.cpu().numpy(), ref_y)
    assert bad == 0


@pytest.mark.parametrize("fmt", [orc.WIRE_F16, orc.WIRE_I8])
def test_decode_then_lm_head(fmt):
    # the lm_head projects the residuals the decode has just written
    V, H, B, k = 20000, 1024, 4, 8
    T, tab = _table(orc.F16, V, H, 42)
    x = wl.residuals(43, B, H, (0.5, 8.0))
    buf_h, _ = orc.wire_encode(fmt, x)
    xh, _ = orc.wire_decode(fmt, buf_h, B, H)
    buf = to_dev(buf_h)
    ref_ids, ref_vals, _, e = lhs.lhs_logits_topk(tab, to_dev(xh), k)
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    y = torch.empty((B, H), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ids = torch.empty((B, k), dtype=torch.int32, device="cuda")
    vals = torch.empty((B, k), dtype=torch.float32, device="cuda")
    ws = torch.empty(lhs.lhs_logits_topk_workspace(tab, B, k, lhs.LHS_F32), dtype=torch.uint8,
                     device="cuda")
    bad = 0
    for _ in range(REPS):
        y.fill_(float("nan"))
        err.zero_()
        torch.cuda.synchronize()
        lhs.lhs_wire_decode(fmt, buf, B, H, out=y, err=err)
        lhs.lhs_logits_topk(tab, y, k, ws=ws, ids=ids, logits=vals, err=err, want_probs=False)
        torch.cuda.synchronize()
        bad += (int(err.item()) != 0 or not torch.equal(ids, ref_ids)
                or not torch.equal(vals, ref_vals))
    assert bad == 0


def test_unique_ids_then_embed():
    # the gather reads the distinct ids the dedup has just written
    V, H, n = 50000, 256, 4096
    T, tab = _table(orc.BF16, V, H, 44)
    ids = wl.zipf_ids(45, n, V)
    ru, _, _ = orc.unique_ids(ids, V)
    ref, _ = orc.embed(T, orc.BF16, V, H, ru, 16.0)
    d_ids = to_dev(ids)
    uniq = torch.empty(n, dtype=torch.int32, device="cuda")
    inv = torch.empty(n, dtype=torch.int32, device="cuda")
    cnt = torch.empty(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(lhs.lib().lhs_unique_ids_workspace(V), dtype=torch.uint8, device="cuda")
    out = torch.empty((ru.size, H), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad = 0
    for _ in range(REPS // 2):
        uniq.fill_(-1)
        err.zero_()
        torch.cuda.synchronize()
        lhs.lhs_unique_ids(d_ids, V, ws=ws, err=err, unique=uniq, inverse=inv, count=cnt)
        lhs.lhs_embed(tab, uniq[:ru.size], 16.0, out=out, err=err)
        torch.cuda.synchronize()
        bad += int(err.item()) != 0 or not np.array_equal(out.cpu().numpy(), ref)
    assert bad == 0
