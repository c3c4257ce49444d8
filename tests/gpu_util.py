"""Helpers for the GPU parity tests: upload seeded inputs, read results back,
and the lm_head tolerance rules."""
import numpy as np
import torch

import embedding_lookup_tied_gb300 as lhs
import oracle as orc

# Logit tolerance: |L_gpu - L_ref| <= RTOL[dtype] * sum_j |T[v][j] x[b][j]|
# (the standard bound for a dot product computed in another order / precision).
RTOL = {orc.F32: 1e-5, orc.F16: 1e-3, orc.BF16: 1e-3, orc.Q8_0: 1e-5}
# Probabilities are checked against the oracle applied to the GPU's own logits.
PROB_RTOL = 1e-5


def to_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(a).to(device)


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def same_f32(got: np.ndarray, ref: np.ndarray) -> bool:
    """Bit-identical binary32 arrays, except that a NaN matches any NaN: the
    payload a NaN carries through arithmetic or widening differs between the
    GPU (canonical 0x7FFFFFFF) and the host CPU (quieted input NaN)."""
    got = np.ascontiguousarray(got, np.float32)
    ref = np.ascontiguousarray(ref, np.float32)
    if got.shape != ref.shape:
        return False
    gn, rn = np.isnan(got), np.isnan(ref)
    if not np.array_equal(gn, rn):
        return False
    return bool(np.array_equal(got.view(np.uint32)[~gn], ref.view(np.uint32)[~rn]))


def upload_table(table_np: np.ndarray, dtype: int, vocab: int, hidden: int):
    t = to_dev(table_np)
    return lhs.lhs_table_init(t, vocab, hidden, dtype)


def guarded(shape, dtype, device="cuda", fill=0x5A):
    """A tensor with canary bytes before and after it (compute-sanitizer is not
    available: out-of-bounds writes show up as damaged canaries)."""
    n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
    pad = 256
    raw = torch.full((n + 2 * pad,), fill, dtype=torch.uint8, device=device)
    view = raw[pad:pad + n].view(dtype).view(shape)
    return raw, view, pad


def canaries_intact(raw: torch.Tensor, pad: int, fill=0x5A) -> bool:
    r = raw.cpu().numpy()
    return bool(np.all(r[:pad] == fill) and np.all(r[-pad:] == fill))


def resid_values(resid_np: np.ndarray, resid_dtype: int) -> np.ndarray:
    """Residual values as float32 for the oracle (bf16 decoded by the oracle)."""
    if resid_dtype == orc.F32:
        return resid_np.astype(np.float32)
    return orc.bf16_to_f32(resid_np)


def check_topk_against_fp64(ids, vals, L64, S64, k, rtol):
    """Acceptance rule against binary64 logits: every returned logit is within
    tolerance of the binary64 logit of its id, and no omitted id beats the
    weakest returned one by more than the tolerance (ties inside the
    tolerance are accepted)."""
    ids = np.asarray(ids)
    assert len(set(ids.tolist())) == k, "duplicate ids"
    tol = rtol * S64
    assert np.all(np.abs(vals.astype(np.float64) - L64[ids]) <= tol[ids] + 1e-30)
    weakest = ids[np.argmin(L64[ids])]
    mask = np.ones(L64.size, bool)
    mask[ids] = False
    excess = L64[mask] - L64[weakest]
    assert np.all(excess <= tol[mask] + tol[weakest] + 1e-30), \
        f"omitted id beats returned: {excess.max()}"
