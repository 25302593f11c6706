"""Comparison helpers for the GPU parity tests (CUDA library vs the CPU oracle).

Bars, from the head's definition:
  * x (the BF16 output of the input stage) must equal the oracle's BF16 rounding of the exact
    sum; the only tolerated difference is the neighbouring BF16 value when the oracle's fp64
    sum lies within 2^-30 (relative) of the rounding midpoint, where both roundings are valid.
  * logits: max |GPU - oracle| <= 2e-2 for the BF16 head, <= 6e-2 for the FP8 head (oracle on
    the dequantised weights).
  * draft: the lowest-index argmax of the GPU's own FP32 logits (exact self-consistency);
    identical to the oracle's draft when the oracle's top-2 gap exceeds the tolerance, else
    an id whose oracle logit is within the tolerance of the oracle's maximum.
"""
from __future__ import annotations

import numpy as np

import oracle

TOL_BF16 = 2e-2
TOL_FP8 = 6e-2


def check_x(x_gpu: np.ndarray, x_ref: np.ndarray, sums: np.ndarray) -> int:
    """Returns the number of accepted midpoint-ambiguous elements (normally 0)."""
    x_gpu = x_gpu.reshape(x_ref.shape)
    diff = np.nonzero(x_gpu != x_ref)
    n_ok = 0
    for idx in zip(*diff):
        g = oracle.bf16_to_f64(np.array([x_gpu[idx]], np.uint16))[0]
        r = oracle.bf16_to_f64(np.array([x_ref[idx]], np.uint16))[0]
        s = sums[idx]
        mid = (g + r) / 2
        adjacent = abs(int(x_gpu[idx]) - int(x_ref[idx])) == 1 and np.sign(g) == np.sign(r)
        near = abs(s - mid) <= abs(mid) * 2.0 ** -30
        assert adjacent and near, (
            f"x mismatch at {idx}: gpu {g!r} oracle {r!r} (fp64 sum {s!r})")
        n_ok += 1
    return n_ok


def lowest_argmax(v: np.ndarray) -> int:
    """Lowest index of the maximum, NaN never wins, -1 if all NaN."""
    ok = ~np.isnan(v)
    if not ok.any():
        return -1
    m = np.max(v[ok])
    return int(np.nonzero(ok & (v == m))[0][0])


def check_logits_and_draft(logits_gpu: np.ndarray, draft_gpu: np.ndarray, ref_logits: np.ndarray,
                           tol: float) -> float:
    """Check every sequence; returns the max abs logit error."""
    lg = logits_gpu.reshape(ref_logits.shape).astype(np.float64)
    draft_gpu = np.asarray(draft_gpu).reshape(-1)
    err = float(np.max(np.abs(lg - ref_logits))) if lg.size else 0.0
    assert err <= tol, f"max |logit error| {err} > {tol}"
    for b in range(ref_logits.shape[0]):
        check_draft(int(draft_gpu[b]), lg[b], ref_logits[b], tol)
    return err


def check_draft(draft: int, logits_gpu_row, ref_row: np.ndarray, tol: float) -> None:
    if logits_gpu_row is not None:
        assert draft == lowest_argmax(np.asarray(logits_gpu_row, np.float64)), \
            "draft is not the lowest-index argmax of the returned logits"
    ref_draft = oracle.argmax(ref_row)
    order = np.sort(ref_row[~np.isnan(ref_row)])
    gap = order[-1] - order[-2] if order.size > 1 else np.inf
    if gap > tol:
        assert draft == ref_draft, f"draft {draft} != oracle draft {ref_draft} (top-2 gap {gap})"
    else:
        assert 0 <= draft < ref_row.size and ref_row[draft] >= order[-1] - tol, \
            f"draft {draft} has oracle logit {ref_row[draft]} < max {order[-1]} - {tol}"
