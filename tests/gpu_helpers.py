"""Comparison helpers for the GPU parity tests (CUDA library vs the CPU oracle).

Bars, from the head's definition:
  * x (the BF16 output of the input stage) is the BF16 rounding of eh_proj . concat with FP32
    accumulation (the source's gemv). It must be the BF16 rounding of some value within the
    kernel's accumulation band E of the exact (fp64) sum s, i.e. lie between the roundings of
    s - E and s + E; E is derived below from each kernel's order of FP32 additions. An x equal
    to the oracle's correctly rounded value always passes.
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


# The batched input stage (B >= 2) sums runs of 128 products per output on tensor cores in FP32
# (eight chained MMAs of 16 exact products; each with at most two roundings of at most 2^-23 of
# the run's sum of |products| so far, so a run total is within 18 * 2^-23 < 2^-18 of that run's
# sum of |products|) and adds the run totals as double-floats before one rounding to BF16. x may
# therefore take another BF16 value where the exact sum lies within
# 2^-18 * sum_k |eh_proj[h, k] * concat[k]| of a rounding midpoint.
BATCHED_X_BAND = 2.0 ** -18


def single_x_band(H: int) -> float:
    """Band of the single-sequence input stage (E / sum_k |eh_proj[h, k] * concat[k]|). Each lane
    keeps eight FP32 accumulators per sequence and adds one exact product (BF16 x BF16 is exact in
    fp32) to each per 16-byte vector of a row; a lane takes at most ceil(vectors / 32) vectors of
    each 8 KB chunk, so an accumulator adds n <= ceil(H / 128) + ceil(4H / 8192) products. The
    first add is exact and each later one rounds by at most 2^-24 of the running sum, so an
    accumulator is within (n - 1) * 2^-24 * (its sum of |products|) of its exact sum (first order;
    the factor 1 + 2^-10 covers the rest for n < 2^13). The 256 accumulator values of a row are
    added as double-floats (relative error ~2^-44, inside check_x's 2^-30 |s|)."""
    n = -(-H // 128) + -(-4 * H // 8192)
    return max(n - 1, 0) * 2.0 ** -24 * (1.0 + 2.0 ** -10)


def x_band(H: int, B: int) -> float:
    """The accumulation band of x from mtp_head_input_batched (no workspace) for B sequences:
    the single-sequence kernel at B = 1; the tensor-core kernel (or, for shapes it does not take,
    the CUDA-core kernels) at B >= 2."""
    single = single_x_band(H)
    return single if B == 1 else max(BATCHED_X_BAND, single)


def context_band(K: int) -> float:
    """Relative band (times sum_k |p_k|) of an FP32 accumulation of K exact BF16 products on the
    tcgen05 tensor cores (the context-row GEMM): the MMAs add K / 16 groups of 16 exact products
    into FP32 accumulators, and each of those additions (with whatever internal alignment the
    hardware uses inside a group) is taken to err by at most 2^-22 of the sum of |products|
    accumulated so far. When the product is split along k, the at most 15 FP32 additions of the
    split partial sums (round to nearest, each within 2^-24 of a value bounded by the sum of
    |products|) fit in the extra 16 * 2^-22."""
    return (K / 16 + 16) * 2.0 ** -22


def step_x_band(H: int, B: int) -> float:
    """The band of x from the whole-step entry points with a workspace of the full
    mtp_head_workspace_bytes: 2..16 sequences at H % 32 == 0 take the context-row GEMM, the rest
    the kernels of mtp_head_input_batched."""
    return context_band(2 * H) if B >= 2 and H % 32 == 0 else x_band(H, B)


def abs_product_sums(eh_proj_bits: np.ndarray, concat_bits: np.ndarray) -> np.ndarray:
    """sum_k |eh_proj[h, k]| * |concat[b, k]| for every (b, h), fp64 ([B, H])."""
    H, K = eh_proj_bits.shape
    c = np.abs(oracle.bf16_to_f64(concat_bits)).reshape(-1, K)
    out = np.empty((c.shape[0], H), np.float64)
    for h0 in range(0, H, 1024):  # row blocks keep the fp64 copy of eh_proj small
        W = np.abs(oracle.bf16_to_f64(eh_proj_bits[h0:h0 + 1024]))
        out[:, h0:h0 + W.shape[0]] = c @ W.T
    return out


def check_x(x_gpu: np.ndarray, x_ref: np.ndarray, sums: np.ndarray, abs_sums: np.ndarray | None = None,
            band: float = BATCHED_X_BAND) -> int:
    """x must be the BF16 rounding of a value within E of the exact (fp64) sum s, i.e. lie
    between the BF16 roundings of s - E and s + E. E = max(2^-30 |s|, band * abs_sums) (without
    abs_sums only the two neighbours of a rounding midpoint are accepted). Returns the number of
    elements that differ from the oracle's correctly rounded x."""
    x_gpu = x_gpu.reshape(x_ref.shape)
    diff = np.nonzero(x_gpu != x_ref)
    if len(diff[0]) == 0:
        return 0
    g = oracle.bf16_to_f64(x_gpu[diff])
    s = sums[diff]
    E = np.abs(s) * 2.0 ** -30
    if abs_sums is not None:
        E = np.maximum(E, band * abs_sums[diff])
    lo = oracle.bf16_to_f64(oracle.f64_to_bf16(s - E))
    hi = oracle.bf16_to_f64(oracle.f64_to_bf16(s + E))
    bad = ~((lo <= g) & (g <= hi))
    if bad.any():
        k = int(np.nonzero(bad)[0][0])
        idx = tuple(int(d[k]) for d in diff)
        r = oracle.bf16_to_f64(np.array([x_ref[idx]], np.uint16))[0]
        raise AssertionError(f"x mismatch at {idx}: gpu {g[k]!r} oracle {r!r} (fp64 sum {s[k]!r}, band {E[k]!r}); "
                             f"{int(bad.sum())} of {len(g)} differing elements outside the band")
    return len(g)


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
