"""Pins for the CPU oracle: each test ties a part of the oracle to something other than the
oracle itself -- the hand-computed worked example, closed forms, invariants, library
conversions (torch's bfloat16 / float8_e4m3fn casts), numpy float64 matmuls and brute force.
A plausible slip (a dropped term, a swapped half of the concat, a wrong row, the 1+w norm, a
transposed projection, a wrong tie rule, a wrong E4M3 bias) fails at least one of them.
No GPU is needed.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle


def bf(values) -> np.ndarray:
    """BF16 bit patterns of values that are exactly representable (or rounded RNE by torch)."""
    t = torch.tensor(np.asarray(values, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def f64(bits) -> np.ndarray:
    return oracle.bf16_to_f64(bits)


@pytest.fixture(scope="module")
def ex(golden_dir):
    with open(os.path.join(golden_dir, "worked_example_4x8.json")) as f:
        return json.load(f)


def _example_weights(ex, hnorm_w=None):
    return dict(embed=bf(ex["embed"]), enorm_w=bf(ex["enorm_w"]),
                hnorm_w=bf(hnorm_w if hnorm_w is not None else ex["hnorm_w"]),
                eh_proj=bf(ex["eh_proj"]), final_norm_w=bf(ex["final_norm_w"]),
                lm_head=bf(ex["lm_head"]))


# --------------------------------------------------------------------------- worked example
def test_worked_example_bf16(ex):
    w = _example_weights(ex)
    x, concat, st = oracle.input_stage(w["embed"], w["enorm_w"], w["hnorm_w"], w["eh_proj"],
                                       [ex["token"]], bf([ex["target_hidden"]]), ex["eps"],
                                       return_concat=True)
    assert st[0] == oracle.OK
    assert f64(concat[0]).tolist() == ex["expected_concat"]
    assert f64(x[0]).tolist() == ex["expected_x"]
    out = oracle.head(w, [ex["token"]], bf([ex["target_hidden"]]), ex["eps"])
    assert f64(out["xhat"][0]).tolist() == ex["expected_xhat"]
    assert out["logits"][0].tolist() == ex["expected_logits"]
    assert int(out["draft"][0]) == ex["expected_draft"]


def test_worked_example_fp8(ex):
    w = _example_weights(ex)
    q, s, st = oracle.quantize(w["lm_head"])
    assert st == oracle.OK
    assert q.tolist() == ex["expected_fp8_codes"]
    assert s[0] == 0.0
    out = oracle.head(w, [ex["token"]], bf([ex["target_hidden"]]), ex["eps"], w_dtype=1,
                      lm_head=q, scale=s)
    np.testing.assert_allclose(out["logits"][0], ex["expected_logits"], rtol=ex["fp8_logit_rel_tol"],
                               atol=1e-12)
    assert out["logits"][0][3] == out["logits"][0][5]  # exact tie survives quantisation
    assert int(out["draft"][0]) == ex["expected_draft"]


def test_worked_example_variant(ex):
    w = _example_weights(ex, hnorm_w=ex["variant_hnorm_w"])
    x, concat, st = oracle.input_stage(w["embed"], w["enorm_w"], w["hnorm_w"], w["eh_proj"],
                                       [ex["token"]], bf([ex["variant_target_hidden"]]), ex["eps"],
                                       return_concat=True)
    assert f64(concat[0]).tolist() == ex["variant_expected_concat"]
    assert f64(x[0]).tolist() == ex["variant_expected_x"]
    out = oracle.head(w, [ex["token"]], bf([ex["variant_target_hidden"]]), ex["eps"])
    assert out["logits"][0].tolist() == ex["expected_logits"]
    assert int(out["draft"][0]) == ex["expected_draft"]


def test_worked_example_wrong_row_changes_result(ex):
    # the gather must read row `token`; a neighbouring row gives a different x
    w = _example_weights(ex)
    x_ok, _ = oracle.input_stage(w["embed"], w["enorm_w"], w["hnorm_w"], w["eh_proj"], [5],
                                 bf([ex["target_hidden"]]), ex["eps"])
    x_4, _ = oracle.input_stage(w["embed"], w["enorm_w"], w["hnorm_w"], w["eh_proj"], [4],
                                bf([ex["target_hidden"]]), ex["eps"])
    assert not np.array_equal(x_ok, x_4)


# --------------------------------------------------------------------------- BF16 codec
def test_bf16_decode_all_patterns_match_torch():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.bf16_to_f64(pats)
    ref = torch.from_numpy(pats.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_bf16_encode_matches_torch_on_fp32_inputs():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * np.float32(10.0) ** rng.integers(-30, 30, 200000).astype(np.float32),
        # every midpoint between neighbouring positive BF16 values of exponent -20..20
        (f64(np.arange(0x3580, 0x4B00, dtype=np.uint16)) * (1 + 2.0 ** -8)).astype(np.float32),
        np.array([0.0, -0.0, 1e-45, -1e-45, 3.3e38, -3.3e38, 3.4e38], np.float32),
    ]).astype(np.float32)
    ours = oracle.f64_to_bf16(vals.astype(np.float64))
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_encode_single_rounding_from_double():
    # 1 + 2^-8 is the midpoint between 1 and 1 + 2^-7; a hair above it must round up.
    # (Rounding through fp32 first would land on the midpoint and tie to 1.0.)
    assert f64(oracle.f64_to_bf16([1 + 2 ** -8 + 2 ** -30]))[0] == 1 + 2 ** -7
    assert f64(oracle.f64_to_bf16([1 + 2 ** -8]))[0] == 1.0                    # tie -> even
    assert f64(oracle.f64_to_bf16([1 + 3 * 2 ** -8]))[0] == 1 + 2 ** -6        # tie -> even (up)
    assert f64(oracle.f64_to_bf16([-(1 + 2 ** -8 + 2 ** -30)]))[0] == -(1 + 2 ** -7)
    assert oracle.f64_to_bf16([2.0 ** 128])[0] == 0x7F80                      # overflow -> inf
    assert oracle.f64_to_bf16([2.0 ** -134])[0] == 0x0000                     # half of min subnormal -> even (0)
    assert oracle.f64_to_bf16([1.5 * 2.0 ** -133])[0] == 0x0002               # tie -> even


# --------------------------------------------------------------------------- E4M3 codec
def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # values the OCP format fixes: max normal, min normal, min subnormal
    assert ours[0x7E] == 448.0 and ours[0x08] == 2.0 ** -6 and ours[0x01] == 2.0 ** -9


def test_e4m3_encode_roundtrip_and_midpoints():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = oracle.e4m3_to_f64(codes)
    assert np.array_equal(oracle.f64_to_e4m3(vals), codes)
    # midpoints between neighbouring non-negative codes round to the even code
    pos = np.arange(0, 0x7E, dtype=np.uint8)
    lo, hi = oracle.e4m3_to_f64(pos), oracle.e4m3_to_f64(pos + 1)
    mid = (lo + hi) / 2
    got = oracle.f64_to_e4m3(mid)
    even = np.where(pos % 2 == 0, pos, pos + 1)
    assert np.array_equal(got, even)
    # a hair either side of a midpoint goes to the nearer code
    assert np.array_equal(oracle.f64_to_e4m3(mid * (1 - 1e-9)), pos)
    assert np.array_equal(oracle.f64_to_e4m3(mid * (1 + 1e-9)), pos + 1)


def test_e4m3_encode_matches_torch_and_saturates():
    rng = np.random.default_rng(2)
    vals = np.concatenate([
        rng.uniform(-463.9, 463.9, 100000),
        rng.standard_normal(100000) * 2.0 ** rng.integers(-12, 8, 100000),
    ]).astype(np.float32)
    vals = vals[np.abs(vals) < 464.0]  # torch's cast is non-saturating (NaN) from 464 up
    ours = oracle.f64_to_e4m3(vals.astype(np.float64))
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)
    # satfinite: anything at or above 448 (including inf) becomes +-448; NaN stays NaN
    big = np.array([448.0, 464.0, 1e6, np.inf, -500.0, -np.inf])
    assert oracle.f64_to_e4m3(big).tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]
    assert oracle.f64_to_e4m3([np.nan])[0] & 0x7F == 0x7F


# --------------------------------------------------------------------------- RMSNorm
def _rms_case(n, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return bf(rng.standard_normal(n) * scale), bf(1 + 0.1 * rng.standard_normal(n))


def test_rmsnorm_all_ones_weight_gives_unit_rms():
    x, _ = _rms_case(4096, 3)
    out = f64(oracle.rms_norm(x, bf(np.ones(4096)), 1e-6))
    ms = np.mean(f64(x) ** 2)
    want = math.sqrt(ms / (ms + float(np.float32(1e-6))))
    assert abs(math.sqrt(np.mean(out ** 2)) - want) < 2 ** -8


def test_rmsnorm_zero_weight_gives_zero_not_unit():
    # the 1+w form would give a unit-RMS output here
    x, _ = _rms_case(512, 4)
    assert np.all(f64(oracle.rms_norm(x, bf(np.zeros(512)), 1e-6)) == 0.0)


def test_rmsnorm_power_of_two_scaling_invariance():
    x, w = _rms_case(1024, 5)
    base = oracle.rms_norm(x, w, 0.0)
    for j in (-20, -3, 1, 7, 40):
        assert np.array_equal(oracle.rms_norm(bf(f64(x) * 2.0 ** j), w, 0.0), base)


def test_rmsnorm_constant_input_gives_sign_times_weight():
    _, w = _rms_case(256, 6)
    for c in (3.0, -0.75):
        out = oracle.rms_norm(bf(np.full(256, c)), w, 0.0)
        assert np.array_equal(f64(out), np.sign(c) * f64(w))


def test_rmsnorm_matches_closed_form_in_fp64():
    x, w = _rms_case(333, 7, scale=5.0)
    xv, wv = f64(x), f64(w)
    eps = float(np.float32(1e-6))
    want = xv * wv / np.sqrt(np.mean(xv ** 2) + eps)
    got = f64(oracle.rms_norm(x, w, 1e-6))
    # one BF16 rounding of the exact value: within half an ulp (2^-9 relative)
    assert np.all(np.abs(got - want) <= np.abs(want) * 2.0 ** -8 + 1e-30)


# --------------------------------------------------------------------------- input stage
def _small_weights(H, V, seed):
    rng = np.random.default_rng(seed)
    return dict(embed=bf(0.02 * rng.standard_normal((V, H))),
                enorm_w=bf(1 + 0.1 * rng.standard_normal(H)),
                hnorm_w=bf(1 + 0.1 * rng.standard_normal(H)),
                eh_proj=bf(0.02 * rng.standard_normal((H, 2 * H))),
                final_norm_w=bf(1 + 0.1 * rng.standard_normal(H)),
                lm_head=bf(0.02 * rng.standard_normal((V, H))))


def test_input_stage_gemv_matches_numpy_fp64():
    H, V = 96, 50
    w = _small_weights(H, V, 8)
    rng = np.random.default_rng(9)
    hid = bf(rng.standard_normal((3, H)))
    toks = [0, 17, V - 1]
    x, concat, st = oracle.input_stage(w["embed"], w["enorm_w"], w["hnorm_w"], w["eh_proj"], toks,
                                       hid, 1e-6, return_concat=True)
    assert np.all(st == 0)
    ref = f64(w["eh_proj"]) @ f64(concat).T           # [H, B] in numpy's own order
    # one BF16 rounding of (almost) the same fp64 value
    ref_b = torch.from_numpy(ref.T.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    diff = np.abs(f64(x) - ref_b)
    assert np.all(diff <= np.abs(ref_b) * 2.0 ** -7)
    assert np.mean(diff == 0) > 0.99


def test_input_stage_concat_order_and_gather():
    # eh_proj = [I | 0] returns the enorm half, [0 | I] the hnorm half: pins the order
    H, V = 64, 20
    w = _small_weights(H, V, 10)
    hid = bf(np.random.default_rng(11).standard_normal((1, H)))
    eye = np.eye(H)
    left = bf(np.concatenate([eye, 0 * eye], 1))
    right = bf(np.concatenate([0 * eye, eye], 1))
    tok = 13
    xl, _ = oracle.input_stage(w["embed"], w["enorm_w"], w["hnorm_w"], left, [tok], hid, 1e-6)
    xr, _ = oracle.input_stage(w["embed"], w["enorm_w"], w["hnorm_w"], right, [tok], hid, 1e-6)
    assert np.array_equal(xl[0], oracle.rms_norm(w["embed"][tok], w["enorm_w"], 1e-6))
    assert np.array_equal(xr[0], oracle.rms_norm(hid[0], w["hnorm_w"], 1e-6))


def test_input_stage_token_out_of_range_gives_zero_row_and_status():
    H, V = 32, 10
    w = _small_weights(H, V, 12)
    hid = bf(np.ones((3, H)))
    x, st = oracle.input_stage(w["embed"], w["enorm_w"], w["hnorm_w"], w["eh_proj"], [V, -1, 2],
                               hid, 1e-6)
    assert st.tolist() == [oracle.ERR_TOKEN_RANGE, oracle.ERR_TOKEN_RANGE, oracle.OK]
    assert np.all(x[:2] == 0) and np.any(x[2] != 0)


# --------------------------------------------------------------------------- lm_head sweep
def test_logits_bf16_match_numpy_matmul():
    H, V = 80, 300
    w = _small_weights(H, V, 13)
    xh = bf(np.random.default_rng(14).standard_normal((2, H)))
    got = oracle.logits(0, w["lm_head"], None, xh)
    ref = f64(xh) @ f64(w["lm_head"]).T
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
    # row ranges, sampled rows and threading agree exactly with the whole sweep
    assert np.array_equal(oracle.logits(0, w["lm_head"], None, xh, 100, 200), got[:, 100:200])
    assert np.array_equal(oracle.logits(0, w["lm_head"], None, xh, threads=4), got)
    assert np.array_equal(oracle.logits_rows(0, w["lm_head"], None, xh[1], [7, 299, 0]),
                          got[1, [7, 299, 0]])


def test_logits_fp8_use_dequantised_weights():
    H, V = 64, 200
    w = _small_weights(H, V, 15)
    q, s, st = oracle.quantize(w["lm_head"])
    assert st == 0
    xh = bf(np.random.default_rng(16).standard_normal(H))
    deq = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64).numpy() * s.astype(np.float64)[:, None]
    ref = deq @ f64(xh)
    np.testing.assert_allclose(oracle.logits(1, q, s, xh), ref, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- argmax
def _brute_argmax(v):
    best = -1
    for i, a in enumerate(v):
        if a != a:
            continue
        if best < 0 or a > v[best]:
            best = i
    return best


@pytest.mark.parametrize("vals,want", [
    ([1.0, 3.0, 3.0, 2.0], 1),
    ([5.0, 5.0, 5.0], 0),
    ([0.0, 1.0, 2.0, 2.0], 2),
    ([-np.inf, -np.inf], 0),
    ([np.nan, -np.inf, np.nan], 1),
    ([np.nan, np.nan], -1),
    ([np.nan, 2.0, np.inf, np.inf], 2),
    ([-0.0, 0.0], 0),
    ([], -1),
])
def test_argmax_special_cases(vals, want):
    assert oracle.argmax(np.array(vals, np.float64)) == want


def test_argmax_brute_force_small_integers():
    rng = np.random.default_rng(17)
    for _ in range(300):
        v = rng.integers(-3, 4, rng.integers(1, 12)).astype(np.float64)
        v[rng.random(v.size) < 0.1] = np.nan
        assert oracle.argmax(v) == _brute_argmax(v.tolist())


# --------------------------------------------------------------------------- quantiser
def _torch_quantise(W_bits):
    """The quantiser reading written with torch's own ops: fp32 absmax/448, fp32 division,
    torch's RNE float8_e4m3fn cast (valid: every quotient is below 464)."""
    w = torch.from_numpy(W_bits.view(np.int16)).view(torch.bfloat16).float()
    s = w.abs().amax(1) / 448.0
    q = torch.where(s[:, None] == 0, torch.zeros_like(w), w / s[:, None])
    return q.to(torch.float8_e4m3fn).view(torch.uint8).numpy(), s.numpy()


def test_quantiser_matches_torch_on_random_rows_with_outliers():
    rng = np.random.default_rng(18)
    W = 0.02 * rng.standard_normal((64, 1024))
    W[rng.random(W.shape) < 0.01] *= 50
    W[3] = 0.0
    W[4, ::2] = -0.0
    W[5] = 0.0
    W[5, 17] = 1e-39          # a BF16 subnormal as the row maximum
    W[6] *= 1e-30
    Wb = bf(W)
    q, s, st = oracle.quantize(Wb)
    q_ref, s_ref = _torch_quantise(Wb)
    assert st == 0
    assert np.array_equal(s.view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(q, q_ref)
    assert s[3] == 0 and np.all(q[3] == 0)
    # every nonzero row uses the full range: its absmax maps to +-448
    dec = oracle.e4m3_to_f64(q)
    nz = s > 0
    assert np.all(np.abs(dec[nz]).max(1) == 448.0)


def test_quantiser_exhaustive_bf16_patterns():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite = pats[(pats & 0x7F80) != 0x7F80]
    rng = np.random.default_rng(19)
    rows = []
    for top in (0x3F80, 0x0001, 0x0080, 0x2000, 0x4300, 0x7F7F):  # row maxima across the range
        r = rng.permutation(finite)
        r = r[(r & 0x7FFF) <= top][:4096]
        r[0] = top
        rows.append(np.resize(r, 4096))
    Wb = np.stack(rows).astype(np.uint16)
    q, s, st = oracle.quantize(Wb)
    q_ref, s_ref = _torch_quantise(Wb)
    assert st == 0
    assert np.array_equal(s.view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(q, q_ref)


def test_quantiser_rejects_nonfinite():
    for bad in (np.nan, np.inf, -np.inf):
        W = np.zeros((2, 16), np.float32)
        W[1, 5] = bad
        q, s, st = oracle.quantize(bf(W))
        assert st == oracle.ERR_NONFINITE


def test_quantiser_error_bound():
    # each dequantised weight is within half an E4M3 spacing of the weight (relative 2^-4 for
    # normals) -- the closed-form bound of round-to-nearest with 3 mantissa bits
    rng = np.random.default_rng(20)
    Wb = bf(0.02 * rng.standard_normal((32, 512)))
    q, s, _ = oracle.quantize(Wb)
    deq = oracle.dequantize(q, s)
    w = f64(Wb)
    sub = np.abs(w) < (2.0 ** -6) * s[:, None]
    err = np.abs(deq - w)
    assert np.all(err[~sub] <= np.abs(w[~sub]) * 2.0 ** -4 * (1 + 1e-6))
    assert np.all(err[sub] <= (2.0 ** -10) * s[:, None].repeat(512, 1)[sub] * (1 + 1e-6))


# --------------------------------------------------------------------------- whole head
def test_head_is_composition_and_draft_is_lowest_max():
    H, V = 64, 500
    w = _small_weights(H, V, 21)
    rng = np.random.default_rng(22)
    hid = bf(rng.standard_normal((2, H)))
    toks = [3, 499]
    out = oracle.head(w, toks, hid, 1e-6)
    x, _ = oracle.input_stage(w["embed"], w["enorm_w"], w["hnorm_w"], w["eh_proj"], toks, hid, 1e-6)
    assert np.array_equal(out["x"], x)
    assert np.array_equal(out["xhat"], oracle.rms_norm(x, w["final_norm_w"], 1e-6))
    ref = f64(out["xhat"]) @ f64(w["lm_head"]).T
    np.testing.assert_allclose(out["logits"], ref, atol=1e-12, rtol=0)
    for b in range(2):
        assert out["draft"][b] == _brute_argmax(out["logits"][b].tolist())


def test_planted_ties_lowest_index_wins():
    # identical rows aligned with sign(xhat) are the largest logits and tie exactly
    H, V = 128, 1000
    w = _small_weights(H, V, 23)
    hid = bf(np.random.default_rng(24).standard_normal((1, H)))
    x, _ = oracle.input_stage(w["embed"], w["enorm_w"], w["hnorm_w"], w["eh_proj"], [7], hid, 1e-6)
    xh = oracle.rms_norm(x, w["final_norm_w"], 1e-6)[0]
    planted = [911, 40, 512]
    W = w["lm_head"].copy()
    W[planted] = bf(0.05 * np.sign(f64(xh)))
    lg = oracle.logits(0, W, None, xh)
    assert lg[40] == lg[512] == lg[911] == lg.max()
    assert oracle.argmax(lg) == 40
    q, s, _ = oracle.quantize(W)
    lg8 = oracle.logits(1, q, s, xh)
    assert lg8[40] == lg8[512] == lg8[911] == lg8.max()
    assert oracle.argmax(lg8) == 40


# ---------------------------------------------------------------------- vocabulary shards
def _bf16_logits(rng, V, levels=7):
    """BF16-valued logits with many exact ties (a few levels), as fp64."""
    vals = rng.integers(-levels, levels + 1, V).astype(np.float64) * 0.125
    return oracle.bf16_to_f64(oracle.f64_to_bf16(vals))


def _edges(rng, V, R):
    """R contiguous ranges covering [0, V): random, possibly empty, cut points."""
    cuts = np.sort(rng.integers(0, V + 1, R - 1))
    return np.concatenate([[0], cuts, [V]]).astype(np.int64)


def test_pick_combine_brute_force_equals_full_argmax():
    """The pick over any split into shards, each offering its own lowest-index maximum, is the
    lowest-index maximum of the whole vocabulary (ties across a boundary go to the lower range,
    the `>=` rule of the source's cross-rank pick); NaN and -inf included."""
    rng = np.random.default_rng(11)
    for trial in range(400):
        V = int(rng.integers(1, 60))
        lg = _bf16_logits(rng, V, levels=int(rng.integers(0, 4)))
        specials = rng.random(V)
        lg[specials < 0.1] = np.nan
        lg[(specials >= 0.1) & (specials < 0.15)] = -np.inf
        lg[(specials >= 0.15) & (specials < 0.17)] = np.inf
        R = int(rng.integers(1, 9))
        e = _edges(rng, V, R)
        offers = [oracle.shard_pick(lg, int(e[r]), int(e[r + 1] - e[r])) for r in range(R)]
        got = oracle.pick_combine([o[0] for o in offers], [o[1] for o in offers])
        assert got == oracle.argmax(lg), (trial, lg, e)


def test_pick_combine_special_cases():
    nan = float("nan")
    assert oracle.pick_combine([], []) == -1
    assert oracle.pick_combine([nan, nan], [-1, -1]) == -1
    assert oracle.pick_combine([nan, 1.0], [3, 7]) == 7          # NaN never wins
    assert oracle.pick_combine([2.0, 2.0], [9, 4]) == 4          # tie: lowest index
    assert oracle.pick_combine([-0.0, 0.0], [5, 2]) == 2         # -0 == +0
    assert oracle.pick_combine([-np.inf, -5.0], [0, 8]) == 8
    assert oracle.pick_combine([-np.inf], [3]) == 3              # -inf wins when alone


def test_xchg_lanes_adding_zero_is_exact():
    """The source's SUM all-reduce hands each rank the other's lanes unchanged because adding
    zero is exact: every non-NaN BF16 pattern plus +0 is itself (-0 + +0 gives +0, equal)."""
    pats = np.arange(65536, dtype=np.uint16)
    keep = ~np.isnan(oracle.bf16_to_f64(pats))
    zero = np.zeros(8, np.uint16)
    for p in pats[keep][::37]:
        lanes = np.full(8, p, np.uint16)
        out = oracle.xchg_sum(lanes, zero)
        want = 0 if p == 0x8000 else p
        assert np.all(out == want)


def test_xchg_lanes_digits_are_exact_only_through_256():
    """BF16 holds the integers 0..256 exactly (eight significant bits), so base-256 digits
    survive the exchange; 257 does not, which is why a token id travels as digits."""
    ints = np.arange(0, 300, dtype=np.float64)
    back = oracle.bf16_to_f64(oracle.f64_to_bf16(ints))
    assert np.array_equal(back[:257], ints[:257])
    assert back[257] != 257.0
    for g in (0, 255, 256, 65535, 65536, 154879, 2 ** 24 - 1):
        lanes = oracle.xchg_pack(1, 0x3F80, g)  # rank 1, value 1.0
        assert oracle.xchg_pick(oracle.xchg_sum(oracle.xchg_pack(0, 0xBF80, 0), lanes)) == g


def test_xchg_lanes_two_ranks_brute_force():
    """With BF16 logits (the source's logit type) the source's two-rank exchange of each
    half's maximum gives the lowest-index maximum of the whole vocabulary: a tie across the
    halves goes to rank 0, the lower range."""
    rng = np.random.default_rng(5)
    for trial in range(300):
        V = 2 * int(rng.integers(1, 40))
        if trial % 50 == 0:
            V = 2 * 100000  # indices beyond 2^16 use the third digit
        lg = _bf16_logits(rng, V, levels=int(rng.integers(0, 3)))
        n = V // 2
        lanes = np.zeros(8, np.uint16)
        for rank in (0, 1):
            v, g = oracle.shard_pick(lg, rank * n, n)
            lanes = oracle.xchg_sum(lanes, oracle.xchg_pack(rank, int(oracle.f64_to_bf16(np.array([v]))[0]), g))
        assert oracle.xchg_pick(lanes) == oracle.argmax(lg), trial


def test_xchg_lanes_round_fp32_maxima_that_the_exact_pick_separates():
    """Reading of the pages: the BF16 value lanes fit the source's BF16 logits. With FP32
    logits two close maxima can round to one BF16 value; the lanes then give rank 0 although
    rank 1 holds the larger logit, while the exact pick does not lose the difference."""
    v0, v1 = 1.0, 1.0 + 2.0 ** -12          # distinct in FP32, equal after BF16 rounding
    b0 = int(oracle.f64_to_bf16(np.array([v0]))[0])
    b1 = int(oracle.f64_to_bf16(np.array([v1]))[0])
    assert b0 == b1
    lanes = oracle.xchg_sum(oracle.xchg_pack(0, b0, 10), oracle.xchg_pack(1, b1, 20))
    assert oracle.xchg_pick(lanes) == 10
    assert oracle.pick_combine([v0, v1], [10, 20]) == 20
