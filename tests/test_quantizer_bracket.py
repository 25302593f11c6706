"""The FP8 quantiser kernel's shortcut, checked on the CPU against the oracle.

The kernel does not divide every weight by its row scale s. It computes r = 1/s and the two
products y_up = w * r (1 + 2^-21) and y_dn = w * r (1 - 2^-21), every operation rounded to
nearest in fp32. When both convert to the same E4M3 code, that code is taken. Otherwise it
falls back to the IEEE division w / s. Rows whose scale is not a normal fp32 number always use
the division.

The argument: the two products bracket fp32(w / s), and the E4M3 conversion is monotonic. This
test restates the rule with numpy fp32 arithmetic and torch's float8_e4m3fn cast (round to
nearest even, inputs kept within +-448). It checks the rule against the oracle's codes for every
finite BF16 pattern under many row maxima, and for Gaussian rows. It also checks that the
fallback is rare enough for the shortcut to pay.
"""
import numpy as np
import torch

import oracle

F32 = np.float32


def e4m3_codes(y: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.clip(y, -448, 448).astype(F32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def bracket_quantize(Wb: np.ndarray):
    """(codes, scales, fallbacks) by the kernel's rule."""
    V, H = Wb.shape
    mx = (Wb & 0x7FFF).astype(np.uint32).max(axis=1)
    f = (Wb.astype(np.uint32) << 16).view(F32)
    s = ((mx << 16).view(F32) / F32(448)).astype(F32)
    s[mx >= 0x7F80] = 0
    q = np.zeros((V, H), np.uint8)
    fallbacks = 0
    for v in range(V):
        if s[v] == 0:
            continue
        exact = e4m3_codes((f[v] / s[v]).astype(F32))
        if s[v] >= F32(1.17549435e-38):
            r = F32(1) / s[v]
            up = e4m3_codes((f[v] * F32(r * F32(1 + 2.0 ** -21))).astype(F32))
            dn = e4m3_codes((f[v] * F32(r * F32(1 - 2.0 ** -21))).astype(F32))
            q[v] = np.where(up == dn, up, exact)
            fallbacks += int((up != dn).sum())
        else:
            q[v] = exact
    return q, s, fallbacks


def test_bracket_rule_matches_oracle_on_every_pattern_under_many_maxima():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite = pats[(pats & 0x7F80) != 0x7F80]
    rng = np.random.default_rng(5)
    tops = np.concatenate([[0x0001, 0x0080, 0x00FF, 0x0100, 0x3F80, 0x4300, 0x7F7F],
                           rng.choice(finite[(finite & 0x7FFF) >= 0x0100] & 0x7FFF, 40, replace=False)])
    total = 0
    for top in tops:
        allp = finite[(finite & 0x7FFF) <= top]
        W = np.concatenate([[top], allp]).astype(np.uint16)[None, :]
        q_ref, s_ref, _ = oracle.quantize(W)
        q, s, _ = bracket_quantize(W)
        assert np.array_equal(s.view(np.uint32), s_ref.view(np.uint32)), hex(int(top))
        assert np.array_equal(q, q_ref), hex(int(top))
        total += W.size
    assert total > 1_000_000


def test_bracket_rule_on_gaussian_rows_and_fallback_rate():
    g = torch.Generator().manual_seed(3)
    W = (torch.randn((32, 4096), generator=g) * 0.02).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    q_ref, s_ref, _ = oracle.quantize(W)
    q, s, fallbacks = bracket_quantize(W)
    assert np.array_equal(q, q_ref) and np.array_equal(s.view(np.uint32), s_ref.view(np.uint32))
    # nearly all fallbacks are exact ties of the E4M3 rounding; they stay around a percent
    assert 0 < fallbacks < 0.02 * W.size
