"""GPU parity of the context-row input stage (mtp_head_context_rows) against the CPU oracle.

For R > 16 rows the library runs two kernels: the normalised concat of every row (checked here
bit for bit against the oracle's concat, read back from the workspace) and x = concat . eh_proj^T
on the tensor cores with FP32 accumulation (checked against the oracle's fp64 sum within the
FP32-accumulation band below, plus a bound on how many elements may differ from the correctly
rounded x at all). R <= 16 must give exactly what the batched input stage gives.
"""
import numpy as np
import pytest
import torch

import mtp_speculative_draft_head_gb300 as m
import oracle
import synth
from gpu_helpers import abs_product_sums, check_x, context_band

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
EPS = synth.EPS


class Ctx:
    def __init__(self, H, R, V=4096, seed=0, tokens=None):
        self.H, self.R, self.V = H, R, V
        w = synth.make_weights(H, V, seed, "cpu")
        t, self.hidden = synth.make_step_inputs(H, V, R, seed + 7, "cpu", distinct=False)
        self.tokens = t if tokens is None else tokens
        self.wb = {k: synth.bits(v) for k, v in w.as_dict().items()}
        self.g = {k: v.to(DEV) for k, v in w.as_dict().items()}

    def run(self, ws_extra=0):
        x = torch.full((self.R, self.H), 7, dtype=torch.bfloat16, device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        n = m.mtp_head_context_workspace_bytes(self.R, self.H)
        ws = torch.empty(n + ws_extra, dtype=torch.uint8, device=DEV) if n else None
        m.mtp_head_context_rows(self.g["embed"], self.g["enorm_w"], self.g["hnorm_w"], self.g["eh_proj"],
                                self.tokens.to(DEV), self.hidden.to(DEV), x, ws, st, EPS)
        torch.cuda.synchronize()
        return x, int(st.item()), ws

    def oracle(self, rows=None):
        rows = np.arange(self.R) if rows is None else np.asarray(rows)
        tok = synth.bits(self.tokens).astype(np.int64)[rows]
        hid = synth.bits(self.hidden)[rows]
        x, concat, st, sums = oracle.input_stage(self.wb["embed"], self.wb["enorm_w"], self.wb["hnorm_w"],
                                                 self.wb["eh_proj"], tok, hid, EPS, return_concat=True,
                                                 return_sums=True)
        return x, concat, st, sums


def workspace_concat(ws, R, H, rows):
    """Rows of the normalised concat the first kernel leaves at the start of the workspace."""
    idx = torch.as_tensor(rows, dtype=torch.long, device=ws.device)
    return ws[: R * 2 * H * 2].view(torch.int16).view(R, 2 * H)[idx].cpu().numpy().view(np.uint16)


def x_rows(x, rows):
    return synth.bits(x[torch.as_tensor(rows, dtype=torch.long, device=x.device)])


def check_rows(c, x_gpu, ws, rows=None):
    rows = np.arange(c.R) if rows is None else np.asarray(rows)
    x_ref, concat_ref, st_ref, sums = c.oracle(rows)
    ok = st_ref == 0
    assert np.array_equal(workspace_concat(ws, c.R, c.H, rows)[ok], concat_ref[ok]), "concat differs from the oracle"
    abs_sums = abs_product_sums(c.wb["eh_proj"], concat_ref)
    K = 2 * c.H
    x_sel = x_rows(x_gpu, rows)
    assert np.all(x_sel[~ok] == 0), "rows with an out-of-range token must be zeros"
    diff = np.nonzero(x_sel[ok] != x_ref[ok])[0].size
    # the FP32-accumulation band, as an interval check around the exact sum
    E = context_band(K) * abs_sums[ok]
    g = oracle.bf16_to_f64(x_sel[ok])
    s = sums[ok]
    lo = oracle.bf16_to_f64(oracle.f64_to_bf16(s - E))
    hi = oracle.bf16_to_f64(oracle.f64_to_bf16(s + E))
    bad = ~((lo <= g) & (g <= hi))
    assert not bad.any(), f"{int(bad.sum())} elements outside the FP32-accumulation band"
    # a systematic error inside the worst-case band would still move many roundings
    assert diff <= max(4, x_sel[ok].size // 100), f"{diff} of {x_sel[ok].size} elements differ from the oracle"
    return diff


@pytest.mark.parametrize("H,R", [
    (256, 17),     # one 128-row tile, 8 k-blocks split 8 ways
    (256, 300),    # three 128-row tiles, the last with 44 rows, split 4 ways
    (1024, 130),   # four column tiles, one 256-row tile (both accumulators, the second with 2
                   # rows), 32 k-blocks split 11 ways (uneven ranges)
    (288, 200),    # H not a multiple of the 256-column tile: ragged last column tile
    (96, 40),      # H below one column tile, 3 k-blocks (fewer than the ring's stages), whole tile
    (2048, 257),   # 24 tiles (the last row tile holds one row), 64 k-blocks split 5 ways
    (6144, 40),    # GLM hidden size, a catch-up-sized batch of rows: 24 tiles split 4 ways
])
def test_context_rows_match_oracle(H, R):
    c = Ctx(H, R, seed=H + R)
    x, st, ws = c.run()
    assert st == 0
    check_rows(c, x, ws)


@pytest.mark.parametrize("R", [
    512,    # the launch the benchmark times: 48 tiles of 256 rows, each split 3 ways along k
    1300,   # 256-row tiles, whole; the last row tile holds 20 rows (one accumulator)
    2048,   # a whole wave of 152 tiles, then 40 tiles split along k
    3000,   # whole tiles only (288 tiles), ragged last row tile; some tokens out of range
])
def test_context_rows_glm_size_sampled(R):
    """GLM hidden size; oracle on sampled rows at both ends of row tiles and halves."""
    c = Ctx(6144, R, seed=11 + R)
    bad = [r for r in (5, 2999) if r < R and R == 3000]
    if bad:
        t = c.tokens.clone()
        t[bad] = -3
        c.tokens = t
    x, st, ws = c.run()
    assert st == (m.ERR_TOKEN_RANGE if bad else 0)
    rows = sorted({0, 1, 127, 128, 255, 256, R // 2, R - 2, R - 1} | set(bad))
    check_rows(c, x, ws, rows=rows)


@pytest.mark.parametrize("H,R", [(512, 150), (2048, 150)])
def test_context_rows_out_of_range_tokens(H, R):
    V = 1000
    c = Ctx(H, R, V=V, seed=3)
    t = c.tokens.clone()
    t[[0, 77, 128, 149]] = torch.tensor([-1, V, 2 ** 31 - 1, -(2 ** 31)], dtype=torch.int32)
    c.tokens = t
    x, st, ws = c.run()
    assert st == m.ERR_TOKEN_RANGE
    check_rows(c, x, ws)


@pytest.mark.parametrize("R", [2, 9, 16])
def test_context_rows_small_r(R):
    """R <= 16: with a workspace (H a multiple of 32) the context-row path, checked like every R;
    without one, the batched input stage, identical to mtp_head_input_batched."""
    H = 1024
    c = Ctx(H, R, seed=5 + R)
    x, st, ws = c.run()
    assert st == 0
    check_rows(c, x, ws)
    xn = torch.full((R, H), 7, dtype=torch.bfloat16, device=DEV)
    stn = torch.zeros(1, dtype=torch.int32, device=DEV)
    m.mtp_head_context_rows(c.g["embed"], c.g["enorm_w"], c.g["hnorm_w"], c.g["eh_proj"], c.tokens.to(DEV),
                            c.hidden.to(DEV), xn, None, stn, EPS)
    xb = torch.full((R, H), 7, dtype=torch.bfloat16, device=DEV)
    stb = torch.zeros(1, dtype=torch.int32, device=DEV)
    m.mtp_head_input_batched(c.g["embed"], c.g["enorm_w"], c.g["hnorm_w"], c.g["eh_proj"], c.tokens.to(DEV),
                             c.hidden.to(DEV), xb, stb, EPS)
    torch.cuda.synchronize()
    assert int(stn.item()) == 0 and int(stb.item()) == 0
    assert np.array_equal(synth.bits(xn), synth.bits(xb))


def test_context_rows_deterministic_and_workspace_checked():
    c = Ctx(512, 200, seed=9)
    x1, _, _ = c.run()
    x2, _, _ = c.run(ws_extra=4096)
    assert torch.equal(x1.view(torch.int16), x2.view(torch.int16))
    small = torch.empty(m.mtp_head_context_workspace_bytes(200, 512) - 1, dtype=torch.uint8, device=DEV)
    x = torch.empty((200, 512), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(m.MTPError) as e:
        m.mtp_head_context_rows(c.g["embed"], c.g["enorm_w"], c.g["hnorm_w"], c.g["eh_proj"], c.tokens.to(DEV),
                                c.hidden.to(DEV), x, small)
    assert e.value.code == m.ERR_WORKSPACE
    with pytest.raises(m.MTPError) as e:  # H % 32 != 0 with R > 16
        c2 = Ctx(100, 20, seed=1)
        x = torch.empty((20, 100), dtype=torch.bfloat16, device=DEV)
        ws = torch.empty(m.mtp_head_context_workspace_bytes(20, 100), dtype=torch.uint8, device=DEV)
        m.mtp_head_context_rows(c2.g["embed"], c2.g["enorm_w"], c2.g["hnorm_w"], c2.g["eh_proj"],
                                c2.tokens.to(DEV), c2.hidden.to(DEV), x, ws)
    assert e.value.code == m.ERR_NOT_IMPLEMENTED


def test_context_rows_maximum_rows_sampled():
    """The largest R the entry point takes (65536) at the GLM hidden size: 6080 whole tiles in 40
    waves and the split remainder; the oracle checks rows at both ends and across tiles."""
    H, R = 6144, 65536
    V = 4096
    c = Ctx(H, R, V=V, seed=77)
    x, st, ws = c.run()
    assert st == 0
    check_rows(c, x, ws, rows=[0, 255, 256, 30001, 65279, 65280, 65535])


def test_context_rows_smallest_gemm_shape_and_all_tokens_invalid():
    # H = 32: one 64-element k-block per half, a single partial column tile
    c = Ctx(32, 17, V=50, seed=4)
    x, st, ws = c.run()
    assert st == 0
    check_rows(c, x, ws)
    # every token out of range: all rows zero, status set, nothing else read from embed
    c2 = Ctx(256, 40, V=100, seed=6)
    c2.tokens = torch.full((40,), 100, dtype=torch.int32)
    x2, st2, _ = c2.run()
    assert st2 == m.ERR_TOKEN_RANGE
    assert bool((x2.view(torch.int16) == 0).all())
