"""GPU parity of the CUDA library (through its C ABI) against the CPU oracle on small and
medium shapes: several tiles and ragged tails, both weight dtypes, every kernel path
(register-xhat and bulk-copy pipelines for B = 1; for B >= 2 the tensor-core kernels -- output
stage when H is a multiple of 8, input stage when H is a multiple of 32 -- and plain-load
kernels otherwise), plus the
edge cases: out-of-range tokens, NaN/Inf, exact ties, determinism, CUDA-graph replay and the
quantiser bit for bit."""
import numpy as np
import pytest
import torch

import mtp_speculative_draft_head_gb300 as m
import oracle
import synth
from gpu_helpers import (TOL_BF16, TOL_FP8, abs_product_sums, check_draft, check_logits_and_draft, check_x, x_band,
                         step_x_band,
                         lowest_argmax)

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
EPS = synth.EPS


def _bits(t):
    return synth.bits(t)


class Case:
    def __init__(self, H, V, B, seed=0):
        self.H, self.V, self.B = H, V, B
        self.w = synth.make_weights(H, V, seed, "cpu")
        self.tokens, self.hidden = synth.make_step_inputs(H, V, B, seed + 100, "cpu")
        self.wb = {k: _bits(v) for k, v in self.w.as_dict().items()}
        self.g = {k: v.to(DEV) for k, v in self.w.as_dict().items()}
        self.ws = m.workspace(B, H, V, DEV)

    def quantize_gpu(self):
        q = torch.empty((self.V, self.H), dtype=torch.uint8, device=DEV)
        s = torch.empty(self.V, dtype=torch.float32, device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        m.mtp_head_quantize_fp8(self.g["lm_head"], q, s, st)
        torch.cuda.synchronize()
        return q, s, int(st.item())

    def input_gpu(self, tokens=None, hidden=None):
        tokens = self.tokens if tokens is None else tokens
        hidden = self.hidden if hidden is None else hidden
        B = tokens.numel()
        x = torch.full((B, self.H), 7, dtype=torch.bfloat16, device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        m.mtp_head_input_batched(self.g["embed"], self.g["enorm_w"], self.g["hnorm_w"], self.g["eh_proj"],
                                 tokens.to(DEV), hidden.to(DEV), x, st, EPS)
        torch.cuda.synchronize()
        return x, int(st.item())

    def output_gpu(self, x, W, scale, wt, want_logits=True):
        B = x.shape[0]
        logits = torch.full((B, self.V), float("nan"), dtype=torch.float32, device=DEV) if want_logits else None
        draft = torch.full((B,), -7, dtype=torch.int32, device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        m.mtp_head_logits_argmax_batched(x, self.g["final_norm_w"], W, scale, wt, logits, draft, self.ws, st, EPS)
        torch.cuda.synchronize()
        return logits, draft, int(st.item())

    def oracle_input(self):
        x, self.concat_ref, st, sums = oracle.input_stage(
            self.wb["embed"], self.wb["enorm_w"], self.wb["hnorm_w"], self.wb["eh_proj"],
            _bits(self.tokens).astype(np.int64), _bits(self.hidden), EPS, return_concat=True, return_sums=True)
        return x, st, sums

    def abs_sums(self):
        """sum_k |eh_proj[h, k] * concat[b, k]|: the scale of the accumulation band of x."""
        return abs_product_sums(self.wb["eh_proj"], self.concat_ref)

    def oracle_logits(self, x_bits, wt, W_bits, scale):
        xhat = oracle.final_norm(x_bits, self.wb["final_norm_w"], EPS)
        return oracle.logits(wt, W_bits, scale, xhat, threads=8).reshape(x_bits.shape[0], -1)


SHAPES = [  # (H, V, B): tiles, ragged tails and every path
    (256, 4096, 1),     # the small workload
    (1000, 5003, 1),    # BF16 rows of 2000 B (one partial chunk); FP8 rows not 16-B -> plain path
    (1000, 5003, 3),    # B >= 2, H % 8 == 0 -> tensor-core kernel (partial last k-block)
    (2056, 1031, 2),    # tensor-core kernel, ragged last row tile
    (2048, 777, 4),
    (6144, 1000, 1),    # GLM hidden size: 3 BF16 chunks, FP8 one full + one partial chunk;
                        # V below the rows fixed per warp (no dynamic hand-out)
    (4096, 3650, 1),    # a few rows past the fixed ones (BF16): dynamic blocks, a partial last one
    (4096, 7300, 1),    # the same for FP8 (12 warps, more fixed rows)
    (4096, 300, 5),
    (512, 2000, 16),    # B = 16: two n-tiles of 8 sequences
    (544, 160000, 9),   # output: more than 8 row tiles per CTA; input: a k-chunk across the
                        # embedding / hidden boundary and a partial last chunk
    (6144, 3000, 16),
    (96, 300, 3),       # input: one partial k-chunk holding both halves
    (16384, 1000, 2),   # input: more 8-row groups than 8 per SM -> more CTAs than SMs
    (8, 300, 2),        # output: a single, partial k-block; input: H % 32 != 0 -> error-free kernel
    (100, 50, 2),       # H % 8 != 0 -> plain kernels
    (8, 7, 1),
    (64, 1, 1),         # V = 1
]


@pytest.mark.parametrize("H,V,B", SHAPES)
@pytest.mark.parametrize("fp8", [False, True])
def test_head_matches_oracle(H, V, B, fp8):
    c = Case(H, V, B, seed=H + V + B)
    x_ref, st_ref, sums = c.oracle_input()
    assert np.all(st_ref == 0)
    x_gpu, st = c.input_gpu()
    assert st == 0
    check_x(_bits(x_gpu), x_ref, sums, c.abs_sums(), x_band(H, B))
    if fp8:
        q, s, qst = c.quantize_gpu()
        assert qst == 0
        q_ref, s_ref, _ = oracle.quantize(c.wb["lm_head"])
        assert np.array_equal(_bits(q), q_ref)
        assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
        W, scale, wt, tol, Wb, sb = q, s, m.W_FP8_E4M3, TOL_FP8, q_ref, s_ref
    else:
        W, scale, wt, tol, Wb, sb = c.g["lm_head"], None, m.W_BF16, TOL_BF16, c.wb["lm_head"], None
    ref = c.oracle_logits(x_ref, wt, Wb, sb)
    # output stage on the GPU's own x (the whole head) ...
    logits, draft, st = c.output_gpu(x_gpu, W, scale, wt)
    assert st == 0
    err = check_logits_and_draft(logits.cpu().numpy(), draft.cpu().numpy(), ref, tol)
    assert err < 5e-3  # the real error is fp32 rounding; the stated bar is far looser
    # ... on the oracle's x (the output stage alone) ...
    x_or = torch.from_numpy(x_ref.view(np.int16)).view(torch.bfloat16).to(DEV)
    logits2, draft2, _ = c.output_gpu(x_or, W, scale, wt)
    check_logits_and_draft(logits2.cpu().numpy(), draft2.cpu().numpy(), ref, tol)
    # ... without storing logits (same draft) ...
    _, draft3, _ = c.output_gpu(x_gpu, W, scale, wt, want_logits=False)
    assert torch.equal(draft3, draft)
    # ... and through the one-call forward: with the full-size workspace its input stage takes
    # the context-row GEMM for 2..16 sequences at H % 32 == 0 (checked against its own band), else
    # the kernels above (bitwise the same); its output stage is the one above, bit for bit
    xf = torch.empty_like(x_gpu)
    lf = torch.empty_like(logits)
    df = torch.empty_like(draft)
    m.mtp_head_forward_batched(c.g["embed"], c.g["enorm_w"], c.g["hnorm_w"], c.g["eh_proj"],
                               c.g["final_norm_w"], W, scale, wt, c.tokens.to(DEV), c.hidden.to(DEV),
                               xf, lf, df, c.ws, None, EPS)
    torch.cuda.synchronize()
    if B >= 2 and H % 32 == 0:
        n_diff = check_x(_bits(xf), x_ref, sums, c.abs_sums(), step_x_band(H, B))
        assert n_diff <= max(1, x_ref.size // 100)
        lo, do, _ = c.output_gpu(xf, W, scale, wt)
        assert torch.equal(df, do) and torch.equal(lf.view(torch.int32), lo.view(torch.int32))
    else:
        assert torch.equal(xf, x_gpu) and torch.equal(df, draft)
        assert torch.equal(lf.view(torch.int32), logits.view(torch.int32))


def test_worked_example_on_gpu(golden_dir):
    import json
    import os
    ex = json.load(open(os.path.join(golden_dir, "worked_example_4x8.json")))

    def t(v):
        return torch.tensor(v, dtype=torch.float32).to(torch.bfloat16).to(DEV).contiguous()

    g = dict(embed=t(ex["embed"]), enorm_w=t(ex["enorm_w"]), hnorm_w=t(ex["hnorm_w"]),
             eh_proj=t(ex["eh_proj"]), final_norm_w=t(ex["final_norm_w"]), lm_head=t(ex["lm_head"]))
    ws = m.workspace(1, 4, 8, DEV)
    for hnorm_w, hid, want_x in ((ex["hnorm_w"], ex["target_hidden"], ex["expected_x"]),
                                 (ex["variant_hnorm_w"], ex["variant_target_hidden"], ex["variant_expected_x"])):
        x = torch.empty((1, 4), dtype=torch.bfloat16, device=DEV)
        m.mtp_head_input(g["embed"], g["enorm_w"], t(hnorm_w), g["eh_proj"],
                         torch.tensor([ex["token"]], dtype=torch.int32, device=DEV), t([hid]), x)
        torch.cuda.synchronize()
        assert x.float().cpu().view(-1).tolist() == want_x
        logits = torch.empty((1, 8), dtype=torch.float32, device=DEV)
        draft = torch.empty(1, dtype=torch.int32, device=DEV)
        m.mtp_head_logits_argmax(x, g["final_norm_w"], g["lm_head"], None, m.W_BF16, logits, draft, ws)
        torch.cuda.synchronize()
        assert logits.cpu().view(-1).tolist() == ex["expected_logits"]
        assert int(draft.item()) == ex["expected_draft"]
    # FP8 copy: codes, then the tie survives and the lower index wins
    q = torch.empty((8, 4), dtype=torch.uint8, device=DEV)
    s = torch.empty(8, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    m.mtp_head_quantize_fp8(g["lm_head"], q, s, st)
    m.mtp_head_logits_argmax(x, g["final_norm_w"], q, s, m.W_FP8_E4M3, logits, draft, ws)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert q.cpu().tolist() == ex["expected_fp8_codes"]
    lg = logits.cpu().view(-1).double().numpy()
    np.testing.assert_allclose(lg, ex["expected_logits"], rtol=ex["fp8_logit_rel_tol"], atol=1e-12)
    assert lg[3] == lg[5] and int(draft.item()) == ex["expected_draft"]


def test_out_of_range_tokens_flag_and_zero_rows():
    c = Case(256, 4096, 3, seed=5)
    tokens = torch.tensor([11, c.V + 3, -1], dtype=torch.int32)
    x, st = c.input_gpu(tokens=tokens)
    assert st == m.ERR_TOKEN_RANGE
    assert torch.all(x[1:] == 0)
    x_ref, concat, _, sums = oracle.input_stage(c.wb["embed"], c.wb["enorm_w"], c.wb["hnorm_w"], c.wb["eh_proj"],
                                                [11, c.V + 3, -1], _bits(c.hidden), EPS, return_concat=True,
                                                return_sums=True)
    check_x(_bits(x), x_ref, sums, abs_product_sums(c.wb["eh_proj"], concat))
    # a zero x gives all-zero logits: every logit ties and index 0 wins
    logits, draft, _ = c.output_gpu(x, c.g["lm_head"], None, m.W_BF16)
    assert torch.all(logits[1:] == 0) and draft[1:].tolist() == [0, 0]


@pytest.mark.parametrize("fp8", [False, True])
def test_nan_input_gives_draft_minus_one(fp8):
    c = Case(256, 1000, 2, seed=6)
    x = torch.ones((2, 256), dtype=torch.bfloat16, device=DEV)
    x[1, 17] = float("nan")
    if fp8:
        q, s, _ = c.quantize_gpu()
        W, scale, wt = q, s, m.W_FP8_E4M3
    else:
        W, scale, wt = c.g["lm_head"], None, m.W_BF16
    logits, draft, _ = c.output_gpu(x, W, scale, wt)
    assert torch.isnan(logits[1]).all() and int(draft[1]) == -1
    assert int(draft[0]) == lowest_argmax(logits[0].double().cpu().numpy())


def test_infinite_logits_and_ties():
    H, V = 64, 12
    W = torch.zeros((V, H), dtype=torch.float32)
    W[1, 0], W[1, 1] = float("inf"), float("-inf")   # inf - inf = NaN: never wins
    W[3, 0] = float("inf")                            # +inf
    W[7, 0] = float("inf")                            # +inf again: tie, 3 wins
    W[5, 0] = float("-inf")
    W[9, 2] = 1e30
    Wd = W.to(torch.bfloat16).to(DEV)
    fw = torch.ones(H, dtype=torch.bfloat16, device=DEV)
    x = torch.ones((1, H), dtype=torch.bfloat16, device=DEV)
    ws = m.workspace(1, H, V, DEV)
    logits = torch.empty((1, V), dtype=torch.float32, device=DEV)
    draft = torch.empty(1, dtype=torch.int32, device=DEV)
    m.mtp_head_logits_argmax(x, fw, Wd, None, m.W_BF16, logits, draft, ws)
    torch.cuda.synchronize()
    lg = logits.cpu().view(-1)
    assert torch.isnan(lg[1]) and lg[3] == float("inf") and lg[7] == float("inf") and lg[5] == float("-inf")
    assert int(draft.item()) == 3
    # all -inf: the lowest index wins
    Wn = torch.zeros((V, H), dtype=torch.float32)
    Wn[:, 0] = float("-inf")
    m.mtp_head_logits_argmax(x, fw, Wn.to(torch.bfloat16).to(DEV), None, m.W_BF16, logits, draft, ws)
    torch.cuda.synchronize()
    assert int(draft.item()) == 0


@pytest.mark.parametrize("fp8", [False, True])
def test_planted_ties_lowest_index_wins(fp8):
    H, V = 2048, 20000
    c = Case(H, V, 1, seed=9)
    x_ref, _, _ = c.oracle_input()
    xhat = oracle.final_norm(x_ref, c.wb["final_norm_w"], EPS)[0]
    rows = synth.pick_rows(V, 16, seed=9)
    sign = torch.from_numpy(oracle.bf16_to_f64(xhat))
    W = synth.plant_rows(c.w.lm_head, rows, sign, 0.05)
    Wd = W.to(DEV)
    x_gpu, _ = c.input_gpu()
    if fp8:
        q = torch.empty((V, H), dtype=torch.uint8, device=DEV)
        s = torch.empty(V, dtype=torch.float32, device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        m.mtp_head_quantize_fp8(Wd, q, s, st)
        logits, draft, _ = c.output_gpu(x_gpu, q, s, m.W_FP8_E4M3)
    else:
        logits, draft, _ = c.output_gpu(x_gpu, Wd, None, m.W_BF16)
    lg = logits.cpu().view(-1)
    planted = rows.tolist()
    assert len(set(lg[planted].view(torch.int32).tolist())) == 1  # bit-identical tie
    assert int(draft.item()) == min(planted)


@pytest.mark.parametrize("B", [5, 16])
@pytest.mark.parametrize("fp8", [False, True])
def test_batched_planted_ties_across_ctas(B, fp8):
    """Each sequence gets its own four identical rows of lm_head (bit-identical largest logits)
    spread over the vocabulary, so over different CTAs of the batched sweep: the lowest planted
    row wins for every sequence, whatever order the CTAs' picks reach the workspace in; one
    sequence with a NaN in x gives -1."""
    H, V = 2048, 20000
    c = Case(H, V, B, seed=31 + B)
    x = synth._normal_bf16((B, H), 0.0, 1.0, torch.Generator().manual_seed(B), "cpu")
    xhat = oracle.final_norm(_bits(x), c.wb["final_norm_w"], EPS)
    rows = synth.pick_rows(V, 4 * B, seed=B).view(-1)
    rows = rows[torch.randperm(4 * B, generator=torch.Generator().manual_seed(7))].view(B, 4)  # disjoint sets
    W = c.w.lm_head
    for b in range(B):
        W = synth.plant_rows(W, rows[b], torch.from_numpy(oracle.bf16_to_f64(xhat[b])), 0.05)
    Wd = W.to(DEV)
    xg = x.to(DEV)
    xg[B - 1, 100] = float("nan")
    if fp8:
        q = torch.empty((V, H), dtype=torch.uint8, device=DEV)
        s = torch.empty(V, dtype=torch.float32, device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        m.mtp_head_quantize_fp8(Wd, q, s, st)
        logits, draft, status = c.output_gpu(xg, q, s, m.W_FP8_E4M3)
    else:
        logits, draft, status = c.output_gpu(xg, Wd, None, m.W_BF16)
    assert status == 0
    lg = logits.cpu()
    for b in range(B - 1):
        planted = rows[b].tolist()
        assert len(set(lg[b, planted].view(torch.int32).tolist())) == 1  # bit-identical tie
        assert int(draft[b]) == min(planted) == lowest_argmax(lg[b].double().numpy())
    assert torch.isnan(lg[B - 1]).all() and int(draft[B - 1]) == -1


@pytest.mark.parametrize("fp8", [False, True])
def test_output_stage_in_its_smallest_workspace(fp8):
    """The output stage needs the same 2304 bytes of workspace for any B: a 16-sequence sweep in
    exactly that much (zero-filled once) gives the bits of a sweep in a whole-step workspace, twice
    in a row (the counters and the running picks are back to zero after each call)."""
    c = Case(1000, 5003, 16, seed=41)
    x = synth._normal_bf16((16, c.H), 0.0, 1.0, torch.Generator().manual_seed(41), "cpu").to(DEV)
    if fp8:
        q, s_, _ = c.quantize_gpu()
        W, scale, wt = q, s_, m.W_FP8_E4M3
    else:
        W, scale, wt = c.g["lm_head"], None, m.W_BF16
    ref_lg, ref_d, st = c.output_gpu(x, W, scale, wt)
    assert st == 0
    small = torch.zeros(2304, dtype=torch.uint8, device=DEV)
    for _ in range(2):
        lg = torch.empty((16, c.V), dtype=torch.float32, device=DEV)
        d = torch.empty(16, dtype=torch.int32, device=DEV)
        m.mtp_head_logits_argmax_batched(x, c.g["final_norm_w"], W, scale, wt, lg, d, small, None, EPS)
        torch.cuda.synchronize()
        assert torch.equal(lg.view(torch.int32), ref_lg.view(torch.int32)) and torch.equal(d, ref_d)


def test_repeat_calls_are_bitwise_identical_and_graph_replay_matches():
    c = Case(2048, 30000, 2, seed=10)
    # x of the whole step (its input stage is the context-row GEMM here), eagerly
    x = torch.empty((2, c.H), dtype=torch.bfloat16, device=DEV)
    d0 = torch.empty(2, dtype=torch.int32, device=DEV)
    m.mtp_head_forward_batched(c.g["embed"], c.g["enorm_w"], c.g["hnorm_w"], c.g["eh_proj"], c.g["final_norm_w"],
                               c.g["lm_head"], None, m.W_BF16, c.tokens.to(DEV), c.hidden.to(DEV), x, None, d0,
                               c.ws, None, EPS)
    torch.cuda.synchronize()
    outs = [c.output_gpu(x, c.g["lm_head"], None, m.W_BF16) for _ in range(3)]
    for lg, dr, _ in outs[1:]:
        assert torch.equal(lg.view(torch.int32), outs[0][0].view(torch.int32)) and torch.equal(dr, outs[0][1])
    tokens, hidden = c.tokens.to(DEV), c.hidden.to(DEV)
    xg = torch.empty_like(x)
    lg = torch.empty((2, c.V), dtype=torch.float32, device=DEV)
    dr = torch.empty(2, dtype=torch.int32, device=DEV)

    def step(stream):
        m.mtp_head_forward_batched(c.g["embed"], c.g["enorm_w"], c.g["hnorm_w"], c.g["eh_proj"],
                                   c.g["final_norm_w"], c.g["lm_head"], None, m.W_BF16, tokens, hidden,
                                   xg, lg, dr, c.ws, None, EPS, stream)

    graph = m.MtpDraftHead.capture(step)
    for _ in range(3):
        lg.zero_()
        dr.fill_(-5)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(xg, x)
        assert torch.equal(lg.view(torch.int32), outs[0][0].view(torch.int32)) and torch.equal(dr, outs[0][1])


def test_workspace_reused_across_batch_sizes():
    c = Case(512, 3000, 4, seed=11)
    x, _ = c.input_gpu()
    ref = c.oracle_logits(_bits(x), 0, c.wb["lm_head"], None)
    for B in (4, 1, 3, 1):
        lg, dr, _ = c.output_gpu(x[:B].contiguous(), c.g["lm_head"], None, m.W_BF16)
        check_logits_and_draft(lg.cpu().numpy(), dr.cpu().numpy(), ref[:B], TOL_BF16)


@pytest.mark.parametrize("B", [1, 3])
@pytest.mark.parametrize("fp8", [False, True])
def test_output_stage_at_the_largest_hidden_size(B, fp8):
    """H = 65536, the largest the entry points take: the single-sequence stage holds xhat in
    128 KB of shared memory (plain kernel), the batched one builds it per stage (tensor-core
    kernel). V = 1031 ends in a ragged row tile."""
    H, V = 65536, 1031
    g = torch.Generator().manual_seed(65536 + B)
    W = (torch.randn((V, H), generator=g) * 0.02).to(torch.bfloat16)
    wf = (1.0 + 0.1 * torch.randn(H, generator=g)).to(torch.bfloat16)
    x = torch.randn((B, H), generator=g).to(torch.bfloat16)
    Wd, wfd, xd = W.to(DEV), wf.to(DEV), x.to(DEV)
    if fp8:
        q = torch.empty((V, H), dtype=torch.uint8, device=DEV)
        sc = torch.empty(V, dtype=torch.float32, device=DEV)
        qst = torch.zeros(1, dtype=torch.int32, device=DEV)
        m.mtp_head_quantize_fp8(Wd, q, sc, qst)
        torch.cuda.synchronize()
        q_ref, s_ref, _ = oracle.quantize(_bits(W))
        assert int(qst.item()) == 0 and np.array_equal(_bits(q), q_ref)
        Wg, scale, wt, tol, Wb, sb = q, sc, m.W_FP8_E4M3, TOL_FP8, q_ref, s_ref
    else:
        Wg, scale, wt, tol, Wb, sb = Wd, None, m.W_BF16, TOL_BF16, _bits(W), None
    xhat = oracle.final_norm(_bits(x), _bits(wf), EPS)
    ref = oracle.logits(wt, Wb, sb, xhat, threads=8).reshape(B, V)
    logits = torch.full((B, V), float("nan"), dtype=torch.float32, device=DEV)
    draft = torch.empty(B, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    m.mtp_head_logits_argmax_batched(xd, wfd, Wg, scale, wt, logits, draft, m.workspace(B, H, V, DEV), st, EPS)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    err = check_logits_and_draft(logits.cpu().numpy(), draft.cpu().numpy(), ref, tol)
    assert err < 5e-3


def test_output_stage_without_a_kernel_for_the_shape():
    """Odd H near the maximum with B >= 2: xhat of two sequences does not fit in shared memory
    and the tensor-core kernel needs H % 8 == 0, so the call returns MTP_ERR_NOT_IMPLEMENTED
    before launching anything, and the outputs stay untouched."""
    H, V, B = 65535, 64, 2
    W = torch.zeros((V, H), dtype=torch.bfloat16, device=DEV)
    wf = torch.ones(H, dtype=torch.bfloat16, device=DEV)
    x = torch.ones((B, H), dtype=torch.bfloat16, device=DEV)
    logits = torch.full((B, V), 3.0, dtype=torch.float32, device=DEV)
    draft = torch.full((B,), -5, dtype=torch.int32, device=DEV)
    with pytest.raises(m.MTPError) as e:
        m.mtp_head_logits_argmax_batched(x, wf, W, None, m.W_BF16, logits, draft, m.workspace(B, H, V, DEV), None, EPS)
    assert e.value.code == m.ERR_NOT_IMPLEMENTED
    torch.cuda.synchronize()
    assert bool((logits == 3.0).all()) and bool((draft == -5).all())


def test_quantizer_exhaustive_patterns_bitexact():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite = pats[(pats & 0x7F80) != 0x7F80]
    rng = np.random.default_rng(19)
    rows = []
    for top in (0x3F80, 0x0001, 0x0080, 0x2000, 0x4300, 0x7F7F, 0x0000):
        r = rng.permutation(finite)
        r = r[(r & 0x7FFF) <= top][:4096]
        r = np.resize(r, 4096)
        r[0] = top
        rows.append(r)
    Wb = np.stack(rows).astype(np.uint16)
    q_ref, s_ref, st_ref = oracle.quantize(Wb)
    assert st_ref == 0
    for H in (4096, 4000):  # vector and plain paths
        Wt = torch.from_numpy(Wb[:, :H].copy().view(np.int16)).view(torch.bfloat16).to(DEV)
        q = torch.empty((Wb.shape[0], H), dtype=torch.uint8, device=DEV)
        s = torch.empty(Wb.shape[0], dtype=torch.float32, device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        m.mtp_head_quantize_fp8(Wt, q, s, st)
        torch.cuda.synchronize()
        qr, sr, _ = oracle.quantize(Wb[:, :H].copy())
        assert int(st.item()) == 0
        assert np.array_equal(s.cpu().numpy().view(np.uint32), sr.view(np.uint32))
        assert np.array_equal(q.cpu().numpy(), qr)


@pytest.mark.parametrize("H", [16400, 12288, 12304])
def test_quantizer_row_widths_bitexact(H):
    """Wide rows: the load batches of both passes end ragged for H = 16400 and 12304 and exactly
    for 12288. Codes and scales must match the oracle bit for bit, for rows that hold every
    finite pattern below their maximum and for a row whose last element is a NaN."""
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite = pats[(pats & 0x7F80) != 0x7F80]
    rng = np.random.default_rng(H)
    rows = []
    for top in (0x3F80, 0x0080, 0x4300, 0x7F7F, 0x0000):
        r = rng.permutation(finite[(finite & 0x7FFF) <= top])
        r = np.resize(r, H)
        r[H // 2] = top
        rows.append(r)
    bad = np.resize(rng.permutation(finite), H)
    bad[H - 1] = 0x7FC0  # NaN in the last element of the row
    rows.append(bad)
    Wb = np.stack(rows).astype(np.uint16)
    q_ref, s_ref, st_ref = oracle.quantize(Wb)
    Wt = torch.from_numpy(Wb.view(np.int16)).view(torch.bfloat16).to(DEV)
    q = torch.empty((Wb.shape[0], H), dtype=torch.uint8, device=DEV)
    s = torch.empty(Wb.shape[0], dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    m.mtp_head_quantize_fp8(Wt, q, s, st)
    torch.cuda.synchronize()
    assert st_ref == m.ERR_NONFINITE and int(st.item()) == m.ERR_NONFINITE
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), q_ref)


def test_quantizer_rejects_nonfinite_rows():
    W = torch.randn((6, 64)) * 0.02
    W[2, 5] = float("nan")
    W[4, 0] = float("inf")
    Wd = W.to(torch.bfloat16).to(DEV)
    q = torch.full((6, 64), 0x55, dtype=torch.uint8, device=DEV)
    s = torch.full((6,), 3.0, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    m.mtp_head_quantize_fp8(Wd, q, s, st)
    torch.cuda.synchronize()
    assert int(st.item()) == m.ERR_NONFINITE
    assert float(s[2]) == 0.0 and float(s[4]) == 0.0 and torch.all(q[2] == 0) and torch.all(q[4] == 0)
    q_ref, s_ref, _ = oracle.quantize(_bits(Wd))
    assert np.array_equal(q.cpu().numpy(), q_ref)


def test_draft_head_class_and_host_forward():
    c = Case(256, 4096, 2, seed=12)
    head = m.MtpDraftHead(c.g["embed"], c.g["lm_head"], c.g["eh_proj"], c.g["enorm_w"], c.g["hnorm_w"],
                          c.g["final_norm_w"], eps=EPS, max_batch=2)
    assert head.quantize_fp8() == 0
    x_ref, _, _ = c.oracle_input()
    for fp8 in (False, True):
        _, logits, draft = head.forward(c.tokens.to(DEV), c.hidden.to(DEV), fp8=fp8, logits=True)
        if fp8:
            ref = c.oracle_logits(x_ref, 1, _bits(head.lm_head_fp8), head.row_scale.cpu().numpy())
        else:
            ref = c.oracle_logits(x_ref, 0, c.wb["lm_head"], None)
        check_logits_and_draft(logits.cpu().numpy(), draft.cpu().numpy(), ref, TOL_FP8 if fp8 else TOL_BF16)
        # host-buffer step: same draft
        th = c.tokens.clone().pin_memory()
        hh = c.hidden.clone().pin_memory()
        dh = torch.empty(2, dtype=torch.int32).pin_memory()
        W, s, wt = head._head(fp8)
        m.mtp_head_forward_host(head.embed, head.enorm_w, head.hnorm_w, head.eh_proj, head.final_norm_w,
                                W, s, wt, th, hh, torch.empty(2, dtype=torch.int32, device=DEV),
                                torch.empty((2, 256), dtype=torch.bfloat16, device=DEV),
                                torch.empty((2, 256), dtype=torch.bfloat16, device=DEV),
                                torch.empty(2, dtype=torch.int32, device=DEV), dh, head.ws,
                                torch.zeros(1, dtype=torch.int32, device=DEV), EPS)
        assert dh.tolist() == draft.cpu().tolist()


def test_short_chain_teacher_forced():
    c = Case(512, 3000, 1, seed=13)
    head = m.MtpDraftHead(c.g["embed"], c.g["lm_head"], c.g["eh_proj"], c.g["enorm_w"], c.g["hnorm_w"],
                          c.g["final_norm_w"], eps=EPS, max_batch=1)
    steps = 6
    hiddens = torch.stack([synth.chain_hidden(512, i + 1, "cpu") for i in range(steps)]).to(DEV)
    first = torch.tensor([17], dtype=torch.int32, device=DEV)
    drafts_graph = head.chain(first, hiddens, graph=True).cpu().view(-1).tolist()
    drafts_eager = head.chain(first, hiddens, graph=False).cpu().view(-1).tolist()
    assert drafts_graph == drafts_eager
    tok = 17
    for i in range(steps):
        out = oracle.head(c.wb, [tok], _bits(hiddens[i].cpu()), EPS)
        check_draft(drafts_graph[i], None, out["logits"][0], TOL_BF16)
        tok = drafts_graph[i]  # teacher-forced: the oracle follows the GPU's token


@pytest.mark.parametrize("H", [6144, 2048, 96])
def test_fp8_every_code_including_subnormals(H):
    # rows made of every finite E4M3 code (subnormals 0x01..0x07 included) with unit-ish scales:
    # the logits depend on each code's exact value, so a decode that lost subnormals would show
    V = 300
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    rng = np.random.default_rng(H)
    Q = codes[rng.integers(0, codes.size, (V, H))].astype(np.uint8)
    Q[0] = 0x01          # a row of only the smallest subnormal
    Q[1, ::2] = 0x07     # the largest subnormal, alternating with zero
    Q[1, 1::2] = 0x00
    s = rng.uniform(0.5, 2.0, V).astype(np.float32)
    x = synth._normal_bf16((1, H), 0.0, 1.0, torch.Generator().manual_seed(H), "cpu")
    fw = synth._normal_bf16((H,), 1.0, 0.1, torch.Generator().manual_seed(H + 1), "cpu")
    xhat = oracle.final_norm(_bits(x), _bits(fw), EPS)
    ref = oracle.logits(1, Q, s, xhat).reshape(1, -1)
    ws = m.workspace(1, H, V, DEV)
    logits = torch.empty((1, V), dtype=torch.float32, device=DEV)
    draft = torch.empty(1, dtype=torch.int32, device=DEV)
    m.mtp_head_logits_argmax(x.to(DEV), fw.to(DEV), torch.from_numpy(Q).to(DEV), torch.from_numpy(s).to(DEV),
                             m.W_FP8_E4M3, logits, draft, ws)
    torch.cuda.synchronize()
    lg = logits.cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(lg, ref, rtol=1e-4, atol=1e-6 * np.abs(ref).max())
    assert lg[0, 0] != 0.0 and lg[0, 1] != 0.0
    check_logits_and_draft(logits.cpu().numpy(), draft.cpu().numpy(), ref, TOL_FP8)


@pytest.mark.parametrize("H,B", [(6144, 16), (1024, 6), (2048, 8), (96, 9), (1024, 2)])
def test_whole_step_input_is_the_context_row_path(H, B):
    """With a full-size workspace, the whole-step entry point runs 2..16 sequences at H % 32 == 0
    through the context-row path (concat kernel + tcgen05 GEMM): its x must equal
    mtp_head_context_rows's bit for bit -- including the zero row of an out-of-range token -- with
    the same status, and lie within that path's band of the oracle."""
    c = Case(H, 700, B, seed=H + 3 * B)
    tokens = c.tokens.clone()
    tokens[B // 2] = c.V + 5
    assert c.ws.numel() >= m.mtp_head_workspace_bytes(B, H, c.V)
    x_cr = torch.full((B, H), 7, dtype=torch.bfloat16, device=DEV)
    st_cr = torch.zeros(1, dtype=torch.int32, device=DEV)
    m.mtp_head_context_rows(c.g["embed"], c.g["enorm_w"], c.g["hnorm_w"], c.g["eh_proj"], tokens.to(DEV),
                            c.hidden.to(DEV), x_cr, m.context_workspace(B, H, DEV), st_cr, EPS)
    x_fw = torch.full((B, H), 7, dtype=torch.bfloat16, device=DEV)
    d = torch.empty(B, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    m.mtp_head_forward_batched(c.g["embed"], c.g["enorm_w"], c.g["hnorm_w"], c.g["eh_proj"], c.g["final_norm_w"],
                               c.g["lm_head"], None, m.W_BF16, tokens.to(DEV), c.hidden.to(DEV), x_fw, None, d,
                               c.ws, st, EPS)
    torch.cuda.synchronize()
    assert int(st.item()) == m.ERR_TOKEN_RANGE and int(st_cr.item()) == m.ERR_TOKEN_RANGE
    assert torch.equal(x_fw.view(torch.int16), x_cr.view(torch.int16))
    assert bool((x_fw[B // 2].view(torch.int16) == 0).all())
    x_ref, concat, _, sums = oracle.input_stage(c.wb["embed"], c.wb["enorm_w"], c.wb["hnorm_w"], c.wb["eh_proj"],
                                                _bits(tokens).astype(np.int64), _bits(c.hidden), EPS,
                                                return_concat=True, return_sums=True)
    n_diff = check_x(_bits(x_fw), x_ref, sums, abs_product_sums(c.wb["eh_proj"], concat), step_x_band(H, B))
    assert n_diff <= max(1, x_ref.size // 100)


@pytest.mark.parametrize("H,B", [(520, 3), (1000, 16), (2056, 2)])
def test_whole_step_input_without_the_gemm_shape(H, B):
    """H not a multiple of 32: the whole-step entry point runs the kernels of
    mtp_head_input_batched even with a full-size workspace, so x is theirs bit for bit."""
    c = Case(H, 900, B, seed=H + B)
    x_in, st_in = c.input_gpu()
    x_fw = torch.full((B, H), 7, dtype=torch.bfloat16, device=DEV)
    d = torch.empty(B, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    m.mtp_head_forward_batched(c.g["embed"], c.g["enorm_w"], c.g["hnorm_w"], c.g["eh_proj"], c.g["final_norm_w"],
                               c.g["lm_head"], None, m.W_BF16, c.tokens.to(DEV), c.hidden.to(DEV), x_fw, None, d,
                               c.ws, st, EPS)
    torch.cuda.synchronize()
    assert st_in == 0 and int(st.item()) == 0
    assert torch.equal(x_fw.view(torch.int16), x_in.view(torch.int16))


# (256, 3): moves as kernels, the small kernel after the sweep hands the drafts back; (4096, 1):
# the register-resident sweep's last CTA hands the draft and the status back itself; (100, 1):
# B * H % 8 != 0, copy operations
@pytest.mark.parametrize("H,B", [(256, 3), (4096, 1), (100, 1)])
@pytest.mark.parametrize("fp8", [False, True])
def test_host_forward_graph_replays_match_device_path(fp8, H, B):
    """On a non-default stream the host-buffer step runs directly on the first call, then replays
    a recorded CUDA graph around mapped staging buffers: every call must give the draft the device
    path gives for its own inputs (fresh host buffers each call), and a bad token must still come
    back as the returned status."""
    V = 4096
    c = Case(H, V, B, seed=21)
    head = m.MtpDraftHead(c.g["embed"], c.g["lm_head"], c.g["eh_proj"], c.g["enorm_w"], c.g["hnorm_w"],
                          c.g["final_norm_w"], eps=EPS, max_batch=B)
    assert head.quantize_fp8() == 0
    W, s, wt = head._head(fp8)
    stream = torch.cuda.Stream()
    td = torch.empty(B, dtype=torch.int32, device=DEV)
    hd = torch.empty((B, H), dtype=torch.bfloat16, device=DEV)
    xd = torch.empty((B, H), dtype=torch.bfloat16, device=DEV)
    dd = torch.empty(B, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    for step in range(5):
        tokens, hidden = synth.make_step_inputs(H, V, B, 500 + step, "cpu")
        if step == 4:
            tokens[B - 1] = V + 1
        th, hh = tokens.pin_memory(), hidden.pin_memory()
        dh = torch.full((B,), -9, dtype=torch.int32).pin_memory()
        args = (head.embed, head.enorm_w, head.hnorm_w, head.eh_proj, head.final_norm_w, W, s, wt, th, hh,
                td, hd, xd, dd, dh, head.ws, st, EPS, stream)
        if step < 4:
            m.mtp_head_forward_host(*args)
            _, _, draft = head.forward(tokens.to(DEV), hidden.to(DEV), fp8=fp8)
            torch.cuda.synchronize()
            assert dh.tolist() == draft.cpu().tolist(), step
        else:
            with pytest.raises(m.MTPError) as e:
                m.mtp_head_forward_host(*args)
            assert e.value.code == m.ERR_TOKEN_RANGE


def test_prepared_host_step_matches_device_path():
    """MtpDraftHead.host_step binds the device buffers once; each call passes host buffers (as
    tensors or addresses) and must give the device path's draft."""
    H, V, B = 512, 3000, 2
    c = Case(H, V, B, seed=23)
    head = m.MtpDraftHead(c.g["embed"], c.g["lm_head"], c.g["eh_proj"], c.g["enorm_w"], c.g["hnorm_w"],
                          c.g["final_norm_w"], eps=EPS, max_batch=B)
    step = head.host_step(B, stream=torch.cuda.Stream())
    dh = torch.empty(B, dtype=torch.int32).pin_memory()
    for i in range(4):
        tokens, hidden = synth.make_step_inputs(H, V, B, 900 + i, "cpu")
        th, hh = tokens.pin_memory(), hidden.pin_memory()
        if i % 2:
            step(th.data_ptr(), hh.data_ptr(), dh.data_ptr())
        else:
            step(th, hh, dh)
        _, _, draft = head.forward(tokens.to(DEV), hidden.to(DEV))
        torch.cuda.synchronize()
        assert dh.tolist() == draft.cpu().tolist()
