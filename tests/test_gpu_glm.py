"""GPU parity at the GLM-5.3 sizes the benchmark runs (H=6144, V=154880; the adversarial case
H=4096, V=131072), in the benchmark's launch configuration. Weights are drawn on the GPU (see
synth), copied to the host, and the oracle computes the full vocabulary of logits with one
plain C loop per thread over disjoint row ranges."""
import os

import numpy as np
import pytest
import torch

import mtp_speculative_draft_head_gb300 as m
import oracle
import synth
from gpu_helpers import (TOL_BF16, TOL_FP8, abs_product_sums, check_draft, check_logits_and_draft, check_x, step_x_band,
                         x_band)

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
EPS = synth.EPS
THREADS = max(1, min(32, os.cpu_count() or 1))


def _bits(t):
    return synth.bits(t)


class Model:
    def __init__(self, H, V, seed, outliers=False):
        self.H, self.V = H, V
        self.w = synth.make_weights(H, V, seed, DEV)
        if outliers:
            self.w.lm_head = synth.add_outliers(self.w.lm_head, 0.01, 50.0, seed)
        self.wb = {k: _bits(v) for k, v in self.w.as_dict().items()}
        self.head = m.MtpDraftHead(self.w.embed, self.w.lm_head, self.w.eh_proj, self.w.enorm_w,
                                   self.w.hnorm_w, self.w.final_norm_w, eps=EPS, max_batch=16)

    def quantize(self):
        assert self.head.quantize_fp8() == 0
        self.qb = _bits(self.head.lm_head_fp8)
        self.sb = self.head.row_scale.cpu().numpy()

    def oracle_x(self, tokens, hidden):
        """(x, status, sums, sums of |products|) -- the last scales the accumulation band of x."""
        x, concat, st, sums = oracle.input_stage(self.wb["embed"], self.wb["enorm_w"], self.wb["hnorm_w"],
                                                 self.wb["eh_proj"], _bits(tokens).astype(np.int64), _bits(hidden),
                                                 EPS, return_concat=True, return_sums=True)
        return x, st, sums, abs_product_sums(self.wb["eh_proj"], concat)

    def oracle_logits(self, x_bits, fp8):
        xhat = oracle.final_norm(x_bits, self.wb["final_norm_w"], EPS)
        if fp8:
            return oracle.logits(1, self.qb, self.sb, xhat, threads=THREADS).reshape(x_bits.shape[0], -1)
        return oracle.logits(0, self.wb["lm_head"], None, xhat, threads=THREADS).reshape(x_bits.shape[0], -1)


@pytest.fixture(scope="module")
def glm():
    md = Model(6144, 154880, 0)
    md.quantize()
    yield md
    del md
    torch.cuda.empty_cache()


def test_glm_quantizer_sampled_rows_bitexact(glm):
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, glm.V - 1], rng.integers(0, glm.V, 512)]))
    q_ref, s_ref, st = oracle.quantize(glm.wb["lm_head"][rows])
    assert st == 0
    assert np.array_equal(glm.qb[rows], q_ref)
    assert np.array_equal(glm.sb[rows].view(np.uint32), s_ref.view(np.uint32))


@pytest.mark.parametrize("B", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("fp8", [False, True])
def test_glm_head(glm, B, fp8):
    seed = 1 if B == 1 else 1000 + B
    tokens, hidden = synth.make_step_inputs(glm.H, glm.V, B, seed, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    x, logits, draft = glm.head.forward(tokens, hidden, fp8=fp8, logits=True, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    x_ref, st, sums, abs_sums = glm.oracle_x(tokens, hidden)
    assert np.all(st == 0)
    n_diff = check_x(_bits(x), x_ref, sums, abs_sums, step_x_band(glm.H, B))
    # the band is a worst-case bound; the FP32 runs differ from the exact sum far more rarely
    assert n_diff <= max(1, x_ref.size // 100)
    ref = glm.oracle_logits(x_ref, fp8)
    err = check_logits_and_draft(logits.cpu().numpy(), draft.cpu().numpy(), ref, TOL_FP8 if fp8 else TOL_BF16)
    assert err < 5e-3


@pytest.mark.parametrize("fp8", [False, True])
def test_glm_chain_1000_teacher_forced(glm, fp8):
    """The 1000-token chain: each step feeds its draft (device-resident) into the next. The graph
    replay and an eager run of the same 1000 steps must give the same drafts at every step; 33
    evenly spaced steps are checked against the oracle, fed the token the GPU used (teacher
    forcing), and on four of them the full logits of that step are compared element by element."""
    steps = 1000
    hiddens = torch.cat([synth.chain_hidden(glm.H, i + 1, DEV) for i in range(steps)]).view(steps, 1, glm.H)
    first = synth.chain_first_token(glm.V, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    drafts = glm.head.chain(first, hiddens, fp8=fp8, graph=True, status=status).cpu().view(-1).numpy()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.all((drafts >= 0) & (drafts < glm.V))
    eager = glm.head.chain(first, hiddens, fp8=fp8, graph=False, status=status).cpu().view(-1).numpy()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(eager, drafts), f"first differing step {int(np.nonzero(eager != drafts)[0][0])}"
    toks = np.concatenate([first.cpu().numpy(), drafts])
    checked = sorted(set(range(0, steps, 31)) | {steps - 1})
    assert len(checked) >= 32
    with_logits = set(checked[::len(checked) // 4][:4])
    tol = TOL_FP8 if fp8 else TOL_BF16
    for i in checked:
        tok = torch.tensor([int(toks[i])], dtype=torch.int32, device=DEV)
        xr, _ = oracle.input_stage(glm.wb["embed"], glm.wb["enorm_w"], glm.wb["hnorm_w"], glm.wb["eh_proj"],
                                   [int(toks[i])], _bits(hiddens[i]), EPS)
        ref = glm.oracle_logits(xr, fp8)
        if i in with_logits:
            # the same step again with the logits stored: its draft is the chain's, bit for bit
            x, logits, d = glm.head.forward(tok, hiddens[i], fp8=fp8, logits=True, status=status)
            torch.cuda.synchronize()
            assert int(status.item()) == 0
            assert int(d.item()) == int(drafts[i])
            check_logits_and_draft(logits.cpu().numpy(), d.cpu().numpy(), ref, tol)
        else:
            check_draft(int(drafts[i]), None, ref[0], tol)


def test_adversarial_ties_and_outliers():
    H, V, seed = 4096, 131072, 7
    md = Model(H, V, seed, outliers=True)
    tokens, hidden = synth.make_step_inputs(H, V, 1, seed, DEV)
    hidden = synth.hidden_with_outlier_channels(hidden, 5, 100.0, seed)
    x_ref, _, sums, abs_sums = md.oracle_x(tokens, hidden)
    xhat = oracle.final_norm(x_ref, md.wb["final_norm_w"], EPS)[0]
    rows = synth.pick_rows(V, 64, seed, DEV)
    md.w.lm_head = synth.plant_rows(md.w.lm_head, rows, torch.from_numpy(oracle.bf16_to_f64(xhat)))
    md.wb["lm_head"] = _bits(md.w.lm_head)
    md.head.lm_head = md.w.lm_head
    md.quantize()
    planted = sorted(rows.cpu().tolist())
    for fp8 in (False, True):
        x, logits, draft = md.head.forward(tokens, hidden, fp8=fp8, logits=True)
        torch.cuda.synchronize()
        n_diff = check_x(_bits(x), x_ref, sums, abs_sums, x_band(H, 1))
        assert n_diff <= max(1, x_ref.size // 100)
        lg = logits.cpu().view(-1)
        assert len(set(lg[planted].view(torch.int32).tolist())) == 1
        assert int(draft.item()) == planted[0]
        ref = md.oracle_logits(x_ref, fp8)
        check_logits_and_draft(logits.cpu().numpy(), draft.cpu().numpy(), ref, TOL_FP8 if fp8 else TOL_BF16)
