"""Bounded device waits, made to run out on purpose (no fault, no hang).

Every wait of the kernels on a shared-memory barrier gives up after a limit, stores
MTP_ERR_TIMEOUT in the caller's status word, lets the kernel's own copies in flight land and
returns. Here the limit is first set to 1 ns, so the stage waits of the single-sequence input
stage, the single-sequence sweep and the 16-sequence tensor-core sweep run out whenever their
weight data is not already there (a call whose waits never came up short returns the normal
results instead), then to 0, where every stage wait gives up at once. A call that gave up must
report MTP_ERR_TIMEOUT and return, the output stage's workspace must be back at zero (the
completion counter and the row hand-out counter), and with the default limit restored the next
calls on the same workspace must give the same x, logits and drafts as before, bit for bit."""
import pytest
import torch

import mtp_speculative_draft_head_gb300 as m
import synth

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
EPS = synth.EPS


def _header_is_zero(ws):
    words = ws[:128].view(torch.int32).cpu()
    return int(words[0]) == 0 and int(words[16]) == 0  # completion counter, row hand-out counter


def test_waits_that_run_out_report_timeout_and_leave_the_workspace_ready():
    torch.cuda.synchronize()
    # output stage: one sequence (register-resident xhat kernel) and 16 (tensor-core kernel)
    H, V = 4096, 131072
    w = synth.make_weights(H, V, 9, DEV)
    head = m.MtpDraftHead(w.embed, w.lm_head, w.eh_proj, w.enorm_w, w.hnorm_w, w.final_norm_w, eps=EPS,
                          max_batch=16)
    assert head.quantize_fp8() == 0
    xs = {B: synth._normal_bf16((B, H), 0.0, 1.0, torch.Generator(device=DEV).manual_seed(B), DEV) for B in (1, 16)}
    # input stage, one sequence, at the GLM hidden size (its stages are two 8 KB chunks per warp)
    Hi, Vi = 6144, 4096
    wi = synth.make_weights(Hi, Vi, 9, DEV)
    tok, hid = synth.make_step_inputs(Hi, Vi, 1, 9, DEV)

    def out_stage(B, fp8, status):
        return head.logits_argmax(xs[B], fp8=fp8, logits=True, status=status)

    def in_stage(status):
        x = torch.empty((1, Hi), dtype=torch.bfloat16, device=DEV)
        m.mtp_head_input_batched(wi.embed, wi.enorm_w, wi.hnorm_w, wi.eh_proj, tok, hid, x, status, EPS)
        return x

    cases = [(B, fp8) for B in (1, 16) for fp8 in (False, True)]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ref = {c: out_stage(*c, st) for c in cases}
    ref_x = in_stage(st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0

    def run_all(limit_ns):
        codes = {}
        prev = m.mtp_head_set_wait_limit_ns(limit_ns)
        try:
            for c in cases:
                st.zero_()
                lg, d = out_stage(*c, st)
                torch.cuda.synchronize()
                codes[c] = int(st.item())
                assert _header_is_zero(head.ws), c
                if codes[c] == 0:
                    # no wait gave up (the data was always there in time): the results stand
                    assert torch.equal(lg.view(torch.int32), ref[c][0].view(torch.int32)), c
                    assert torch.equal(d, ref[c][1]), c
            st.zero_()
            x = in_stage(st)
            torch.cuda.synchronize()
            codes["input"] = int(st.item())
            if codes["input"] == 0:
                assert torch.equal(x, ref_x)
        finally:
            assert m.mtp_head_set_wait_limit_ns(prev) == limit_ns
        assert all(v in (0, m.ERR_TIMEOUT) for v in codes.values()), codes
        return codes

    # 1 ns: the waits that find their data missing run out. Whether a given call meets such a wait
    # depends on timing (the device clock the limit is compared with advances about once a
    # microsecond, and a kernel whose rings stay ahead of its warps never waits that long); the
    # tensor-core sweeps, whose stages pass between producer, builder and consumer warps, have
    # met one in every run so far. Calls that never came up short returned exact results above.
    codes = run_all(1)
    assert codes[(16, False)] == m.ERR_TIMEOUT or codes[(16, True)] == m.ERR_TIMEOUT, codes
    # 0: every stage wait gives up at once
    codes = run_all(0)
    assert all(v == m.ERR_TIMEOUT for v in codes.values()), codes

    st.zero_()
    again = {c: out_stage(*c, st) for c in cases}
    x = in_stage(st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for c in cases:
        assert torch.equal(again[c][0].view(torch.int32), ref[c][0].view(torch.int32)), c
        assert torch.equal(again[c][1], ref[c][1]), c
    assert torch.equal(x, ref_x)
