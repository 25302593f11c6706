"""The output stage's no-allocation entry point, through the C ABI.

mtp_head_logits_argmax_batched_noalloc is for callers of this library that cannot allocate
device memory (a plug-in that only gets the buffers its host hands it, a process whose device
memory another allocator has already claimed): it keeps the output stage's small workspace in
a fixed array inside the library instead of taking one from the caller. Here it must give the
same logits (bit for bit) and drafts as mtp_head_logits_argmax_batched with a caller-provided
workspace, on two calls in a row (the second call reuses the array the first one left behind).

This file is collected last on purpose, and needs nothing from the other test files.
"""
import ctypes

import numpy as np
import pytest
import torch

import mtp_speculative_draft_head_gb300 as m
import synth
from gpu_helpers import TOL_BF16, TOL_FP8

DEV = "cuda:0"


def _raw_noalloc(lib, x, fw, W, s, wt, logits, draft, status, B, H, V):
    P = lambda t: None if t is None else t.data_ptr()
    return lib.mtp_head_logits_argmax_batched_noalloc(
        P(x), P(fw), P(W), P(s), wt, P(logits), P(draft), P(status), B, H, V, ctypes.c_float(synth.EPS),
        torch.cuda.current_stream().cuda_stream)


def test_noalloc_rejects_batches_beyond_its_scratch():
    lib = m.load()
    A = 0x10000  # never dereferenced: the size check comes first
    for B in (0, 17, 64):
        assert lib.mtp_head_logits_argmax_batched_noalloc(A, A, A, None, m.W_BF16, None, A, None, B, 64,
                                                          100, ctypes.c_float(1e-6), None) == m.ERR_SHAPE


@pytest.mark.gpu
@pytest.mark.parametrize("H,V,B", [(6144, 20000, 1), (2048, 7777, 3), (512, 3000, 16)])
@pytest.mark.parametrize("fp8", [False, True])
def test_noalloc_matches_workspace_entry_point_twice(H, V, B, fp8):
    lib = m.load()
    w = synth.make_weights(H, V, 5, "cpu")
    g = {k: v.to(DEV) for k, v in w.as_dict().items()}
    x = synth._normal_bf16((B, H), 0.0, 1.0, torch.Generator().manual_seed(H + B), "cpu").to(DEV)
    if fp8:
        W = torch.empty((V, H), dtype=torch.uint8, device=DEV)
        s = torch.empty(V, dtype=torch.float32, device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        m.mtp_head_quantize_fp8(g["lm_head"], W, s, st)
        wt, tol = m.W_FP8_E4M3, TOL_FP8
    else:
        W, s, wt, tol = g["lm_head"], None, m.W_BF16, TOL_BF16
    # reference: the workspace entry point
    ws = m.workspace(B, H, V, DEV)
    ref_logits = torch.empty((B, V), dtype=torch.float32, device=DEV)
    ref_draft = torch.empty(B, dtype=torch.int32, device=DEV)
    m.mtp_head_logits_argmax_batched(x, g["final_norm_w"], W, s, wt, ref_logits, ref_draft, ws)
    torch.cuda.synchronize()
    for _ in range(2):  # two calls in a row on the shared scratch
        logits = torch.full((B, V), float("nan"), dtype=torch.float32, device=DEV)
        draft = torch.full((B,), -5, dtype=torch.int32, device=DEV)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        assert _raw_noalloc(lib, x, g["final_norm_w"], W, s, wt, logits, draft, status, B, H, V) == m.OK
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        # the same kernels on the same inputs: the logits must agree bit for bit, not only within
        # the parity tolerance (which still bounds any difference, were there one)
        err = float((logits.double() - ref_logits.double()).abs().max())
        assert err <= tol, err
        assert torch.equal(logits.view(torch.int32), ref_logits.view(torch.int32))
        assert torch.equal(draft, ref_draft)
        lg = logits.cpu().numpy()
        for b in range(B):  # each draft is the lowest-index argmax of its own logits
            assert int(draft[b]) == int(np.argmax(lg[b]))
