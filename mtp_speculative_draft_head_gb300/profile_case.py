"""A small, self-contained run of the draft head for profilers (ncu) and quick timing.

    python -m mtp_speculative_draft_head_gb300.profile_case [--H 6144] [--V 32768] [--B 1] [--reps 3]
    python -m mtp_speculative_draft_head_gb300.profile_case --R 512 [--H 6144] [--reps 3]

Draws seeded synthetic weights on the GPU (see synth), builds the FP8 copy, then runs `reps`
draft steps with the BF16 head and `reps` with the FP8 head (input stage + output stage each).
With --R it runs `reps` context-row input stages over R rows instead (concat + GEMM).
The default V keeps the BF16 lm_head (403 MB) above the L2 size while the whole run holds about
1.3 GB on the device, so a multi-pass profiler capture of one launch ends in seconds.
"""
import argparse
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

from . import MtpDraftHead, context_workspace, mtp_head_context_rows  # noqa: E402


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--H", type=int, default=6144)
    ap.add_argument("--V", type=int, default=32768)
    ap.add_argument("--B", type=int, default=1)
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--R", type=int, default=0)
    a = ap.parse_args()
    dev = torch.device("cuda:0")
    w = synth.make_weights(a.H, a.V, 0, dev)
    if a.R:
        tokens, hidden = synth.make_step_inputs(a.H, a.V, a.R, 2, dev, distinct=False)
        x = torch.empty((a.R, a.H), dtype=torch.bfloat16, device=dev)
        ws = context_workspace(a.R, a.H, dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        for _ in range(a.reps):
            mtp_head_context_rows(w.embed, w.enorm_w, w.hnorm_w, w.eh_proj, tokens, hidden, x, ws, status)
        torch.cuda.synchronize()
        if int(status.item()) != 0:
            raise RuntimeError(f"status {int(status.item())}")
        print("ok")
        return
    head = MtpDraftHead(w.embed, w.lm_head, w.eh_proj, w.enorm_w, w.hnorm_w, w.final_norm_w,
                        max_batch=a.B)
    if head.quantize_fp8() != 0:
        raise RuntimeError("FP8 quantisation failed")
    tokens, hidden = synth.make_step_inputs(a.H, a.V, a.B, 1, dev)
    for _ in range(a.reps):
        for fp8 in (False, True):
            head.forward(tokens, hidden, fp8=fp8)
    torch.cuda.synchronize()
    print("ok")


if __name__ == "__main__":
    main()
