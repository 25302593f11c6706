"""``MtpDraftHead``: the GLM-5.3 MTP draft head on one GPU, as a thin owner of buffers around
the C ABI (include/mtp_head.h).

It mirrors the source's `Glm5NextMtpHead` ("metrale_model_arch / glm5next_mtp_head.rs"): the
weights it holds are ``embed_tokens``, ``eh_proj``, ``enorm``, ``hnorm``, ``final_norm`` and the
target's ``lm_head`` (plus the optional FP8 copy of the `head_fp8` doc); its per-sequence scratch
is the ``x`` / ``logits`` / ``draft`` buffers of the proposer state. The decoder layer between
the two stages is the identity here. Every computation is a call into libmtphead.so.
"""
from __future__ import annotations

import torch

from . import _lib
from ._lib import W_BF16, W_FP8_E4M3


class MtpDraftHead:
    def __init__(self, embed, lm_head, eh_proj, enorm_w, hnorm_w, final_norm_w, eps: float = 1e-6,
                 max_batch: int = 16):
        for name, t in (("embed", embed), ("lm_head", lm_head), ("eh_proj", eh_proj),
                        ("enorm_w", enorm_w), ("hnorm_w", hnorm_w), ("final_norm_w", final_norm_w)):
            if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous bfloat16 CUDA tensor")
        self.embed, self.lm_head, self.eh_proj = embed, lm_head, eh_proj
        self.enorm_w, self.hnorm_w, self.final_norm_w = enorm_w, hnorm_w, final_norm_w
        self.V, self.H = embed.shape
        if lm_head.shape != (self.V, self.H) or eh_proj.shape != (self.H, 2 * self.H):
            raise ValueError("shapes: embed/lm_head [V, H], eh_proj [H, 2H]")
        self.eps = float(eps)
        self.device = embed.device
        self.max_batch = max_batch
        self.lm_head_fp8 = None
        self.row_scale = None
        self.ws = _lib.workspace(max_batch, self.H, self.V, self.device)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)

    # ------------------------------------------------------------------ FP8 copy
    def quantize_fp8(self) -> int:
        """Build the E4M3 copy of lm_head with per-row FP32 scales; returns the device status
        (0, or MTP_ERR_NONFINITE when a weight is NaN/Inf -- the copy is then dropped)."""
        q = torch.empty((self.V, self.H), dtype=torch.uint8, device=self.device)
        s = torch.empty(self.V, dtype=torch.float32, device=self.device)
        st = torch.zeros(1, dtype=torch.int32, device=self.device)
        _lib.mtp_head_quantize_fp8(self.lm_head, q, s, st)
        code = int(st.item())
        if code == 0:
            self.lm_head_fp8, self.row_scale = q, s
        else:
            self.lm_head_fp8, self.row_scale = None, None
        return code

    def _head(self, fp8: bool):
        if fp8:
            if self.lm_head_fp8 is None:
                raise RuntimeError("no FP8 copy: call quantize_fp8() first")
            return self.lm_head_fp8, self.row_scale, W_FP8_E4M3
        return self.lm_head, None, W_BF16

    # ------------------------------------------------------------------ stages
    def input(self, tokens, hidden, x=None, status=None, stream=None):
        B = tokens.numel()
        x = torch.empty((B, self.H), dtype=torch.bfloat16, device=self.device) if x is None else x
        _lib.mtp_head_input_batched(self.embed, self.enorm_w, self.hnorm_w, self.eh_proj, tokens,
                                    hidden, x, status, self.eps, stream)
        return x

    def logits_argmax(self, x, fp8: bool = False, logits=True, draft=None, status=None, stream=None):
        B = x.shape[0]
        W, s, wt = self._head(fp8)
        if logits is True:
            logits = torch.empty((B, self.V), dtype=torch.float32, device=self.device)
        elif logits is False:
            logits = None
        draft = torch.empty(B, dtype=torch.int32, device=self.device) if draft is None else draft
        _lib.mtp_head_logits_argmax_batched(x, self.final_norm_w, W, s, wt, logits, draft, self.ws,
                                            status, self.eps, stream)
        return logits, draft

    def forward(self, tokens, hidden, fp8: bool = False, logits=False, x=None, draft=None,
                status=None, stream=None):
        """One draft step for B sequences (device buffers): returns (x, logits|None, draft)."""
        B = tokens.numel()
        W, s, wt = self._head(fp8)
        x = torch.empty((B, self.H), dtype=torch.bfloat16, device=self.device) if x is None else x
        if logits is True:
            logits = torch.empty((B, self.V), dtype=torch.float32, device=self.device)
        elif logits is False:
            logits = None
        draft = torch.empty(B, dtype=torch.int32, device=self.device) if draft is None else draft
        _lib.mtp_head_forward_batched(self.embed, self.enorm_w, self.hnorm_w, self.eh_proj,
                                      self.final_norm_w, W, s, wt, tokens, hidden, x, logits, draft,
                                      self.ws, status, self.eps, stream)
        return x, logits, draft

    def host_step(self, B: int = 1, fp8: bool = False, stream=None, status=None) -> "_lib.HostStep":
        """A prepared synchronous draft step from host buffers (the source's forward_one shape):
        device buffers for B sequences are allocated here and bound once; call the result with
        (tokens_host [B] int32, hidden_host [B, H] bf16, draft_host [B] int32), pinned."""
        W, s, wt = self._head(fp8)
        dev = self.device
        return _lib.HostStep(self.embed, self.enorm_w, self.hnorm_w, self.eh_proj, self.final_norm_w, W, s, wt,
                             torch.empty(B, dtype=torch.int32, device=dev),
                             torch.empty((B, self.H), dtype=torch.bfloat16, device=dev),
                             torch.empty((B, self.H), dtype=torch.bfloat16, device=dev),
                             torch.empty(B, dtype=torch.int32, device=dev), self.ws, status, self.eps, stream)

    # ------------------------------------------------------------------ draft chains
    def chain(self, first_tokens, hiddens, fp8: bool = False, graph: bool = True, status=None):
        """Draft ``steps`` tokens per sequence, each step feeding its draft (device-resident) into
        the next step's input stage: hiddens is [steps, B, H]; returns drafts [steps, B] int32.
        With ``graph`` the whole chain is captured once in a CUDA graph and replayed."""
        steps, B, _ = hiddens.shape
        tok = torch.empty((steps + 1, B), dtype=torch.int32, device=self.device)
        tok[0].copy_(first_tokens.view(-1))
        x = torch.empty((B, self.H), dtype=torch.bfloat16, device=self.device)
        W, s, wt = self._head(fp8)

        def run(stream=None):
            for i in range(steps):
                _lib.mtp_head_forward_batched(self.embed, self.enorm_w, self.hnorm_w, self.eh_proj,
                                              self.final_norm_w, W, s, wt, tok[i], hiddens[i], x,
                                              None, tok[i + 1], self.ws, status, self.eps, stream)

        if not graph:
            run()
            return tok[1:]
        g = self.capture(run)
        g.replay()
        return tok[1:]

    @staticmethod
    def capture(fn) -> torch.cuda.CUDAGraph:
        """Capture fn(stream) into a CUDA graph on a side stream (warming the launch path first)."""
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                fn(s)
        torch.cuda.current_stream().wait_stream(s)
        return g


# ---------------------------------------------------------------------- vocabulary shards
def shard_geometry(V: int, rank: int, world: int) -> tuple[int, int]:
    """(v0, n): the rows [v0, v0 + n) of lm_head that rank ``rank`` of ``world`` sweeps. As in the
    source's head ("glm5next_mtp_head.rs", `head_v0` / `head_n`): the vocabulary splits into
    ``world`` equal ranges when it divides evenly, and otherwise every rank sweeps all of it
    (``n == V``, no exchange needed)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("need 0 <= rank < world")
    if V % world != 0:
        return 0, V
    n = V // world
    return rank * n, n


def exchange_picks(picks: torch.Tensor, group=None) -> torch.Tensor:
    """The cross-rank step of the sharded head: every rank's [B] int64 exchange keys become their
    element-wise maximum on every rank -- one MAX all-reduce of 8 bytes per sequence (the keys'
    order is the argmax order, so the maximum is the pick). A no-op without a process group or on
    one rank. Runs on the process group's backend (NCCL for CUDA tensors, gloo for CPU ones)."""
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(picks, op=dist.ReduceOp.MAX, group=group)
    return picks


class VocabShard:
    """The output stage of one rank of a vocabulary-sharded head: final norm, the sweep of this
    rank's rows of lm_head (BF16, or an FP8 copy of these rows only, as in the source's
    `head_fp8` doc), the per-sequence exchange key, the exchange with the other ranks and the
    decode of the winning key into the draft. On one GPU, several shards' keys can also be
    combined directly (``mtp_head_pick_combine`` with R > 1)."""

    def __init__(self, lm_head: torch.Tensor, final_norm_w: torch.Tensor, rank: int, world: int,
                 eps: float = 1e-6, max_batch: int = 16):
        V, H = lm_head.shape
        self.V, self.H = V, H
        self.rank, self.world = rank, world
        self.v0, self.n = shard_geometry(V, rank, world)
        self.sharded = self.n != V
        self.lm_head = lm_head[self.v0:self.v0 + self.n]
        self.final_norm_w = final_norm_w
        self.eps = float(eps)
        self.device = lm_head.device
        self.lm_head_fp8 = None
        self.row_scale = None
        self.ws = _lib.workspace(max_batch, H, self.n, self.device)

    def quantize_fp8(self) -> int:
        """E4M3 copy of this shard's rows with their FP32 scales; returns the device status."""
        q = torch.empty((self.n, self.H), dtype=torch.uint8, device=self.device)
        s = torch.empty(self.n, dtype=torch.float32, device=self.device)
        st = torch.zeros(1, dtype=torch.int32, device=self.device)
        _lib.mtp_head_quantize_fp8(self.lm_head, q, s, st)
        code = int(st.item())
        self.lm_head_fp8, self.row_scale = (q, s) if code == 0 else (None, None)
        return code

    def picks(self, x, fp8: bool = False, pick=None, logits=None, status=None, stream=None) -> torch.Tensor:
        """This shard's exchange keys [B] for the block outputs x [B, H] (logits [B, n] optional)."""
        B = x.shape[0]
        if fp8 and self.lm_head_fp8 is None:
            raise RuntimeError("no FP8 copy: call quantize_fp8() first")
        W, s, wt = (self.lm_head_fp8, self.row_scale, W_FP8_E4M3) if fp8 else (self.lm_head, None, W_BF16)
        pick = torch.empty(B, dtype=torch.int64, device=self.device) if pick is None else pick
        _lib.mtp_head_logits_argmax_shard(x, self.final_norm_w, W, s, wt, self.v0, logits, pick, None, self.ws,
                                          status, self.eps, stream)
        return pick

    def draft(self, x, fp8: bool = False, group=None, draft=None, status=None, stream=None) -> torch.Tensor:
        """The draft [B] (global token ids) of the whole vocabulary: this shard's keys, the MAX
        exchange with the other ranks (when sharded), then the decode. ``stream``, if given, is a
        torch.cuda.Stream."""
        pick = self.picks(x, fp8=fp8, status=status, stream=stream)
        if self.sharded:
            # the all-reduce runs on torch's current stream: order it between the two kernels
            if stream is not None:
                torch.cuda.current_stream().wait_stream(stream)
            exchange_picks(pick, group)
            if stream is not None:
                stream.wait_stream(torch.cuda.current_stream())
        draft = torch.empty(x.shape[0], dtype=torch.int32, device=self.device) if draft is None else draft
        _lib.mtp_head_pick_combine(pick, draft, stream=stream)
        return draft
