"""GB300 (sm_103a) hot path of the GLM-5.3 MTP speculative draft head.

The computation lives in ``libmtphead.so`` (CUDA, C ABI declared in ``include/mtp_head.h``):
the fused input stage (embedding gather, enorm/hnorm RMSNorm, concat, eh_proj GEMV), the fused
output stage (shared_head.norm, lm_head vocabulary sweep in BF16 or FP8 E4M3, argmax) and the
FP8 quantiser, and the output stage over one vocabulary shard with the exact pick between
shards. ``_lib`` binds those entry points by name with ctypes; ``MtpDraftHead`` and
``VocabShard`` own buffers around them. PyTorch provides device memory, streams and (between
the ranks of a sharded head) the one MAX all-reduce of the pick keys.
"""
from ._lib import (  # noqa: F401
    ERR_ALIGN, ERR_ARG, ERR_CUDA, ERR_NONFINITE, ERR_NOT_IMPLEMENTED, ERR_SHAPE, ERR_TIMEOUT,
    ERR_TOKEN_RANGE, ERR_WORKSPACE, OK, W_BF16, W_FP8_E4M3, HostStep, MTPError, SIGNATURES, context_workspace, load,
    mtp_head_context_rows, mtp_head_context_workspace_bytes,
    mtp_head_forward_batched, mtp_head_forward_host, mtp_head_input, mtp_head_input_batched,
    mtp_head_logits_argmax, mtp_head_logits_argmax_batched,
    mtp_head_logits_argmax_batched_noalloc, mtp_head_logits_argmax_shard, mtp_head_pick_combine,
    mtp_head_pick_index, mtp_head_pick_key, mtp_head_pick_value, mtp_head_quantize_fp8,
    mtp_head_set_wait_limit_ns,
    mtp_head_workspace_bytes, strerror, workspace,
)
from .head import MtpDraftHead, VocabShard, exchange_picks, shard_geometry  # noqa: F401
