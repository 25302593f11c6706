"""Seeded synthetic inputs for the MTP draft head.

Shared by the oracle tests, the GPU parity tests and the benchmark. This module draws
random numbers and lays out tensors; it holds none of the head's arithmetic (no norm, no
projection, no argmax, no quantisation). Every tensor is BF16 (weights, hidden states) or
int32 (tokens) and is drawn with ``torch.Generator`` on the requested device:

* the small workload (H=256, V=4096) is drawn on the CPU, so it is the same on every host;
* the GLM-scale workloads (H=6144, V=154880 and H=4096, V=131072; 1.9 GB tables) are drawn
  on the GPU with torch's CUDA generator, because host generation of 2e9 normals takes
  minutes. Host copies for the oracle are then made from those device tensors.

Value recipe (the GLM-5.3 head's shapes; the distributions are synthetic):
  embed [V, H], lm_head [V, H], eh_proj [H, 2H]   ~ N(0, 0.02)
  enorm_w, hnorm_w, final_norm_w [H]               ~ 1 + N(0, 0.1)
  target_hidden [B, H]                             ~ N(0, 1)
  token                                            ~ U[0, V)  (distinct across a batch)
  eps = 1e-6
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

EPS = 1e-6

# Workloads by name (sizes from the GLM-5.3 head; B is per sweep).
WORKLOADS = {
    "tiny": dict(H=256, V=4096, B=1, seed=0),
    "glm": dict(H=6144, V=154880, B=1, seed=0),
    "adversarial": dict(H=4096, V=131072, B=1, seed=7),
}

# Independent random streams derived from one seed.
_STREAM_WEIGHTS = 0
_STREAM_OUTLIERS = 1
_STREAM_PLANT = 2
_STREAM_HIDDEN_OUTLIERS = 3


def _gen(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1_000_003 + stream)
    return g


def _normal_bf16(shape, mean: float, std: float, g: torch.Generator, device) -> torch.Tensor:
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return (t * std + mean).to(torch.bfloat16)


@dataclass
class Weights:
    embed: torch.Tensor      # [V, H] bf16
    lm_head: torch.Tensor    # [V, H] bf16
    eh_proj: torch.Tensor    # [H, 2H] bf16
    enorm_w: torch.Tensor    # [H] bf16
    hnorm_w: torch.Tensor    # [H] bf16
    final_norm_w: torch.Tensor  # [H] bf16

    @property
    def H(self) -> int:
        return self.embed.shape[1]

    @property
    def V(self) -> int:
        return self.embed.shape[0]

    def as_dict(self) -> dict:
        return dict(embed=self.embed, lm_head=self.lm_head, eh_proj=self.eh_proj,
                    enorm_w=self.enorm_w, hnorm_w=self.hnorm_w, final_norm_w=self.final_norm_w)


def make_weights(H: int, V: int, seed: int, device="cpu") -> Weights:
    g = _gen(seed, _STREAM_WEIGHTS, device)
    embed = _normal_bf16((V, H), 0.0, 0.02, g, device)
    lm_head = _normal_bf16((V, H), 0.0, 0.02, g, device)
    eh_proj = _normal_bf16((H, 2 * H), 0.0, 0.02, g, device)
    enorm_w = _normal_bf16((H,), 1.0, 0.1, g, device)
    hnorm_w = _normal_bf16((H,), 1.0, 0.1, g, device)
    final_norm_w = _normal_bf16((H,), 1.0, 0.1, g, device)
    return Weights(embed, lm_head, eh_proj, enorm_w, hnorm_w, final_norm_w)


def make_step_inputs(H: int, V: int, B: int, seed: int, device="cpu", distinct: bool = True):
    """Tokens [B] int32 (uniform in [0, V), distinct when asked) and target_hidden [B, H]."""
    g = _gen(seed, _STREAM_WEIGHTS, device)
    if distinct and B <= V:
        tokens = torch.randperm(V, generator=g, device=device)[:B]
    else:
        tokens = torch.randint(0, V, (B,), generator=g, device=device)
    hidden = _normal_bf16((B, H), 0.0, 1.0, g, device)
    return tokens.to(torch.int32), hidden


def chain_hidden(H: int, step: int, device="cpu") -> torch.Tensor:
    """target_hidden for draft step ``step`` (1-based) of the 1000-token chain: seed = step."""
    g = _gen(step, _STREAM_WEIGHTS, device)
    return _normal_bf16((1, H), 0.0, 1.0, g, device)


def chain_first_token(V: int, device="cpu") -> torch.Tensor:
    """First token of the chain: uniform in [0, V) from seed 1."""
    g = _gen(1, _STREAM_PLANT, device)
    return torch.randint(0, V, (1,), generator=g, device=device).to(torch.int32)


def add_outliers(W: torch.Tensor, frac: float, factor: float, seed: int) -> torch.Tensor:
    """Return a copy of W with a uniformly chosen ``frac`` of its elements scaled by
    ``factor`` (BF16 rounding of the scaled value)."""
    g = _gen(seed, _STREAM_OUTLIERS, W.device)
    mask = torch.rand(W.shape, generator=g, device=W.device) < frac
    out = W.clone()
    out[mask] = (W[mask].float() * factor).to(torch.bfloat16)
    return out


def pick_rows(V: int, n: int, seed: int, device="cpu") -> torch.Tensor:
    """n distinct row indices, uniform without replacement, sorted ascending."""
    g = _gen(seed, _STREAM_PLANT, device)
    return torch.randperm(V, generator=g, device=device)[:n].sort().values


def plant_rows(W: torch.Tensor, rows: torch.Tensor, sign_pattern: torch.Tensor,
               magnitude: float = 0.05) -> torch.Tensor:
    """Return a copy of W whose ``rows`` all equal bf16(magnitude * sign(sign_pattern)).

    Identical rows give identical logits, so they tie exactly; with the sign pattern of the
    head's own normalised input they are also the largest logits. The sign pattern is passed
    in by the caller, so this module computes nothing of the head itself.
    """
    out = W.clone()
    row = (torch.sign(sign_pattern.float()) * magnitude).to(torch.bfloat16).to(W.device)
    out[rows.to(W.device)] = row
    return out


def hidden_with_outlier_channels(hidden: torch.Tensor, n_channels: int, magnitude: float,
                                 seed: int) -> torch.Tensor:
    """Set n distinct channels of every row to +-magnitude (random sign)."""
    g = _gen(seed, _STREAM_HIDDEN_OUTLIERS, "cpu")
    H = hidden.shape[-1]
    ch = torch.randperm(H, generator=g)[:n_channels]
    sign = torch.where(torch.rand(n_channels, generator=g) < 0.5, -1.0, 1.0)
    out = hidden.clone()
    out[..., ch.to(hidden.device)] = (sign * magnitude).to(torch.bfloat16).to(hidden.device)
    return out


def bits(t: torch.Tensor):
    """Host numpy view of a tensor's raw bits (bf16 -> uint16, fp8 codes -> uint8)."""
    import numpy as np
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return t.view(torch.uint8).numpy()
    return t.numpy()
