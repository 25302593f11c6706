"""ctypes binding of libmtphead.so (include/mtp_head.h): argument marshalling only.

Each function has the name of the C entry point it calls and takes torch tensors where the C
function takes device (or host) pointers: the binding passes ``tensor.data_ptr()``, the
current CUDA stream (or the one given) and the sizes, and raises ``MTPError`` when the C call
returns a nonzero status. Every step of the computation runs in the library's CUDA kernels;
there is no fallback. If the shared library cannot be built or loaded, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

W_BF16 = 0
W_FP8_E4M3 = 1

OK = 0
ERR_ARG = -1
ERR_SHAPE = -2
ERR_ALIGN = -3
ERR_WORKSPACE = -4
ERR_CUDA = -5
ERR_NONFINITE = -6
ERR_TOKEN_RANGE = -7
ERR_NOT_IMPLEMENTED = -8
ERR_TIMEOUT = -9

# name -> (restype, argtypes); mirrors include/mtp_head.h
P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "mtp_head_input_batched": (I, [P, P, P, P, P, P, P, P, I, I, I, F, P]),
    "mtp_head_input": (I, [P, P, P, P, P, P, P, P, I, I, F, P]),
    "mtp_head_logits_argmax_batched": (I, [P, P, P, P, I, P, P, P, P, Z, I, I, I, F, P]),
    "mtp_head_logits_argmax": (I, [P, P, P, P, I, P, P, P, P, Z, I, I, F, P]),
    "mtp_head_logits_argmax_batched_noalloc": (I, [P, P, P, P, I, P, P, P, I, I, I, F, P]),
    "mtp_head_workspace_bytes": (Z, [I, I, I]),
    "mtp_head_forward_batched": (I, [P, P, P, P, P, P, P, I, P, P, P, P, P, P, P, Z, I, I, I, F, P]),
    "mtp_head_forward_host": (I, [P, P, P, P, P, P, P, I, P, P, P, P, P, P, P, P, P, Z, I, I, I, F, P]),
    "mtp_head_forward_host_args": (I, [P, P, P, P]),
    "mtp_head_quantize_fp8": (I, [P, P, P, P, I, I, P]),
    "mtp_head_context_rows": (I, [P, P, P, P, P, P, P, P, P, Z, I, I, I, F, P]),
    "mtp_head_context_workspace_bytes": (Z, [I, I]),
    "mtp_head_logits_argmax_shard": (I, [P, P, P, P, I, I, I, P, P, P, P, P, Z, I, I, F, P]),
    "mtp_head_pick_combine": (I, [P, I, I, P, P, P]),
    "mtp_head_pick_key": (ctypes.c_int64, [F, ctypes.c_int32]),
    "mtp_head_pick_index": (ctypes.c_int32, [ctypes.c_int64]),
    "mtp_head_pick_value": (F, [ctypes.c_int64]),
    "mtp_head_set_wait_limit_ns": (ctypes.c_ulonglong, [ctypes.c_ulonglong]),
    "mtp_head_strerror": (ctypes.c_char_p, [I]),
}

_lib = None
_lock = threading.Lock()


class MTPError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: status {code}: {strerror(code)}")


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) libmtphead.so and declare its signatures."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        lib_path = path or _build.build()
        if not os.path.exists(lib_path):
            raise RuntimeError(f"libmtphead.so not found at {lib_path}")
        lib = ctypes.CDLL(lib_path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib


def mtp_head_set_wait_limit_ns(ns: int) -> int:
    """Give-up time (ns) of the kernels' stage waits for later launches; returns the previous
    one. ns = 0: every stage wait gives up at once (the error path on demand)."""
    return int(load().mtp_head_set_wait_limit_ns(int(ns)))


def strerror(code: int) -> str:
    return load().mtp_head_strerror(int(code)).decode()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _dev(t, name):
    if t is not None and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    return _ptr(t)


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(code: int, where: str) -> int:
    if code != OK:
        raise MTPError(code, where)
    return code


def mtp_head_workspace_bytes(B: int, H: int, V: int) -> int:
    return int(load().mtp_head_workspace_bytes(B, H, V))


def workspace(B: int, H: int, V: int, device=None) -> torch.Tensor:
    """A zero-filled workspace tensor for the output stage (reusable across calls)."""
    n = mtp_head_workspace_bytes(B, H, V)
    if n == 0:
        raise MTPError(ERR_SHAPE, "workspace")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def mtp_head_input_batched(embed, enorm_w, hnorm_w, eh_proj, tokens, target_hidden, x_out,
                           status=None, eps: float = 1e-6, stream=None) -> None:
    V, H = embed.shape
    B = tokens.numel()
    _check(load().mtp_head_input_batched(
        _dev(embed, "embed"), _dev(enorm_w, "enorm_w"), _dev(hnorm_w, "hnorm_w"),
        _dev(eh_proj, "eh_proj"), _dev(tokens, "tokens"), _dev(target_hidden, "target_hidden"),
        _dev(x_out, "x_out"), _dev(status, "status"), B, H, V, eps, _stream(stream)),
        "mtp_head_input_batched")


def mtp_head_context_workspace_bytes(R: int, H: int) -> int:
    return int(load().mtp_head_context_workspace_bytes(R, H))


def context_workspace(R: int, H: int, device=None) -> torch.Tensor:
    """Scratch for mtp_head_context_rows (no initialisation needed)."""
    n = mtp_head_context_workspace_bytes(R, H)
    if n == 0:
        raise MTPError(ERR_SHAPE, "context_workspace")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def mtp_head_context_rows(embed, enorm_w, hnorm_w, eh_proj, tokens, target_hidden, x_out, ws=None,
                          status=None, eps: float = 1e-6, stream=None) -> None:
    V, H = embed.shape
    R = tokens.numel()
    _check(load().mtp_head_context_rows(
        _dev(embed, "embed"), _dev(enorm_w, "enorm_w"), _dev(hnorm_w, "hnorm_w"),
        _dev(eh_proj, "eh_proj"), _dev(tokens, "tokens"), _dev(target_hidden, "target_hidden"),
        _dev(x_out, "x_out"), _dev(status, "status"), _dev(ws, "workspace"),
        0 if ws is None else ws.numel() * ws.element_size(), R, H, V, eps, _stream(stream)),
        "mtp_head_context_rows")


def mtp_head_input(embed, enorm_w, hnorm_w, eh_proj, token, target_hidden, x_out, status=None,
                   eps: float = 1e-6, stream=None) -> None:
    V, H = embed.shape
    _check(load().mtp_head_input(
        _dev(embed, "embed"), _dev(enorm_w, "enorm_w"), _dev(hnorm_w, "hnorm_w"),
        _dev(eh_proj, "eh_proj"), _dev(token, "token"), _dev(target_hidden, "target_hidden"),
        _dev(x_out, "x_out"), _dev(status, "status"), H, V, eps, _stream(stream)),
        "mtp_head_input")


def mtp_head_logits_argmax_batched(x, final_norm_w, lm_head, row_scale, w_dtype: int, logits,
                                   draft, ws, status=None, eps: float = 1e-6, stream=None) -> None:
    V, H = lm_head.shape
    B = draft.numel()
    _check(load().mtp_head_logits_argmax_batched(
        _dev(x, "x"), _dev(final_norm_w, "final_norm_w"), _dev(lm_head, "lm_head"),
        _dev(row_scale, "row_scale"), int(w_dtype), _dev(logits, "logits"), _dev(draft, "draft"),
        _dev(status, "status"), _dev(ws, "workspace"), ws.numel() * ws.element_size(), B, H, V,
        eps, _stream(stream)),
        "mtp_head_logits_argmax_batched")


def mtp_head_logits_argmax(x, final_norm_w, lm_head, row_scale, w_dtype: int, logits, draft, ws,
                           status=None, eps: float = 1e-6, stream=None) -> None:
    V, H = lm_head.shape
    _check(load().mtp_head_logits_argmax(
        _dev(x, "x"), _dev(final_norm_w, "final_norm_w"), _dev(lm_head, "lm_head"),
        _dev(row_scale, "row_scale"), int(w_dtype), _dev(logits, "logits"), _dev(draft, "draft"),
        _dev(status, "status"), _dev(ws, "workspace"), ws.numel() * ws.element_size(), H, V, eps,
        _stream(stream)),
        "mtp_head_logits_argmax")


def mtp_head_logits_argmax_batched_noalloc(x, final_norm_w, lm_head, row_scale, w_dtype: int,
                                           logits, draft, status=None, eps: float = 1e-6,
                                           stream=None) -> None:
    """Output stage on the library's own fixed device scratch (no workspace argument): for
    callers that cannot allocate device memory. Calls that overlap on the GPU race on it."""
    V, H = lm_head.shape
    B = draft.numel()
    _check(load().mtp_head_logits_argmax_batched_noalloc(
        _dev(x, "x"), _dev(final_norm_w, "final_norm_w"), _dev(lm_head, "lm_head"),
        _dev(row_scale, "row_scale"), int(w_dtype), _dev(logits, "logits"), _dev(draft, "draft"),
        _dev(status, "status"), B, H, V, eps, _stream(stream)),
        "mtp_head_logits_argmax_batched_noalloc")


def mtp_head_logits_argmax_shard(x, final_norm_w, lm_head_shard, row_scale_shard, w_dtype: int, v0: int,
                                 logits, pick, draft, ws, status=None, eps: float = 1e-6, stream=None) -> None:
    """Output stage over the vocabulary rows [v0, v0 + n) (lm_head_shard holds those n rows):
    pick [B] int64 receives each sequence's exchange key; logits [B, n] and draft [B] (a global
    index) are optional."""
    n, H = lm_head_shard.shape
    B = pick.numel()
    _check(load().mtp_head_logits_argmax_shard(
        _dev(x, "x"), _dev(final_norm_w, "final_norm_w"), _dev(lm_head_shard, "lm_head_shard"),
        _dev(row_scale_shard, "row_scale_shard"), int(w_dtype), int(v0), n, _dev(logits, "logits"),
        _dev(pick, "pick"), _dev(draft, "draft"), _dev(status, "status"), _dev(ws, "workspace"),
        ws.numel() * ws.element_size(), B, H, eps, _stream(stream)),
        "mtp_head_logits_argmax_shard")


def mtp_head_pick_combine(picks, draft, value=None, stream=None) -> None:
    """draft [B] (and value [B]) from the exchange keys picks [R, B] of R vocabulary shards."""
    B = draft.numel()
    R = picks.numel() // B
    _check(load().mtp_head_pick_combine(_dev(picks, "picks"), R, B, _dev(draft, "draft"), _dev(value, "value"),
                                        _stream(stream)),
           "mtp_head_pick_combine")


def mtp_head_pick_key(value: float, index: int) -> int:
    """The exchange key of (value, global index), computed on the host."""
    return int(load().mtp_head_pick_key(float(value), int(index)))


def mtp_head_pick_index(key: int) -> int:
    return int(load().mtp_head_pick_index(int(key)))


def mtp_head_pick_value(key: int) -> float:
    return float(load().mtp_head_pick_value(int(key)))


def mtp_head_forward_batched(embed, enorm_w, hnorm_w, eh_proj, final_norm_w, lm_head, row_scale,
                             w_dtype: int, tokens, target_hidden, x, logits, draft, ws,
                             status=None, eps: float = 1e-6, stream=None) -> None:
    V, H = embed.shape
    B = tokens.numel()
    _check(load().mtp_head_forward_batched(
        _dev(embed, "embed"), _dev(enorm_w, "enorm_w"), _dev(hnorm_w, "hnorm_w"),
        _dev(eh_proj, "eh_proj"), _dev(final_norm_w, "final_norm_w"), _dev(lm_head, "lm_head"),
        _dev(row_scale, "row_scale"), int(w_dtype), _dev(tokens, "tokens"),
        _dev(target_hidden, "target_hidden"), _dev(x, "x"), _dev(logits, "logits"),
        _dev(draft, "draft"), _dev(status, "status"), _dev(ws, "workspace"),
        ws.numel() * ws.element_size(), B, H, V, eps, _stream(stream)),
        "mtp_head_forward_batched")


def mtp_head_forward_host(embed, enorm_w, hnorm_w, eh_proj, final_norm_w, lm_head, row_scale,
                          w_dtype: int, tokens_host, hidden_host, tokens_dev, hidden_dev, x_dev,
                          draft_dev, draft_host, ws, status=None, eps: float = 1e-6,
                          stream=None) -> None:
    """Synchronous draft step from host buffers (tokens_host, hidden_host, draft_host are CPU
    tensors, pinned for asynchronous copies)."""
    V, H = embed.shape
    B = tokens_host.numel()
    for t, n in ((tokens_host, "tokens_host"), (hidden_host, "hidden_host"), (draft_host, "draft_host")):
        if t.is_cuda:
            raise ValueError(f"{n} must be a host tensor")
    _check(load().mtp_head_forward_host(
        _dev(embed, "embed"), _dev(enorm_w, "enorm_w"), _dev(hnorm_w, "hnorm_w"),
        _dev(eh_proj, "eh_proj"), _dev(final_norm_w, "final_norm_w"), _dev(lm_head, "lm_head"),
        _dev(row_scale, "row_scale"), int(w_dtype), _ptr(tokens_host), _ptr(hidden_host),
        _dev(tokens_dev, "tokens_dev"), _dev(hidden_dev, "hidden_dev"), _dev(x_dev, "x_dev"),
        _dev(draft_dev, "draft_dev"), _ptr(draft_host), _dev(status, "status"),
        _dev(ws, "workspace"), ws.numel() * ws.element_size(), B, H, V, eps, _stream(stream)),
        "mtp_head_forward_host")


class _HostStepArgs(ctypes.Structure):
    """mtp_host_step_args (include/mtp_head.h), field for field."""
    _fields_ = [("embed", P), ("enorm_w", P), ("hnorm_w", P), ("eh_proj", P), ("final_norm_w", P),
                ("lm_head", P), ("row_scale", P), ("w_dtype", I), ("tokens_dev", P), ("hidden_dev", P),
                ("x_dev", P), ("draft_dev", P), ("status", P), ("workspace", P), ("workspace_bytes", Z),
                ("B", I), ("H", I), ("V", I), ("eps", F), ("stream", P)]


class HostStep:
    """mtp_head_forward_host with its device buffers bound once: a call passes only the three host
    buffers (tensors, or their addresses as ints) to mtp_head_forward_host_args, so a synchronous
    draft step costs one four-argument ctypes call on the host. The bound tensors stay referenced
    for the object's lifetime."""

    def __init__(self, embed, enorm_w, hnorm_w, eh_proj, final_norm_w, lm_head, row_scale, w_dtype: int,
                 tokens_dev, hidden_dev, x_dev, draft_dev, ws, status=None, eps: float = 1e-6, stream=None):
        V, H = embed.shape
        B = tokens_dev.numel()
        self.B, self.H, self.V = B, H, V
        self._keep = (embed, enorm_w, hnorm_w, eh_proj, final_norm_w, lm_head, row_scale, tokens_dev,
                      hidden_dev, x_dev, draft_dev, ws, status, stream)
        self._fn = load().mtp_head_forward_host_args
        self._args = _HostStepArgs(
            _dev(embed, "embed"), _dev(enorm_w, "enorm_w"), _dev(hnorm_w, "hnorm_w"), _dev(eh_proj, "eh_proj"),
            _dev(final_norm_w, "final_norm_w"), _dev(lm_head, "lm_head"), _dev(row_scale, "row_scale"),
            int(w_dtype), _dev(tokens_dev, "tokens_dev"), _dev(hidden_dev, "hidden_dev"), _dev(x_dev, "x_dev"),
            _dev(draft_dev, "draft_dev"), _dev(status, "status"), _dev(ws, "workspace"),
            ws.numel() * ws.element_size(), B, H, V, float(eps), _stream(stream))
        self._addr = ctypes.addressof(self._args)

    def __call__(self, tokens_host, hidden_host, draft_host) -> None:
        t = tokens_host if isinstance(tokens_host, int) else tokens_host.data_ptr()
        h = hidden_host if isinstance(hidden_host, int) else hidden_host.data_ptr()
        d = draft_host if isinstance(draft_host, int) else draft_host.data_ptr()
        code = self._fn(self._addr, t, h, d)
        if code != OK:
            raise MTPError(code, "mtp_head_forward_host")


def mtp_head_quantize_fp8(w, q, row_scale, status, stream=None) -> None:
    V, H = w.shape
    _check(load().mtp_head_quantize_fp8(
        _dev(w, "w"), _dev(q, "q"), _dev(row_scale, "row_scale"), _dev(status, "status"), V, H,
        _stream(stream)),
        "mtp_head_quantize_fp8")
