"""CPU oracle for the GLM-5.3 MTP draft head -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference leg of
``bench.py`` may import this package. The CUDA library never does, and shares no code with
it. The arithmetic lives in ``mtp_oracle.c`` (plain C, fp64); this module only builds that
file with gcc, loads it with ctypes and marshals numpy arrays. BF16 values travel as their
``uint16`` bit patterns, E4M3 codes as ``uint8``.

Every function cites, in the C source, the passage of the pages it follows
("metrale_model_arch / glm5next_mtp_head.rs": module doc, ``norm``, ``forward_one``,
``head_fp8``; "glm5next_layer / mod.rs": the rms_norm_vanilla invariant).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mtp_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libmtporacle.so")

OK = 0
ERR_NONFINITE = -6
ERR_TOKEN_RANGE = -7

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable flags: no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
               "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.mo_bf16_to_f64_array.argtypes = [P, P, I64]
        lib.mo_f64_to_bf16_array.argtypes = [P, P, I64]
        lib.mo_e4m3_to_f64_array.argtypes = [P, P, I64]
        lib.mo_f64_to_e4m3_array.argtypes = [P, P, I64]
        lib.mo_rms_norm.argtypes = [P, P, I64, ctypes.c_double, P]
        lib.mo_input_stage.argtypes = [P, P, P, P, I64, P, I64, I64, ctypes.c_double, P, P, P, P]
        lib.mo_input_stage.restype = ctypes.c_int
        lib.mo_logits.argtypes = [ctypes.c_int, P, P, P, I64, I64, I64, P]
        lib.mo_logits_rows.argtypes = [ctypes.c_int, P, P, P, I64, P, I64, P]
        lib.mo_argmax.argtypes = [P, I64]
        lib.mo_argmax.restype = I64
        lib.mo_quantize_row.argtypes = [P, I64, P, P]
        lib.mo_quantize_row.restype = ctypes.c_int
        lib.mo_quantize.argtypes = [P, I64, I64, P, P]
        lib.mo_quantize.restype = ctypes.c_int
        lib.mo_pick_combine.argtypes = [P, P, I64]
        lib.mo_pick_combine.restype = I64
        lib.mo_xchg_pack.argtypes = [ctypes.c_int, ctypes.c_uint16, I64, P]
        lib.mo_xchg_sum.argtypes = [P, P, P]
        lib.mo_xchg_pick.argtypes = [P]
        lib.mo_xchg_pick.restype = I64
        _lib = lib
        return lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype).name}, got {a.dtype}")
    return np.ascontiguousarray(a)


def _p(a: np.ndarray | None):
    return None if a is None else a.ctypes.data


# ---------------------------------------------------------------------------- codecs
def bf16_to_f64(bits) -> np.ndarray:
    a = _c(bits, np.uint16)
    out = np.empty(a.shape, np.float64)
    _load().mo_bf16_to_f64_array(_p(a), _p(out), a.size)
    return out


def f64_to_bf16(values) -> np.ndarray:
    a = _c(np.asarray(values, np.float64), np.float64)
    out = np.empty(a.shape, np.uint16)
    _load().mo_f64_to_bf16_array(_p(a), _p(out), a.size)
    return out


def e4m3_to_f64(codes) -> np.ndarray:
    a = _c(codes, np.uint8)
    out = np.empty(a.shape, np.float64)
    _load().mo_e4m3_to_f64_array(_p(a), _p(out), a.size)
    return out


def f64_to_e4m3(values) -> np.ndarray:
    a = _c(np.asarray(values, np.float64), np.float64)
    out = np.empty(a.shape, np.uint8)
    _load().mo_f64_to_e4m3_array(_p(a), _p(out), a.size)
    return out


# ---------------------------------------------------------------------------- the head
def rms_norm(x, w, eps: float) -> np.ndarray:
    """rms_norm_vanilla on a [n] or [rows, n] BF16 array; returns BF16 bits."""
    x = _c(x, np.uint16)
    w = _c(w, np.uint16)
    n = x.shape[-1]
    assert w.shape == (n,)
    out = np.empty_like(x)
    xr, orr = x.reshape(-1, n), out.reshape(-1, n)
    for r in range(xr.shape[0]):
        _load().mo_rms_norm(_p(xr[r]), _p(w), n, float(np.float32(eps)), _p(orr[r]))
    return out


def input_stage(embed, enorm_w, hnorm_w, eh_proj, tokens, hidden, eps: float,
                return_concat: bool = False, return_sums: bool = False):
    """x[b] = eh_proj( concat( enorm(embed[tokens[b]]), hnorm(hidden[b]) ) ), BF16.

    Returns (x [B, H] uint16, status [B] int); with return_concat the concat [B, 2H] comes
    second; with return_sums the fp64 sums before rounding [B, H] come last.
    """
    embed = _c(embed, np.uint16)
    V, H = embed.shape
    eh_proj = _c(eh_proj, np.uint16)
    assert eh_proj.shape == (H, 2 * H)
    hidden = _c(hidden, np.uint16).reshape(-1, H)
    tokens = np.asarray(tokens, np.int64).reshape(-1)
    B = tokens.shape[0]
    assert hidden.shape[0] == B
    x = np.empty((B, H), np.uint16)
    concat = np.empty((B, 2 * H), np.uint16)
    scratch = np.empty(2 * H, np.uint16)
    sums = np.empty((B, H), np.float64)
    status = np.empty(B, np.int64)
    ew, hw = _c(enorm_w, np.uint16), _c(hnorm_w, np.uint16)
    for b in range(B):
        status[b] = _load().mo_input_stage(
            _p(embed), _p(ew), _p(hw), _p(eh_proj), int(tokens[b]), _p(hidden[b]), H, V,
            float(np.float32(eps)), _p(concat[b]), _p(x[b]), _p(sums[b]), _p(scratch))
    out = (x, concat, status) if return_concat else (x, status)
    return out + (sums,) if return_sums else out


def final_norm(x, final_norm_w, eps: float) -> np.ndarray:
    """shared_head.norm: rms_norm_vanilla of x with the final-norm weight."""
    return rms_norm(x, final_norm_w, eps)


def logits(w_dtype: int, W, scale, xhat, v0: int = 0, v1: int | None = None,
           threads: int = 1) -> np.ndarray:
    """fp64 logits of rows [v0, v1) for each BF16 vector in xhat ([H] or [B, H]).

    ``threads`` > 1 splits the row range over Python threads; each thread runs the same
    plain C loop on its own rows (ctypes releases the GIL), so the values are identical.
    """
    if w_dtype == 0:
        W = _c(W, np.uint16)
        scale_a = None
    else:
        W = _c(W, np.uint8)
        scale_a = _c(scale, np.float32)
    V, H = W.shape
    v1 = V if v1 is None else v1
    xh = _c(xhat, np.uint16).reshape(-1, H)
    out = np.empty((xh.shape[0], v1 - v0), np.float64)
    lib = _load()

    def run(b, a, z):
        lib.mo_logits(w_dtype, _p(W), _p(scale_a), _p(xh[b]), H, a, z,
                      out[b].ctypes.data + 8 * (a - v0))

    jobs = []
    for b in range(xh.shape[0]):
        if threads <= 1:
            jobs.append((b, v0, v1))
        else:
            edges = np.linspace(v0, v1, threads + 1).astype(np.int64)
            jobs += [(b, int(edges[i]), int(edges[i + 1])) for i in range(threads) if edges[i] < edges[i + 1]]
    if threads <= 1:
        for j in jobs:
            run(*j)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(lambda j: run(*j), jobs))
    return out if np.ndim(xhat) > 1 else out[0]


def logits_rows(w_dtype: int, W, scale, xhat, rows) -> np.ndarray:
    """fp64 logits of an explicit list of rows for one vector xhat [H]."""
    W = _c(W, np.uint16 if w_dtype == 0 else np.uint8)
    H = W.shape[1]
    scale_a = None if w_dtype == 0 else _c(scale, np.float32)
    rows = _c(np.asarray(rows, np.int64), np.int64)
    xh = _c(xhat, np.uint16)
    assert xh.shape == (H,)
    out = np.empty(rows.shape[0], np.float64)
    _load().mo_logits_rows(w_dtype, _p(W), _p(scale_a), _p(xh), H, _p(rows), rows.shape[0], _p(out))
    return out


def argmax(values) -> int:
    """Lowest index among equal maxima; NaN never wins; -1 if all are NaN."""
    a = _c(np.asarray(values, np.float64), np.float64)
    return int(_load().mo_argmax(_p(a), a.size))


def shard_pick(logits, v0: int, n: int) -> tuple[float, int]:
    """A vocabulary shard's offer: (value, global index) of the lowest-index maximum of the
    logits of rows [v0, v0 + n), or (nan, -1) when there is none."""
    seg = np.asarray(logits, np.float64)[v0:v0 + n]
    i = argmax(seg)
    return (float("nan"), -1) if i < 0 else (float(seg[i]), v0 + i)


def pick_combine(values, indices) -> int:
    """The draft from R shards' offers (value, global index): largest value, lowest index."""
    v = _c(np.asarray(values, np.float64), np.float64)
    i = _c(np.asarray(indices, np.int64), np.int64)
    assert v.shape == i.shape
    return int(_load().mo_pick_combine(_p(v), _p(i), v.size))


def xchg_pack(rank: int, value_bf16: int, global_index: int) -> np.ndarray:
    """The source's eight BF16 exchange lanes as rank ``rank`` (0 or 1) writes them."""
    lanes = np.zeros(8, np.uint16)
    _load().mo_xchg_pack(int(rank), int(value_bf16), int(global_index), _p(lanes))
    return lanes


def xchg_sum(a, b) -> np.ndarray:
    """The SUM all-reduce of two ranks' lanes (BF16 element sums)."""
    a = _c(np.asarray(a, np.uint16), np.uint16)
    b = _c(np.asarray(b, np.uint16), np.uint16)
    out = np.zeros(8, np.uint16)
    _load().mo_xchg_sum(_p(a), _p(b), _p(out))
    return out


def xchg_pick(lanes) -> int:
    """The global index the source's exchange decides for (`>=`: rank 0 wins a tie)."""
    lanes = _c(np.asarray(lanes, np.uint16), np.uint16)
    return int(_load().mo_xchg_pick(_p(lanes)))


def quantize(W):
    """FP8 E4M3 copy: returns (codes [V, H] uint8, scale [V] float32, status)."""
    W = _c(W, np.uint16)
    V, H = W.shape
    q = np.zeros((V, H), np.uint8)
    s = np.zeros(V, np.float32)
    st = _load().mo_quantize(_p(W), V, H, _p(q), _p(s))
    return q, s, st


def dequantize(q, s) -> np.ndarray:
    """decode(code) * scale in fp64 (exact): the weights the FP8 head computes with."""
    return e4m3_to_f64(q) * np.asarray(s, np.float64)[:, None]


def head(weights: dict, tokens, hidden, eps: float, w_dtype: int = 0, lm_head=None,
         scale=None, threads: int = 1) -> dict:
    """The whole head, block = identity: x, xhat, fp64 logits [B, V], draft [B]."""
    x, status = input_stage(weights["embed"], weights["enorm_w"], weights["hnorm_w"],
                            weights["eh_proj"], tokens, hidden, eps)
    xhat = final_norm(x, weights["final_norm_w"], eps)
    W = weights["lm_head"] if lm_head is None else lm_head
    lg = logits(w_dtype, W, scale, xhat, threads=threads)
    lg = lg.reshape(xhat.shape[0], -1)
    draft = np.array([argmax(r) for r in lg], np.int64)
    return {"x": x, "xhat": xhat, "logits": lg, "draft": draft, "status": status}
