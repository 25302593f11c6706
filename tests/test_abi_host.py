"""The C ABI without a GPU: the library builds and loads, exports every function the header
declares, the Python binding declares each with the header's arity, and host-side validation
returns the documented status codes before anything is launched (the fake device addresses
below are never dereferenced: every call here fails validation first)."""
import ctypes
import os
import re

import pytest

import mtp_speculative_draft_head_gb300 as m

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "mtp_head.h")


def _declarations():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    decls = {}
    for mt in re.finditer(r"\b(mtp_head_\w+)\s*\(([^;{]*?)\)\s*;", text, flags=re.S):
        name, params = mt.group(1), mt.group(2).strip()
        decls[name] = 0 if params in ("", "void") else params.count(",") + 1
    return decls


@pytest.fixture(scope="module")
def lib():
    return m.load()


def test_header_declares_the_entry_points():
    d = _declarations()
    for name in ("mtp_head_input", "mtp_head_input_batched", "mtp_head_logits_argmax",
                 "mtp_head_logits_argmax_batched", "mtp_head_quantize_fp8",
                 "mtp_head_workspace_bytes", "mtp_head_forward_batched", "mtp_head_forward_host",
                 "mtp_head_forward_host_args",
                 "mtp_head_context_rows", "mtp_head_context_workspace_bytes",
                 "mtp_head_logits_argmax_batched_noalloc", "mtp_head_logits_argmax_shard",
                 "mtp_head_pick_combine", "mtp_head_pick_key", "mtp_head_pick_index", "mtp_head_pick_value",
                 "mtp_head_strerror"):
        assert name in d


def test_library_exports_every_declared_symbol(lib):
    for name in _declarations():
        assert hasattr(lib, name), f"{name} is declared in mtp_head.h but not exported"


def test_binding_matches_header_arity():
    d = _declarations()
    assert set(m.SIGNATURES) == set(d)
    for name, (_, args) in m.SIGNATURES.items():
        assert len(args) == d[name], name


def test_strerror_covers_every_code(lib):
    for code in range(0, -10, -1):
        assert m.strerror(code) != "unknown status"
    assert m.strerror(-99) == "unknown status"


def test_workspace_bytes(lib):
    assert m.mtp_head_workspace_bytes(0, 6144, 154880) == 0
    assert m.mtp_head_workspace_bytes(17, 6144, 154880) == 0
    assert m.mtp_head_workspace_bytes(1, 0, 10) == 0
    # the output stage's part (2304 bytes whatever B), then room for the context-row input stage
    for B in (1, 2, 7, 16):
        for H in (64, 1000, 6144):
            assert m.mtp_head_workspace_bytes(B, H, 154880) == 2304 + m.mtp_head_context_workspace_bytes(B, H)
    assert m.mtp_head_workspace_bytes(16, 6144, 154880) >= 2304 + 16 * 2 * 6144 * 2 + 16 * 4  # concat, row flags


def test_context_workspace_bytes(lib):
    f = m.mtp_head_context_workspace_bytes
    assert f(0, 6144) == 0 and f(65537, 6144) == 0 and f(17, 0) == 0 and f(17, 65537) == 0
    for R, H in ((17, 32), (512, 6144), (65536, 6144)):
        assert f(R, H) >= R * 2 * H * 2 + R * 4  # the concat and the row flags, at least
    sizes = [f(R, 1024) for R in (17, 100, 256, 257, 4096)]
    assert sizes == sorted(sizes)


A = 0x10000  # an aligned fake device address (never dereferenced)


def _input(lib, **kw):
    args = dict(embed=A, enorm_w=A, hnorm_w=A, eh_proj=A, tokens=A, hidden=A, x=A, status=None,
                B=1, H=64, V=100, eps=1e-6)
    args.update(kw)
    return lib.mtp_head_input_batched(args["embed"], args["enorm_w"], args["hnorm_w"], args["eh_proj"],
                                      args["tokens"], args["hidden"], args["x"], args["status"],
                                      args["B"], args["H"], args["V"], args["eps"], None)


def _output(lib, **kw):
    args = dict(x=A, fw=A, W=A, scale=None, wt=m.W_BF16, logits=None, draft=A, status=None, ws=A,
                ws_bytes=1 << 20, B=1, H=64, V=100, eps=1e-6)
    args.update(kw)
    return lib.mtp_head_logits_argmax_batched(args["x"], args["fw"], args["W"], args["scale"], args["wt"],
                                              args["logits"], args["draft"], args["status"], args["ws"],
                                              args["ws_bytes"], args["B"], args["H"], args["V"],
                                              args["eps"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(embed=None), m.ERR_ARG),
    (dict(tokens=None), m.ERR_ARG),
    (dict(x=None), m.ERR_ARG),
    (dict(eps=float("nan")), m.ERR_ARG),
    (dict(eps=-1.0), m.ERR_ARG),
    (dict(eps=float("inf")), m.ERR_ARG),
    (dict(B=0), m.ERR_SHAPE),
    (dict(B=17), m.ERR_SHAPE),
    (dict(H=0), m.ERR_SHAPE),
    (dict(H=65537), m.ERR_SHAPE),
    (dict(V=0), m.ERR_SHAPE),
    (dict(eh_proj=A + 8), m.ERR_ALIGN),
    (dict(hidden=A + 2), m.ERR_ALIGN),
    (dict(tokens=A + 2), m.ERR_ALIGN),
])
def test_input_stage_validation(lib, kw, code):
    assert _input(lib, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(x=None), m.ERR_ARG),
    (dict(W=None), m.ERR_ARG),
    (dict(draft=None), m.ERR_ARG),
    (dict(wt=2), m.ERR_ARG),
    (dict(wt=m.W_FP8_E4M3, scale=None), m.ERR_ARG),
    (dict(eps=float("nan")), m.ERR_ARG),
    (dict(B=0), m.ERR_SHAPE),
    (dict(B=17), m.ERR_SHAPE),
    (dict(V=-5), m.ERR_SHAPE),
    (dict(W=A + 4), m.ERR_ALIGN),
    (dict(draft=A + 1), m.ERR_ALIGN),
    (dict(ws=A + 8), m.ERR_ALIGN),
    (dict(ws=None), m.ERR_WORKSPACE),
    (dict(ws_bytes=16), m.ERR_WORKSPACE),
    (dict(ws_bytes=2303), m.ERR_WORKSPACE),            # one byte short of the output stage's part
    (dict(ws_bytes=2303, B=16), m.ERR_WORKSPACE),      # ... which is the same for every B
])
def test_output_stage_validation(lib, kw, code):
    assert _output(lib, **kw) == code


def test_quantizer_validation(lib):
    q = lib.mtp_head_quantize_fp8
    assert q(None, A, A, A, 10, 16, None) == m.ERR_ARG
    assert q(A, A, A, None, 10, 16, None) == m.ERR_ARG  # status is required here
    assert q(A, A, A, A, 0, 16, None) == m.ERR_SHAPE
    assert q(A + 2, A, A, A, 10, 16, None) == m.ERR_ALIGN


def test_forward_host_validation(lib):
    f = lib.mtp_head_forward_host
    args = [A, A, A, A, A, A, None, m.W_BF16, A, A, A, A, A, A, A, None, A, 1 << 20, 1, 64, 100,
            ctypes.c_float(1e-6), None]
    bad = list(args)
    bad[8] = None  # tokens_host
    assert f(*bad) == m.ERR_ARG
    bad = list(args)
    bad[16] = None  # workspace
    assert f(*bad) == m.ERR_WORKSPACE
    bad = list(args)
    bad[18] = 0  # B
    assert f(*bad) == m.ERR_SHAPE


# mtp_host_step_args field -> position of the same argument of mtp_head_forward_host
_HOST_FIELDS = {"embed": 0, "enorm_w": 1, "hnorm_w": 2, "eh_proj": 3, "final_norm_w": 4, "lm_head": 5,
                "row_scale": 6, "w_dtype": 7, "tokens_dev": 10, "hidden_dev": 11, "x_dev": 12, "draft_dev": 13,
                "status": 15, "workspace": 16, "workspace_bytes": 17, "B": 18, "H": 19, "V": 20, "eps": 21,
                "stream": 22}


@pytest.mark.parametrize("field,value", [
    ("embed", None), ("enorm_w", None), ("hnorm_w", None), ("eh_proj", A + 2), ("final_norm_w", None),
    ("lm_head", A + 8), ("row_scale", A + 2), ("w_dtype", 7), ("tokens_dev", None), ("hidden_dev", A + 4),
    ("x_dev", None), ("draft_dev", A + 2), ("status", A + 1), ("workspace", None), ("workspace_bytes", 16),
    ("B", 0), ("B", 17), ("H", 0), ("V", 0), ("eps", float("nan")), ("eps", -1.0),
])
def test_forward_host_args_reads_every_field(lib, field, value):
    # each variant breaks one field; both entry points must reject it with the same status before
    # anything runs, which they can only do if the struct's layout matches the header
    base = [A, A, A, A, A, A, None, m.W_BF16, A, A, A, A, A, A, A, None, A, 1 << 20, 1, 64, 100, 1e-6, None]
    fh = list(base)
    fh[_HOST_FIELDS[field]] = value
    want = lib.mtp_head_forward_host(*[ctypes.c_float(v) if i == 21 else v for i, v in enumerate(fh)])
    assert want in (m.ERR_ARG, m.ERR_SHAPE, m.ERR_ALIGN, m.ERR_WORKSPACE)  # rejected before any CUDA call
    sa = m._lib._HostStepArgs(*[fh[i] for i in _HOST_FIELDS.values()])
    assert lib.mtp_head_forward_host_args(ctypes.addressof(sa), fh[8], fh[9], fh[14]) == want


def test_forward_host_args_null(lib):
    assert lib.mtp_head_forward_host_args(None, A, A, A) == m.ERR_ARG
    sa = m._lib._HostStepArgs(A, A, A, A, A, A, None, m.W_BF16, A, A, A, A, None, A, 1 << 20, 0, 64, 100, 1e-6,
                              None)
    assert lib.mtp_head_forward_host_args(ctypes.addressof(sa), None, A, A) == m.ERR_ARG  # tokens_host


def _context(lib, **kw):
    args = dict(embed=A, enorm_w=A, hnorm_w=A, eh_proj=A, tokens=A, hidden=A, x=A, status=None, ws=A,
                ws_bytes=1 << 30, R=300, H=256, V=100, eps=1e-6)
    args.update(kw)
    return lib.mtp_head_context_rows(args["embed"], args["enorm_w"], args["hnorm_w"], args["eh_proj"],
                                     args["tokens"], args["hidden"], args["x"], args["status"], args["ws"],
                                     args["ws_bytes"], args["R"], args["H"], args["V"], args["eps"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(embed=None), m.ERR_ARG),
    (dict(eh_proj=None), m.ERR_ARG),
    (dict(tokens=None), m.ERR_ARG),
    (dict(x=None), m.ERR_ARG),
    (dict(eps=float("nan")), m.ERR_ARG),
    (dict(R=0), m.ERR_SHAPE),
    (dict(R=65537), m.ERR_SHAPE),
    (dict(H=0), m.ERR_SHAPE),
    (dict(V=0), m.ERR_SHAPE),
    (dict(x=A + 8), m.ERR_ALIGN),
    (dict(tokens=A + 2), m.ERR_ALIGN),
    (dict(ws=A + 8), m.ERR_ALIGN),
    (dict(H=100), m.ERR_NOT_IMPLEMENTED),  # R > 16 runs the GEMM, which needs H % 32 == 0
    (dict(ws=None), m.ERR_WORKSPACE),
    (dict(ws_bytes=1024), m.ERR_WORKSPACE),
])
def test_context_rows_validation(lib, kw, code):
    assert _context(lib, **kw) == code


def test_noalloc_output_stage_validation(lib):
    f = lib.mtp_head_logits_argmax_batched_noalloc
    assert f(A, A, A, None, m.W_BF16, None, A, None, 0, 64, 100, ctypes.c_float(1e-6), None) == m.ERR_SHAPE
    assert f(A, A, A, None, m.W_BF16, None, A, None, 17, 64, 100, ctypes.c_float(1e-6), None) == m.ERR_SHAPE


# ---------------------------------------------------------------------- vocabulary shards
def test_shard_entry_point_validation(lib):
    A = 0x10000  # fake, 16-byte aligned; never dereferenced
    eps = ctypes.c_float(1e-6)
    ws = m.mtp_head_workspace_bytes(1, 64, 100)

    def call(v0=0, n=100, pick=A, draft=None, B=1, H=64):
        return lib.mtp_head_logits_argmax_shard(A, A, A, None, m.W_BF16, v0, n, None, pick, draft, None, A, ws, B,
                                                H, eps, None)
    assert call(pick=None) == m.ERR_ARG
    assert call(v0=-1) == m.ERR_SHAPE
    assert call(n=0) == m.ERR_SHAPE
    assert call(v0=2 ** 31 - 100, n=100) == m.ERR_SHAPE
    assert call(pick=A + 4) == m.ERR_ALIGN
    assert call(B=17) == m.ERR_SHAPE
    assert call(draft=A + 2) == m.ERR_ALIGN


def test_pick_combine_validation(lib):
    A = 0x10000
    assert lib.mtp_head_pick_combine(None, 2, 1, A, None, None) == m.ERR_ARG
    assert lib.mtp_head_pick_combine(A, 2, 1, None, None, None) == m.ERR_ARG
    assert lib.mtp_head_pick_combine(A, 0, 1, A, None, None) == m.ERR_SHAPE
    assert lib.mtp_head_pick_combine(A, 2, 0, A, None, None) == m.ERR_SHAPE
    assert lib.mtp_head_pick_combine(A, 2, 17, A, None, None) == m.ERR_SHAPE
    assert lib.mtp_head_pick_combine(A + 4, 2, 1, A, None, None) == m.ERR_ALIGN


def test_pick_key_order_is_the_argmax_order(lib):
    """Host side of the exchange key: for random (value, index) pairs, including ties, +-0,
    +-inf and subnormals, key(a) > key(b) exactly when a beats b in the argmax order (larger
    value, then lower index); the key decodes back to its index and value."""
    import numpy as np
    rng = np.random.default_rng(3)
    specials = np.array([0.0, -0.0, np.inf, -np.inf, 1e-45, -1e-45, 3.4e38, -3.4e38, 1.0, -1.0], np.float32)
    vals = np.concatenate([specials, rng.standard_normal(200).astype(np.float32),
                           np.round(rng.standard_normal(100)).astype(np.float32)])
    idx = rng.integers(0, 2 ** 31 - 1, vals.size)
    idx[:20] = [0, 1, 2 ** 31 - 2, 5, 5, 7, 0, 3, 3, 9] * 2
    keys = [m.mtp_head_pick_key(float(v), int(i)) for v, i in zip(vals, idx)]
    for k, v, i in zip(keys, vals, idx):
        assert m.mtp_head_pick_index(k) == int(i)
        got = m.mtp_head_pick_value(k)
        assert got == float(v) and (v != 0 or np.signbit(np.float32(got)) == False)  # noqa: E712
    for a in range(0, vals.size, 3):
        for b in range(vals.size):
            va, vb, ia, ib = float(vals[a]), float(vals[b]), int(idx[a]), int(idx[b])
            beats = va > vb or (va == vb and ia < ib)
            assert (keys[a] > keys[b]) == beats, (va, ia, vb, ib)


def test_pick_key_empty(lib):
    empty = -2 ** 63
    assert m.mtp_head_pick_key(float("nan"), 4) == empty
    assert m.mtp_head_pick_key(1.0, -1) == empty
    assert m.mtp_head_pick_index(empty) == -1
    assert m.mtp_head_pick_value(empty) != m.mtp_head_pick_value(empty)  # NaN
    assert m.mtp_head_pick_key(float("-inf"), 2 ** 31 - 1) > empty


def test_wait_limit_setter_returns_the_previous_limit(lib):
    """The stage-wait limit is process-wide state: 2 s by default, and every set returns the
    limit it replaces (nothing is launched here)."""
    prev = m.mtp_head_set_wait_limit_ns(5)
    try:
        assert prev == 2_000_000_000
        assert m.mtp_head_set_wait_limit_ns(0) == 5
        assert m.mtp_head_set_wait_limit_ns(7) == 0
    finally:
        assert m.mtp_head_set_wait_limit_ns(prev) == 7
    assert m.mtp_head_set_wait_limit_ns(prev) == prev
