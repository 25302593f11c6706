"""GPU parity of the vocabulary-sharded output stage ("glm5next_mtp_head.rs": the vocab-shard
geometry `head_rank` / `head_v0` / `head_n` and `forward_one`'s sharded branch with its
cross-rank pick), on one GPU: the vocabulary is cut into k shards, each shard runs
mtp_head_logits_argmax_shard on its own rows (its own FP8 rows and scales for the FP8 head), and
mtp_head_pick_combine picks the draft from the k exchange keys. The same kernels sweep every row
with the same arithmetic whatever the shard, so each shard's logits must equal the matching
columns of the full sweep's logits bit for bit, and the combined draft and its value must equal
the full sweep's draft and maximum. Rows planted on both sides of every shard boundary tie for
the maximum, so a tie across a boundary must go to the lower index. The draft is also checked
against the oracle's logits."""
import math

import numpy as np
import pytest
import torch

import mtp_speculative_draft_head_gb300 as m
import oracle
import synth
from gpu_helpers import TOL_BF16, TOL_FP8, check_draft

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
EPS = synth.EPS


def _edges(V, k, rng):
    """k contiguous shards of [0, V), uneven, none empty, one of a single row when k > 2."""
    cuts = np.sort(rng.choice(np.arange(2, V - 1), size=k - 1, replace=False))
    if k > 2:
        cuts[1] = cuts[0] + 1
    return np.concatenate([[0], cuts, [V]]).astype(np.int64)


def _setup(H, V, B, fp8, plant_edges=None):
    w = synth.make_weights(H, V, 3, "cpu")
    x = synth._normal_bf16((B, H), 0.0, 1.0, torch.Generator().manual_seed(77 + B), "cpu")
    fw = synth.bits(w.final_norm_w)
    lm = w.lm_head
    if plant_edges is not None:
        # rows on both sides of every inner boundary, all equal to 0.05 sign(xhat of sequence 0)
        xhat0 = oracle.final_norm(synth.bits(x[:1]), fw, EPS)[0]
        rows = sorted({int(e) + d for e in plant_edges[1:-1] for d in (-1, 0)})
        lm = synth.plant_rows(lm, torch.tensor(rows), torch.from_numpy(oracle.bf16_to_f64(xhat0)))
    g = {k: v.to(DEV) for k, v in w.as_dict().items()}
    g["lm_head"] = lm.to(DEV)
    if fp8:
        W = torch.empty((V, H), dtype=torch.uint8, device=DEV)
        s = torch.empty(V, dtype=torch.float32, device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        m.mtp_head_quantize_fp8(g["lm_head"], W, s, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        return g, x.to(DEV), W, s, m.W_FP8_E4M3
    return g, x.to(DEV), g["lm_head"], None, m.W_BF16


@pytest.mark.parametrize("H,V,B", [(6144, 20000, 1), (2048, 7777, 3), (256, 4096, 16)])
@pytest.mark.parametrize("k", [2, 3, 8])
@pytest.mark.parametrize("fp8", [False, True])
def test_shards_combine_to_the_full_sweep(H, V, B, k, fp8):
    rng = np.random.default_rng(H + V + k)
    e = _edges(V, k, rng)
    g, x, W, s, wt = _setup(H, V, B, fp8, plant_edges=e)
    ws = m.workspace(B, H, V, DEV)
    full_lg = torch.empty((B, V), dtype=torch.float32, device=DEV)
    full_d = torch.empty(B, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    m.mtp_head_logits_argmax_batched(x, g["final_norm_w"], W, s, wt, full_lg, full_d, ws, status, EPS)
    picks = torch.empty((k, B), dtype=torch.int64, device=DEV)
    shard_lg, shard_d = [], []
    for r in range(k):
        v0, v1 = int(e[r]), int(e[r + 1])
        lg = torch.full((B, v1 - v0), float("nan"), dtype=torch.float32, device=DEV)
        d = torch.full((B,), -5, dtype=torch.int32, device=DEV)
        m.mtp_head_logits_argmax_shard(x, g["final_norm_w"], W[v0:v1], None if s is None else s[v0:v1], wt, v0,
                                       lg, picks[r], d, ws, status, EPS)
        shard_lg.append(lg)
        shard_d.append(d)
    draft = torch.full((B,), -5, dtype=torch.int32, device=DEV)
    value = torch.empty(B, dtype=torch.float32, device=DEV)
    m.mtp_head_pick_combine(picks, draft, value)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    full = full_lg.cpu()
    for r in range(k):
        v0, v1 = int(e[r]), int(e[r + 1])
        assert torch.equal(shard_lg[r].cpu().view(torch.int32), full[:, v0:v1].contiguous().view(torch.int32)), r
        lg = shard_lg[r].cpu().numpy()
        for b in range(B):
            want = v0 + int(np.argmax(lg[b]))
            assert int(shard_d[r][b]) == want
            key = int(picks[r, b])
            assert m.mtp_head_pick_index(key) == want
            assert m.mtp_head_pick_value(key) == float(lg[b].max())
    assert torch.equal(draft.cpu(), full_d.cpu())
    assert torch.equal(value.cpu(), full.max(dim=1).values)
    assert int(draft[0]) == int(e[1]) - 1  # the planted tie straddling the first boundary
    # against the oracle
    xhat = oracle.final_norm(synth.bits(x), synth.bits(g["final_norm_w"]), EPS)
    if fp8:
        ref = oracle.logits(1, synth.bits(W), s.cpu().numpy(), xhat, threads=8)
    else:
        ref = oracle.logits(0, synth.bits(W), None, xhat, threads=8)
    ref = ref.reshape(B, V)
    for b in range(B):
        check_draft(int(draft[b]), full[b].numpy(), ref[b], TOL_FP8 if fp8 else TOL_BF16)


@pytest.mark.parametrize("world", [1, 2, 7, 8])
@pytest.mark.parametrize("fp8", [False, True])
def test_vocab_shard_ranks_on_one_gpu(world, fp8):
    """VocabShard with the source's geometry (equal ranges when V divides by the rank count,
    else every rank sweeps all of V), each rank with its own FP8 copy of its rows: the keys of
    all ranks, combined, give the full sweep's draft."""
    H, V, B = 2048, 9600, 4
    g, x, W, s, wt = _setup(H, V, B, False)
    head = m.MtpDraftHead(g["embed"], g["lm_head"], g["eh_proj"], g["enorm_w"], g["hnorm_w"],
                          g["final_norm_w"], eps=EPS, max_batch=B)
    if fp8:
        assert head.quantize_fp8() == 0
    _, want = head.logits_argmax(x, fp8=fp8, logits=False)
    ranks = [m.VocabShard(g["lm_head"], g["final_norm_w"], r, world, eps=EPS, max_batch=B) for r in range(world)]
    keys = []
    for vs in ranks:
        if fp8:
            assert vs.quantize_fp8() == 0
        keys.append(vs.picks(x, fp8=fp8))
    if world == 7:  # 9600 does not divide by 7: every rank sweeps the whole vocabulary
        assert all(not vs.sharded and vs.n == V for vs in ranks)
    draft = torch.empty(B, dtype=torch.int32, device=DEV)
    m.mtp_head_pick_combine(torch.stack(keys), draft)
    # one rank alone, as a single-rank job runs it (no exchange)
    single = ranks[0].draft(x, fp8=fp8) if world == 1 else None
    torch.cuda.synchronize()
    assert torch.equal(draft, want)
    if single is not None:
        assert torch.equal(single, want)


def test_all_nan_sequence_gives_empty_keys_and_draft_minus_one():
    H, V, B = 256, 4096, 2
    g, x, W, s, wt = _setup(H, V, B, False)
    x[1, 7] = float("nan")  # every logit of sequence 1 is NaN
    ws = m.workspace(B, H, V, DEV)
    picks = torch.empty((2, B), dtype=torch.int64, device=DEV)
    for r, (v0, v1) in enumerate(((0, 1000), (1000, V))):
        m.mtp_head_logits_argmax_shard(x, g["final_norm_w"], W[v0:v1], None, wt, v0, None, picks[r], None, ws,
                                       None, EPS)
    draft = torch.empty(B, dtype=torch.int32, device=DEV)
    m.mtp_head_pick_combine(picks, draft)
    torch.cuda.synchronize()
    assert int(picks[0, 1]) == -2 ** 63 and int(picks[1, 1]) == -2 ** 63
    assert int(draft[1]) == -1
    assert 0 <= int(draft[0]) < V


@pytest.mark.parametrize("R", [1, 7, 33, 1000])
def test_pick_combine_many_keys(R):
    """The combine kernel over R shards' keys for 16 sequences (a lane loop and a shuffle tree when
    R > 32): keys made on the host from random (value, global index) pairs with ties, +-0, +-inf
    and empty picks; the draft and value must be those of the largest key, which is the argmax
    order's winner (larger value, then lower index; -1 and NaN when every key is empty)."""
    B = 16
    rng = np.random.default_rng(R)
    vals = np.round(rng.standard_normal((R, B)) * 2).astype(np.float32)
    vals[rng.random((R, B)) < 0.05] = np.float32(-0.0)
    vals[rng.random((R, B)) < 0.02] = np.float32(np.inf)
    vals[rng.random((R, B)) < 0.02] = np.float32(-np.inf)
    idx = rng.integers(0, 2 ** 31 - 1, (R, B))
    empty = rng.random((R, B)) < 0.1
    empty[:, 3] = True  # sequence 3: every shard empty
    keys = np.array([[m.mtp_head_pick_key(float(vals[r, b]), -1 if empty[r, b] else int(idx[r, b])) for b in range(B)]
                     for r in range(R)], dtype=np.int64)
    draft = torch.full((B,), -5, dtype=torch.int32, device=DEV)
    value = torch.empty(B, dtype=torch.float32, device=DEV)
    m.mtp_head_pick_combine(torch.from_numpy(keys).to(DEV), draft, value)
    torch.cuda.synchronize()
    for b in range(B):
        ok = ~empty[:, b]
        if not ok.any():
            assert int(draft[b]) == -1 and math.isnan(float(value[b]))
            continue
        v, i = vals[ok, b].astype(np.float64), idx[ok, b]
        best = v.max()
        want = int(i[v == best].min())
        assert int(draft[b]) == want
        assert float(value[b]) == best
