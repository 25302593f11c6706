"""The cross-rank step of the vocabulary-sharded head on CPU: two gloo ranks, each holding one
half of the vocabulary ("glm5next_mtp_head.rs": `head_v0` / `head_n` and `forward_one`'s
sharded branch). Each rank takes its half's lowest-index maximum (from the oracle's logits,
rounded to FP32 as the GPU returns them), makes the exchange key with the library's host
function, and calls the package's exchange (one MAX all-reduce of the [B] keys); both ranks must
then decode the lowest-index maximum of the whole vocabulary, also when the maximum ties across
the boundary between the halves. The source's own exchange (eight BF16 lanes through a SUM
all-reduce) runs over the same process group and must agree wherever the source's BF16 lanes
can tell the two halves' maxima apart."""
import os
import socket

import numpy as np
import torch.multiprocessing as mp

H, V, B = 64, 1000, 3


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _problem():
    """Weights, xhat for B sequences, and the fp32 logits of the whole vocabulary."""
    import oracle
    import synth
    w = synth.make_weights(H, V, 21, "cpu")
    lm = synth.bits(w.lm_head).copy()
    rng = np.random.default_rng(4)
    planted = oracle.f64_to_bf16(0.05 * np.sign(rng.standard_normal(H)))
    lm[V // 2 - 1] = lm[V // 2] = planted  # identical rows on both sides of the boundary
    xhat = oracle.f64_to_bf16(rng.standard_normal((B, H)))
    xhat[1] = oracle.f64_to_bf16(oracle.bf16_to_f64(planted) * 20.0)  # sequence 1: the planted rows win
    logits = oracle.logits(0, lm, None, xhat).astype(np.float32)
    return lm, xhat, logits


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch
    import torch.distributed as dist

    import mtp_speculative_draft_head_gb300 as m
    import oracle
    dist.init_process_group("gloo", rank=rank, world_size=world)
    _, _, logits = _problem()
    v0, n = m.shard_geometry(V, rank, world)
    keys = torch.empty(B, dtype=torch.int64)
    lanes = torch.zeros((B, 8), dtype=torch.bfloat16)
    for b in range(B):
        val, g = oracle.shard_pick(logits[b].astype(np.float64), v0, n)
        keys[b] = m.mtp_head_pick_key(val, g)
        pack = oracle.xchg_pack(rank, int(oracle.f64_to_bf16(np.array([val]))[0]), g)
        lanes[b] = torch.from_numpy(pack.view(np.int16)).view(torch.bfloat16)
    m.exchange_picks(keys)                     # exact keys: one MAX all-reduce
    dist.all_reduce(lanes, op=dist.ReduceOp.SUM)  # the source's lanes: one BF16 SUM all-reduce
    out[rank] = ([m.mtp_head_pick_index(int(k)) for k in keys],
                 [oracle.xchg_pick(lanes[b].view(torch.int16).numpy().view(np.uint16)) for b in range(B)])
    dist.destroy_process_group()


def test_two_rank_exchange_gives_the_full_vocabulary_draft():
    import oracle
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    _, _, logits = _problem()
    want = [oracle.argmax(logits[b].astype(np.float64)) for b in range(B)]
    assert want[1] == V // 2 - 1  # the tie across the boundary goes to the lower half
    for r in range(world):
        exact, lanes = res[r]
        assert exact == want
        for b in range(B):
            # the source's lanes round each half's maximum to BF16: they agree with the exact
            # pick unless the two maxima round to one BF16 value
            halves = [oracle.shard_pick(logits[b].astype(np.float64), h * (V // 2), V // 2)[0] for h in (0, 1)]
            bf = oracle.f64_to_bf16(np.array(halves))
            if bf[0] != bf[1] or halves[0] == halves[1]:
                assert lanes[b] == want[b]
