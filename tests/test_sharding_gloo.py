"""Multi-rank host logic on CPU ranks (gloo, world size 2): sequence sharding covers the
batch once, per-rank results assemble into the single-process result, and the timing
reductions (slowest rank, total work) that bench.py uses. No GPU; no collective is on
the data path -- the all_gather below is the test's own check."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from speculative_decoding_token_temp_gb300 import sharding


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_shard_bounds_cover_once():
    for total in (0, 1, 5, 256, 513):
        for world in (1, 2, 3, 8):
            spans = [sharding.shard_bounds(total, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == total
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [hi - lo for lo, hi in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        sharding.shard_bounds(10, 2, 2)
    assert len({sharding.rank_seed(2, r) for r in range(8)}) == 8 and sharding.rank_seed(2, 0) == 2


def _rank_main(rank, world, port, q):
    import torch
    import torch.distributed as dist

    from oracle import oracle as O
    from speculative_decoding_token_temp_gb300 import sharding, synth
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = synth.make_stochastic(5, 300, synth.BF16, 0.8, seed=7, gamma_range=(0, 4), agreement=0.7)
        lo, hi = sharding.shard_bounds(w.B, world, rank)
        mine = O.verify_stochastic(w.target, w.draft, w.tokens, w.cu_draft, w.T, w.u_accept, w.u_sample, w.dtype,
                                   seqs=range(lo, hi))
        got = [None] * world
        dist.all_gather_object(got, {b: (r["n"], list(r["tokens"])) for b, r in mine.items()})
        slowest = sharding.max_over_ranks(1.5 + rank, world, torch.device("cpu"))
        total = sharding.sum_over_ranks(10 * (rank + 1), world, torch.device("cpu"))
        if rank == 0:
            merged = {}
            for part in got:
                assert not set(part) & set(merged)
                merged.update(part)
            q.put((merged, slowest, total))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_gloo_ranks_reassemble_the_batch():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    merged, slowest, total = q.get(timeout=240)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    from oracle import oracle as O
    from speculative_decoding_token_temp_gb300 import synth
    w = synth.make_stochastic(5, 300, synth.BF16, 0.8, seed=7, gamma_range=(0, 4), agreement=0.7)
    ref = O.verify_stochastic(w.target, w.draft, w.tokens, w.cu_draft, w.T, w.u_accept, w.u_sample, w.dtype)
    assert sorted(merged) == list(range(w.B))
    for b, r in ref.items():
        assert merged[b][0] == r["n"] and merged[b][1] == list(r["tokens"])
    assert slowest == 2.5 and total == 30.0
    assert np.all(np.diff(w.cu_draft) >= 0)


def _vocab_rank_main(rank, world, port, q):
    """Rank r holds vocabulary shard r of every row pair (tensor-parallel logits): it
    computes its shard statistics, the ranks exchange them (all_gather, the one exchange
    step), every rank merges them in shard order, and the residual draw is resolved by a
    second exchange of per-shard masses and an exclusive scan."""
    import math

    import numpy as np
    import torch.distributed as dist

    from oracle import oracle as O
    from speculative_decoding_token_temp_gb300 import sharding, synth
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = synth.make_stochastic(4, 1000, synth.F32, 0.8, seed=9, gamma=2, agreement=0.7)
        lo, hi = sharding.shard_bounds(w.V, world, rank)
        rows_t = O.widen(w.target[:w.total_draft], w.dtype)      # rows 0..7 paired with draft rows 0..7
        rows_d = O.widen(w.draft, w.dtype)
        mine = [O.shard_stats(rows_t[i, lo:hi], rows_d[i, lo:hi], w.T, lo) for i in range(len(rows_d))]
        got = [None] * world
        dist.all_gather_object(got, mine)
        merged = []
        for i in range(len(rows_d)):
            st = got[0][i]
            for r in range(1, world):
                st = O.merge_stats(st, got[r][i])
            merged.append(O.stats_outputs(st, w.V))
        # residual draw of row pair 0 with u = 0.37: each rank's shard of max(0, p - q)
        out0 = merged[0]
        p = np.exp(rows_t[0, lo:hi] / w.T - out0["lse_t"])
        qd = np.exp(rows_d[0, lo:hi] / w.T - out0["lse_d"])
        wsh = np.maximum(0.0, p - qd)
        zs = [None] * world
        dist.all_gather_object(zs, float(np.sum(wsh)))
        Z = sum(zs)
        target = 0.37 * Z
        base = sum(zs[:rank])
        tok = -1
        if base <= target < base + zs[rank] or (rank == world - 1 and target >= base + zs[rank]):
            C = base + np.cumsum(wsh)
            hit = np.nonzero(C > target)[0]
            tok = lo + int(hit[0] if hit.size else np.nonzero(wsh > 0)[0][-1])
        toks = [None] * world
        dist.all_gather_object(toks, tok)
        if rank == 0:
            q.put((merged, [t for t in toks if t >= 0], Z))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
@pytest.mark.parametrize("world", [2, 3])
def test_vocabulary_shards_merge_across_gloo_ranks(world):
    import numpy as np

    from oracle import oracle as O
    from speculative_decoding_token_temp_gb300 import synth
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_vocab_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    merged, owners, Z = q.get(timeout=240)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    w = synth.make_stochastic(4, 1000, synth.F32, 0.8, seed=9, gamma=2, agreement=0.7)
    rows_t = O.widen(w.target[:w.total_draft], w.dtype)
    rows_d = O.widen(w.draft, w.dtype)
    for i, out in enumerate(merged):
        assert out["argmax"] == int(np.argmax(rows_t[i]))
        assert out["nkl"] == pytest.approx(O.nkl_pair(rows_t[i], rows_d[i], w.T)[0], rel=1e-9)
    p = O.softmax_T(rows_t[0], w.T)
    qd = O.softmax_T(rows_d[0], w.T)
    y, Z0, c0, c1 = O.inverse_cdf(O.residual(p, qd), 0.37)
    assert len(owners) == 1 and owners[0] == y and Z == pytest.approx(Z0, rel=1e-12)
