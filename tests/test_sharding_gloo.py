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
