"""Seeded random configurations of every call against the oracle: vocabularies from one
token to 210000 (with extra weight on the lengths around 16-byte blocks and vocabulary
chunks), dense and ragged batches (gamma up to 16, and up to 128 on short rows), both
dtypes, logit buffers shifted alike or apart, temperatures from 0.3 to 1.5, a separate
draft temperature, position-adaptive NKL thresholds, block-accept, trees of 1-64 nodes of
any shape, and multi-draft groups of K = 2-4. Each case is compared with the oracle on
every sequence, with the tolerances of the parity tests; a failure names its case."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from speculative_decoding_token_temp_gb300 import api, synth

from gpu_util import (NKL_ABS, REL, compare_greedy, compare_nkl, compare_stochastic, compare_tree, handmade,
                      run_greedy, run_nkl, run_stochastic, run_tree, to_dev)

pytestmark = pytest.mark.gpu

CASES = 60   # per call kind; about 5 s each on a GB300

_EDGE = [1, 2, 3, 7, 8, 9, 15, 16, 17, 31, 33, 255, 257, 4095, 4096, 4097, 32767, 32768, 32769, 49151, 49152,
         49153, 65535, 65536, 65537, 98303, 98304, 98305, 131071, 131072, 131073, 196607, 196608, 196609]


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def _V(rng):
    r = rng.random()
    if r < 0.3:
        return int(rng.choice(_EDGE))
    if r < 0.5:
        return int(rng.integers(1, 400))
    if r < 0.8:
        return int(rng.integers(400, 70000))
    return int(rng.integers(70000, 210000))


def _dtype(rng):
    return synth.BF16 if rng.random() < 0.7 else synth.F32


def _offsets(rng, vec):
    r = rng.random()
    if r < 0.5:
        return (0, 0)
    if r < 0.7:
        o = int(rng.integers(0, vec))
        return (o, o)
    return (int(rng.integers(0, vec)), int(rng.integers(0, vec)))


def _workload(rng, V, dtype, T, elems=12_000_000):
    """A dense or ragged batch of at most about `elems` logits."""
    if V < 64:
        return handmade(int(rng.integers(1, 9)), int(rng.integers(0, 9)), V, dtype, T=T,
                        seed=int(rng.integers(0, 1 << 30)))
    maxrows = max(2, elems // V)
    seed = int(rng.integers(0, 1 << 30))
    agreement = float(rng.uniform(0.3, 0.95))
    if rng.random() < 0.5:
        g = int(rng.integers(0, 129)) if (V <= 6000 and rng.random() < 0.15) else int(rng.integers(0, 17))
        B = int(rng.integers(1, max(1, min(48, maxrows // (2 * g + 1))) + 1))
        return synth.make_stochastic(B, V, dtype, T, seed=seed, gamma=g, agreement=agreement)
    lo = int(rng.integers(0, 6))
    hi = int(rng.integers(lo, 17))
    B = int(rng.integers(1, max(1, min(48, maxrows // (2 * hi + 1))) + 1))
    return synth.make_stochastic(B, V, dtype, T, seed=seed, gamma_range=(lo, hi), agreement=agreement)


def _run_cases(kind, fn, seed):
    rng = np.random.default_rng([20261202, seed])
    for i in range(CASES):
        desc = {}
        try:
            fn(rng, desc)
        except Exception as e:
            raise AssertionError(f"{kind} case {i}: {desc}") from e


def test_random_stochastic(dev):
    def one(rng, desc):
        dtype = _dtype(rng)
        V, T = _V(rng), float(rng.uniform(0.3, 1.5))
        w = _workload(rng, V, dtype, T)
        off = _offsets(rng, 8 if dtype == synth.BF16 else 4)
        opts, Td, pos, mbl = {}, None, None, 0
        if rng.random() < 0.3:
            Td = opts["temperature_draft"] = float(rng.uniform(0.2, 1.2))
        if rng.random() < 0.2:
            pos = opts["position"] = rng.integers(1, 3000, size=w.B).astype(np.int32)
        if rng.random() < 0.2:
            mbl = opts["min_block_len"] = int(rng.integers(2, 5))
        want_nkl = rng.random() < 0.8
        desc.update(V=V, dtype=dtype, B=w.B, dense=w.dense, gamma_max=w.gamma_max, T=T, offsets=off, T_draft=Td,
                    position=pos is not None, min_block_len=mbl, nkl=want_nkl)
        res = run_stochastic(w, dev, offset=off, options=opts or None, want_nkl=want_nkl)
        assert int(res["device_status"][0]) == 0
        compare_stochastic(w, res, range(w.B), T_draft=Td, positions=pos, min_block_len=mbl)
    _run_cases("stochastic", one, 1)


def test_random_greedy(dev):
    def one(rng, desc):
        dtype = _dtype(rng)
        V = _V(rng)
        w = _workload(rng, V, dtype, 1.0)
        off = int(rng.integers(0, 8 if dtype == synth.BF16 else 4)) if rng.random() < 0.5 else 0
        mbl = int(rng.integers(2, 5)) if rng.random() < 0.3 else 0
        desc.update(V=V, dtype=dtype, B=w.B, dense=w.dense, gamma_max=w.gamma_max, offset=off, min_block_len=mbl)
        res = run_greedy(w, dev, options={"min_block_len": mbl} if mbl else None, offset=off)
        assert int(res["device_status"][0]) == 0
        compare_greedy(w, res, range(w.B), min_block_len=mbl)
    _run_cases("greedy", one, 2)


def test_random_nkl(dev):
    def one(rng, desc):
        dtype = _dtype(rng)
        V, T = _V(rng), float(rng.uniform(0.3, 1.5))
        w = _workload(rng, V, dtype, T)
        off = _offsets(rng, 8 if dtype == synth.BF16 else 4)
        pos = rng.integers(1, 3000, size=w.B).astype(np.int32) if rng.random() < 0.3 else None
        desc.update(V=V, dtype=dtype, B=w.B, dense=w.dense, gamma_max=w.gamma_max, T=T, offsets=off,
                    position=pos is not None)
        res = run_nkl(w, dev, positions=pos, offset=off)
        assert int(res["device_status"][0]) == 0
        compare_nkl(w, res, range(w.B), positions=pos)
    _run_cases("nkl", one, 3)


def test_random_tree(dev):
    def one(rng, desc):
        dtype = _dtype(rng)
        V = max(8, _V(rng))
        N = int(rng.integers(1, 65))
        parent = [-1] + [int(rng.integers(-1, j)) if rng.random() < 0.7 else j - 1 for j in range(1, N)]
        B = int(rng.integers(1, max(1, min(24, 8_000_000 // (V * (N + 1)))) + 1))
        t32 = rng.normal(0, 1, (B * (N + 1), V)).astype(np.float32)
        hot = int(rng.integers(0, V))
        t32[:, hot] = 5.0                        # most nodes match their parent's argmax
        if rng.random() < 0.3:
            t32[:, (hot + 1) % V] = 5.0          # a tie: the lower index wins
        tok = np.where(rng.random((B, N)) < 0.85, hot, rng.integers(0, V, (B, N))).astype(np.int32)
        w = synth.TreeWorkload(B=B, N=N, V=V, dtype=dtype, parent=np.array(parent, np.int32),
                               target=synth.storage(t32, dtype), node_tokens=tok)
        off = int(rng.integers(0, 8 if dtype == synth.BF16 else 4)) if rng.random() < 0.4 else 0
        desc.update(V=V, dtype=dtype, B=B, N=N, offset=off)
        res = run_tree(w, dev, offset=off)
        assert int(res["device_status"][0]) == 0
        compare_tree(w, res, range(B))
    _run_cases("tree", one, 4)


def test_random_multi(dev):
    def one(rng, desc):
        dtype = _dtype(rng)
        K, gamma = int(rng.integers(2, 5)), int(rng.integers(0, 9))
        V = max(16, _V(rng))
        G = int(rng.integers(1, max(1, min(12, 8_000_000 // (V * K * (2 * gamma + 1)))) + 1))
        T = float(rng.uniform(0.4, 1.3))
        stochastic = bool(rng.random() < 0.6)
        w = synth.make_multi(G, K, gamma, V, dtype, T, seed=int(rng.integers(0, 1 << 30)))
        desc.update(V=V, dtype=dtype, G=G, K=K, gamma=gamma, T=T, stochastic=stochastic)
        res = api.spec_verify_multi(to_dev(w.target, dev), to_dev(w.draft, dev), to_dev(w.tokens, dev), K, w.T,
                                    stochastic=stochastic, u_accept=to_dev(w.u_accept, dev),
                                    u_sample=to_dev(w.u_sample, dev), consensus_nkl=0.1, divergence_nkl=0.15)
        torch.cuda.synchronize()
        res = {k: v.cpu().numpy() for k, v in res.items()}
        assert int(res["device_status"][0]) == 0
        ref = O.verify_multi(w.target, w.draft, w.tokens, G, K, gamma, w.T, w.dtype, stochastic, w.u_accept,
                             w.u_sample, 0.1, 0.15)
        mismatched = 0
        for g in range(G):
            r = ref[g]
            same = True
            for k, c in enumerate(r["cand"]):
                b = g * K + k
                ok = int(res["n_accepted"][b]) == c["n"] and \
                    list(res["out_tokens"][b * (gamma + 1):(b + 1) * (gamma + 1)]) == list(c["tokens"])
                assert ok or c["flag"], (g, k)
                same = same and ok
            if same:
                assert int(res["best_k"][g]) == r["best_k"] and int(res["best_n"][g]) == r["best_n"], g
                assert list(res["best_tokens"][g * (gamma + 1):(g + 1) * (gamma + 1)]) == list(r["best_tokens"]), g
            else:
                mismatched += 1
            if gamma:
                got = res["pair_nkl"][g * gamma * K * K:(g + 1) * gamma * K * K].reshape(gamma, K, K)
                assert np.allclose(got.astype(np.float64), r["pair_nkl"], rtol=REL, atol=NKL_ABS, equal_nan=True), g
        assert mismatched <= 1
    _run_cases("multi", one, 5)
