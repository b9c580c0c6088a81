"""GPU parity of multi-draft verification (spec_verify_multi) against the oracle: every
candidate's result, the kept candidate and its tokens, the pairwise NKL matrix and the
consensus / divergence flags. Tolerances as in test_gpu_parity.py."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from speculative_decoding_token_temp_gb300 import _lib, api, synth

from gpu_util import NKL_ABS, REL, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def run_multi(w, K, dev, stochastic, c_thr=0.1, d_thr=0.15):
    res = api.spec_verify_multi(to_dev(w.target, dev), to_dev(w.draft, dev), to_dev(w.tokens, dev), K, w.T,
                                stochastic=stochastic, u_accept=to_dev(w.u_accept, dev),
                                u_sample=to_dev(w.u_sample, dev), consensus_nkl=c_thr, divergence_nkl=d_thr)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in res.items()}


def compare_multi(w, res, G, K, gamma, stochastic, c_thr=0.1, d_thr=0.15):
    ref = O.verify_multi(w.target, w.draft, w.tokens, G, K, gamma, w.T, w.dtype, stochastic, w.u_accept,
                         w.u_sample, c_thr, d_thr)
    mismatched = 0
    for g in range(G):
        r = ref[g]
        flagged = any(c["flag"] for c in r["cand"])
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
            assert flagged
            mismatched += 1
        got = res["pair_nkl"][g * gamma * K * K:(g + 1) * gamma * K * K].reshape(gamma, K, K).astype(np.float64)
        assert np.allclose(got, r["pair_nkl"], rtol=REL, atol=NKL_ABS, equal_nan=True), (g, got, r["pair_nkl"])
        for i in range(gamma):
            M = r["pair_nkl"][i]
            off = [(a, bb) for a in range(K) for bb in range(K) if a != bb]
            near_c = any(abs(M[a, bb] - c_thr) <= REL * c_thr + NKL_ABS for a, bb in off)
            near_d = any(abs(M[a, bb] - d_thr) <= REL * d_thr + NKL_ABS for a, bb in off)
            assert res["consensus"][g * gamma + i] == r["consensus"][i] or near_c, (g, i)
            assert res["divergence"][g * gamma + i] == r["divergence"][i] or near_d, (g, i)
    assert mismatched <= 1
    return ref


@pytest.mark.parametrize("K,V,dtype,stochastic", [(2, 4096, synth.BF16, False), (3, 32000, synth.BF16, True),
                                                  (4, 128256, synth.BF16, False), (3, 5001, synth.F32, True),
                                                  (4, 40000, synth.F32, True), (3, 128256, synth.BF16, True),
                                                  (2, 50257, synth.BF16, False), (3, 50257, synth.BF16, True)])
def test_multi_draft(dev, K, V, dtype, stochastic):
    G, gamma = 6, 4
    w = synth.make_multi(G, K, gamma, V, dtype, 0.8, seed=K * 1000 + V % 997)
    res = run_multi(w, K, dev, stochastic)
    assert res["device_status"][0] == 0
    ref = compare_multi(w, res, G, K, gamma, stochastic)
    assert any(np.any(ref[g]["consensus"]) for g in range(G)) and any(np.any(ref[g]["divergence"]) for g in range(G))
    # every candidate's result is the batch call's on the same G*K sequences
    t, d, tok = to_dev(w.target, dev), to_dev(w.draft, dev), to_dev(w.tokens, dev)
    if stochastic:
        b = api.spec_verify_stochastic(t, d, tok, w.T, to_dev(w.u_accept, dev), to_dev(w.u_sample, dev), gamma=gamma)
    else:
        b = api.spec_verify_greedy(t, tok, gamma=gamma)
    assert np.array_equal(b["n_accepted"].cpu().numpy(), res["n_accepted"])
    assert np.array_equal(b["out_tokens"].cpu().numpy(), res["out_tokens"])


def test_multi_draft_edge_cases(dev):
    # gamma = 0: nothing to compare, every candidate keeps 0 drafts
    w = synth.make_multi(3, 2, 0, 300, synth.BF16, 0.8, seed=5)
    res = run_multi(w, 2, dev, True)
    assert np.all(res["best_k"] == 0) and np.all(res["best_n"] == 0)
    compare_multi(w, res, 3, 2, 0, True)
    # a non-finite row in one candidate: that candidate is an error, its matrix entries NaN
    G, K, gamma, V = 3, 3, 3, 3000
    w = synth.make_multi(G, K, gamma, V, synth.F32, 0.8, seed=6)
    w.draft[(1 * K + 2) * gamma + 1, 17] = np.float32(np.inf)
    res = run_multi(w, K, dev, False)
    assert res["device_status"][0] & _lib.SPEC_DEV_NONFINITE
    M = res["pair_nkl"][(1 * gamma + 1) * K * K:(1 * gamma + 2) * K * K].reshape(K, K)
    assert np.isnan(M[2, 0]) and np.isnan(M[0, 2]) and not np.isnan(M[0, 1])
    ref = O.verify_multi(w.target, w.draft, w.tokens, G, K, gamma, w.T, w.dtype, False)
    for g in range(G):
        assert int(res["best_k"][g]) == ref[g]["best_k"] and int(res["best_n"][g]) == ref[g]["best_n"]
    # the thresholds are parameters
    w = synth.make_multi(4, 3, 2, 4096, synth.BF16, 0.8, seed=7)
    res = run_multi(w, 3, dev, False, c_thr=0.3, d_thr=0.05)
    compare_multi(w, res, 4, 3, 2, False, c_thr=0.3, d_thr=0.05)
