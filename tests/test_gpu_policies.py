"""GPU parity of the policy variants (spec_options) against the oracle: a draft
temperature of its own, the position-adaptive NKL mask, block-accept and the device
acceptance statistics. Same tolerances as test_gpu_parity.py."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from speculative_decoding_token_temp_gb300 import _lib, api, synth

from gpu_util import (compare_greedy, compare_nkl, compare_stochastic, handmade, run_greedy, run_nkl,
                      run_stochastic)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def _argmax_drafts(w, frac, seed):
    """Each draft token becomes the target argmax of its position with probability frac,
    so that runs of matches (block-accept) and accepted prefixes occur."""
    rng = np.random.default_rng(seed)
    for b in range(w.B):
        g = int(w.gammas[b])
        t0, d0 = w.target_base(b), w.draft_base(b)
        if g == 0:
            continue
        am = np.argmax(O.widen(w.target[t0:t0 + g], w.dtype), axis=1)
        w.tokens[d0:d0 + g] = np.where(rng.random(g) < frac, am, w.tokens[d0:d0 + g])
    return w


# ---------------------------------------------------------------- separate temperatures

@pytest.mark.parametrize("V,dtype,offset", [(4096, synth.BF16, 0), (128256, synth.BF16, 0), (40000, synth.F32, 0),
                                            (4097, synth.BF16, 0), (5000, synth.BF16, 1)])
def test_separate_draft_temperature(dev, V, dtype, offset):
    """T_t = 0.8, T_d = 0.4 ([PD] 4.4's ranges): q(x), alpha and the residual at T_d, NKL at
    T_t; vector path (one and several chunks), staged path (odd V), phased tiles (rows
    shifted by one element)."""
    w = handmade(4, 5, V, dtype, T=0.8, seed=V + offset)
    w.draft[:] = synth.storage(0.5 * O.widen(w.draft, w.dtype), dtype)  # a peakier drafter at T_d = 0.4
    res = run_stochastic(w, dev, offset=offset, options={"temperature_draft": 0.4})
    assert res["device_status"][0] == 0
    compare_stochastic(w, res, range(w.B), T_draft=0.4)


@pytest.mark.parametrize("V,dtype,offset", [(128256, synth.BF16, 0), (5000, synth.BF16, 1), (40000, synth.F32, 0),
                                            (50257, synth.BF16, 0)])
def test_separate_draft_temperature_without_nkl(dev, V, dtype, offset):
    """Without the NKL outputs (the only ones that need the draft row at the target's
    temperature as well) a call with its own draft temperature runs on the single-scale
    tiles, the draft at T_d alone: decisions, p(x), q(x), alpha and the greedy outputs as the
    oracle's, on aligned rows, rows shifted by one element, and a vocabulary off the grid."""
    w = handmade(4, 5, V, dtype, T=0.8, seed=V + 7 + offset)
    w.draft[:] = synth.storage(0.5 * O.widen(w.draft, w.dtype), dtype)
    res = run_stochastic(w, dev, offset=offset, options={"temperature_draft": 0.4}, want_nkl=False)
    assert res["device_status"][0] == 0 and "nkl" not in res
    compare_stochastic(w, res, range(w.B), T_draft=0.4)


def test_draft_temperature_equal_to_target_is_the_plain_call(dev):
    w = handmade(6, 4, 32000, synth.BF16, T=0.7, seed=81)
    a = run_stochastic(w, dev)
    b = run_stochastic(w, dev, options={"temperature_draft": 0.7})
    for k in ("n_accepted", "out_tokens", "p_x", "q_x", "alpha", "nkl", "nkl_mask", "greedy_tokens"):
        assert np.array_equal(a[k], b[k]), k


def test_separate_temperature_on_the_synthetic_generator(dev):
    """Drafts sampled at T_d from the generator's draft rows (the lossless setting)."""
    w = synth.make_stochastic(24, 32000, synth.BF16, 0.4, seed=82, gamma_range=(1, 8), agreement=0.8)
    res = run_stochastic(w, dev, T=0.9, options={"temperature_draft": 0.4})
    assert res["device_status"][0] == 0
    compare_stochastic(w, res, range(w.B), T=0.9, T_draft=0.4)


# ---------------------------------------------------------------- position-adaptive mask

def test_position_adaptive_mask(dev):
    w = synth.make_stochastic(16, 32000, synth.BF16, 0.8, seed=83, gamma_range=(1, 8), agreement=0.8)
    rng = np.random.default_rng(83)
    pos = rng.integers(1, 4000, w.B).astype(np.int32)
    pos[3] = 1
    res = run_stochastic(w, dev, options={"position": pos})
    assert res["device_status"][0] == 0
    compare_stochastic(w, res, range(w.B), positions=pos)
    nk = run_nkl(w, dev, positions=pos)
    compare_nkl(w, nk, range(w.B), positions=pos)
    nkl = res["nkl"].astype(np.float64)
    print("NKL range", float(np.nanmin(nkl)), float(np.nanmax(nkl)))


def test_position_below_one_is_reported(dev):
    w = synth.make_stochastic(5, 4096, synth.BF16, 0.8, seed=84, gamma_range=(2, 4), agreement=0.8)
    pos = np.array([1, 0, 7, -3, 100], dtype=np.int32)
    res = run_stochastic(w, dev, options={"position": pos})
    assert res["device_status"][0] == _lib.SPEC_DEV_POSITION
    compare_stochastic(w, res, range(w.B), positions=pos)
    nk = run_nkl(w, dev, positions=pos)
    assert nk["device_status"][0] == _lib.SPEC_DEV_POSITION
    compare_nkl(w, nk, range(w.B), positions=pos)


# ---------------------------------------------------------------- block-accept

@pytest.mark.parametrize("min_len", [1, 3, 5])
def test_block_accept(dev, min_len):
    w = _argmax_drafts(handmade(12, 12, 5000, synth.BF16, seed=85 + min_len), 0.8, 85)
    g = run_greedy(w, dev, options={"min_block_len": min_len})
    assert g["device_status"][0] == 0
    compare_greedy(w, g, range(w.B), min_block_len=min_len)
    assert np.any(g["block_n"] > 0) and np.any(g["block_n"] > g["n_accepted"])
    s = run_stochastic(w, dev, options={"min_block_len": min_len})
    compare_stochastic(w, s, range(w.B), min_block_len=min_len)


def test_block_accept_ragged_and_errors(dev):
    w = _argmax_drafts(synth.make_stochastic(9, 3000, synth.BF16, 0.8, seed=86, gamma_range=(0, 9),
                                             agreement=0.7), 0.9, 86)
    g = run_greedy(w, dev, options={"min_block_len": 3})
    compare_greedy(w, g, range(w.B), min_block_len=3)
    bad = handmade(3, 4, 600, synth.F32, seed=87)
    bad.target[5, 7] = np.float32(np.nan)   # a row of sequence 1
    r = run_greedy(bad, dev, options={"min_block_len": 3})
    assert r["block_n"][1] == -1 and np.all(r["block_tokens"][4:8] == -1)
    compare_greedy(bad, r, [0, 2], min_block_len=3)


@pytest.mark.parametrize("ragged", [False, True])
def test_block_accept_without_drafts(dev, ragged):
    """A batch in which no sequence has a draft: block_tokens has no elements (its pointer
    is NULL), every block_n is 0, and the greedy and stochastic decisions are the bonus
    tokens alone."""
    if ragged:
        w = synth.make_stochastic(5, 777, synth.BF16, 0.8, seed=88, gamma_range=(0, 0))
    else:
        w = handmade(6, 0, 4097, synth.F32, seed=88)
    g = run_greedy(w, dev, options={"min_block_len": 3})
    assert g["device_status"][0] == 0 and np.all(g["block_n"] == 0)
    compare_greedy(w, g, range(w.B), min_block_len=3)
    s = run_stochastic(w, dev, options={"min_block_len": 3})
    assert s["device_status"][0] == 0 and np.all(s["block_n"] == 0)
    compare_stochastic(w, s, range(w.B), min_block_len=3)


# ---------------------------------------------------------------- acceptance statistics

def test_acceptance_statistics_over_buckets(dev):
    """Calls of both modes in several time buckets, one bucket reusing a slot of the ring
    (3 and 3 + 64), ragged batches with empty sequences; summaries over several windows
    against the oracle's definition on the same per-sequence counts."""
    stats = api.new_accept_stats(dev)
    records = []
    plan = [(1, "stoch", 90), (1, "greedy", 91), (2, "stoch", 92), (3, "greedy", 93), (3 + 64, "stoch", 94),
            (3 + 64, "greedy", 95), (70, "stoch", 96)]
    for bucket, mode, seed in plan:
        w = _argmax_drafts(synth.make_stochastic(20, 4096, synth.BF16, 0.8, seed=seed, gamma_range=(0, 8),
                                                 agreement=0.8), 0.6, seed)
        opts = {"stats": stats, "stats_bucket": bucket}
        res = run_stochastic(w, dev, options=opts) if mode == "stoch" else run_greedy(w, dev, options=opts)
        assert res["device_status"][0] == 0
        records += [(bucket, int(res["n_accepted"][b]), int(w.gammas[b])) for b in range(w.B)]
    for now, window in [(70, 1), (70, 4), (67, 1), (67, 64), (2, 2), (5, 3)]:
        got = api.spec_accept_summary(stats, now, window).cpu().numpy()
        live = [r for r in records if r[0] != 3]   # bucket 67 took slot 3 over: bucket 3 is gone
        want = O.acceptance_summary(live, now, window)
        assert got[0] == want["rounds"] and got[1] == want["accepted"] and got[2] == want["drafted"], (now, window)
        assert got[3] == pytest.approx(want["mean_accepted"], rel=1e-12, abs=1e-12)
        assert got[4] == pytest.approx(want["mean_rate"], rel=1e-9, abs=1e-9)
        assert abs(got[5] ** 2 - want["arsd"] ** 2) <= 1e-9, (now, window, got[5], want["arsd"])
