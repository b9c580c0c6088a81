"""Randomised layouts against the oracle: vocabularies of every length class (a single
element, less than one 16-byte block, rows of whole blocks and not, one to three
vocabulary chunks), logit buffers shifted by random element counts (target and draft alike
or apart), both dtypes, dense and ragged batches; every stochastic (with its greedy and NKL
outputs), greedy and NKL output compared with the oracle on every sequence. The partial
16-byte blocks at the chunks' ends are the point: stochastic rows fold their elements in
the row merge of the finalisation, the NKL and greedy tiles fold them themselves."""
import numpy as np
import pytest
import torch

from speculative_decoding_token_temp_gb300 import synth

from gpu_util import (compare_greedy, compare_nkl, compare_stochastic, handmade, run_greedy, run_nkl,
                      run_stochastic)

pytestmark = pytest.mark.gpu

_VOCABS = [1, 2, 7, 9, 15, 17, 1000, 4095, 4097, 8191, 32003, 50257, 65535, 65537, 70001, 131073, 140001]


def _cases():
    rng = np.random.default_rng(20261202)
    out = []
    for i, V in enumerate(_VOCABS):
        dtype = synth.BF16 if i % 3 != 2 else synth.F32
        vec = 8 if dtype == synth.BF16 else 4
        ot = int(rng.integers(0, vec))
        od = ot if rng.random() < 0.4 else int(rng.integers(0, vec))
        out.append((V, dtype, ot, od, int(rng.integers(1, 1 << 30))))
    return out


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


@pytest.mark.parametrize("V,dtype,ot,od,seed", _cases())
def test_random_layout(dev, V, dtype, ot, od, seed):
    if V < 64:
        w = handmade(3, 4, V, dtype, T=0.9, seed=seed % 1000)  # dense; the generator wants more tokens
    else:
        B = 3 if V > 100000 else 5
        w = synth.make_stochastic(B, V, dtype, 0.8, seed=seed % 100000, gamma_range=(0, 6), agreement=0.7)
    res = run_stochastic(w, dev, offset=(ot, od))
    assert int(res["device_status"][0]) == 0
    compare_stochastic(w, res, range(w.B))
    g = run_greedy(w, dev, offset=ot)
    assert int(g["device_status"][0]) == 0
    compare_greedy(w, g, range(w.B))
    n = run_nkl(w, dev, offset=(ot, od))
    assert int(n["device_status"][0]) == 0
    compare_nkl(w, n, range(w.B))
