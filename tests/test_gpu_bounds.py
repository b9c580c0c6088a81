"""The bounds-checked build (libspecverify_bounds.so, SPEC_BOUNDS_CHECK=1) on the layouts whose
index arithmetic is the most intricate: vocabularies off the 16-byte grid, buffers shifted
by whole elements (rows at one offset and pairs at two), ragged batches with empty
sequences, non-monotone offsets, trees of several shapes, multi-draft groups on both of
their paths, the longest drafts, a vocabulary whose slice table outgrows shared memory.
In that build every computed access is checked against its buffer (widened to the 16-byte
blocks holding its first and last byte) and one outside sets SPEC_DEV_BOUNDS instead of
touching memory; here the bit must stay clear, and every output must equal the ordinary
build's on the same inputs."""
import contextlib

import numpy as np
import pytest
import torch

from speculative_decoding_token_temp_gb300 import _lib, api, synth

from gpu_util import handmade, put, run_greedy, run_nkl, run_stochastic, run_tree, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


@pytest.fixture(scope="module")
def checked(dev):
    return _lib.bounds_lib()


@contextlib.contextmanager
def using(handle):
    saved = _lib._LIB
    _lib._LIB = handle
    try:
        yield
    finally:
        _lib._LIB = saved


def both(checked, fn):
    """fn() through the ordinary library, then through the bounds-checked one."""
    plain = fn()
    with using(checked):
        chk = fn()
    return plain, chk


def same(plain, chk, allow=0):
    """No SPEC_DEV_BOUNDS in the checked run, the same status otherwise, equal outputs."""
    st_p, st_c = int(plain["device_status"][0]), int(chk["device_status"][0])
    assert st_c & _lib.SPEC_DEV_BOUNDS == 0, st_c
    assert st_p == st_c and (st_p & ~allow) == 0, (st_p, st_c)
    for k, v in plain.items():
        if k == "device_status":
            continue
        a, b = np.asarray(v), np.asarray(chk[k])
        if a.dtype.kind == "f":
            assert np.array_equal(a, b, equal_nan=True), k
        else:
            assert np.array_equal(a, b), k


@pytest.mark.parametrize("V", [1, 7, 9, 4097, 40000])
@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
def test_odd_vocabularies(dev, checked, V, dtype):
    w = handmade(3, 3, V, dtype, T=0.8, seed=V)
    same(*both(checked, lambda: run_stochastic(w, dev)))
    same(*both(checked, lambda: run_greedy(w, dev)))
    same(*both(checked, lambda: run_nkl(w, dev)))


@pytest.mark.parametrize("offset", [1, (0, 3), (5, 2), (2, 7)])
@pytest.mark.parametrize("V,dtype", [(3 * 4096 + 37, synth.BF16), (3 * 4096, synth.BF16), (5001, synth.F32)])
def test_rows_off_the_grid(dev, checked, offset, V, dtype):
    w = handmade(4, 5, V, dtype, T=0.7, seed=11 + V % 7)
    same(*both(checked, lambda: run_stochastic(w, dev, offset=offset)))
    same(*both(checked, lambda: run_nkl(w, dev, offset=offset)))
    ot = offset[0] if isinstance(offset, tuple) else offset
    same(*both(checked, lambda: run_greedy(w, dev, offset=ot)))


def test_ragged_batch_with_empty_sequences(dev, checked):
    w = synth.make_stochastic(9, 3000, synth.BF16, 0.8, seed=26, gamma_range=(0, 5), agreement=0.7)
    same(*both(checked, lambda: run_stochastic(w, dev)))
    same(*both(checked, lambda: run_greedy(w, dev)))
    same(*both(checked, lambda: run_nkl(w, dev)))
    w = synth.make_stochastic(40, 50257, synth.BF16, 0.8, seed=27, gamma_range=(0, 9), agreement=0.7)
    same(*both(checked, lambda: run_stochastic(w, dev)))


def test_non_monotone_offsets(dev, checked):
    """Offsets out of order are reported as SPEC_DEV_OFFSETS, and no access leaves its buffer."""
    def call():
        cu = torch.tensor([0, 5, 3, 8], dtype=torch.int32, device=dev)
        t = torch.zeros(11, 64, dtype=torch.bfloat16, device=dev)
        d = torch.zeros(8, 64, dtype=torch.bfloat16, device=dev)
        r = api.spec_verify_stochastic(t, d, torch.zeros(8, dtype=torch.int32, device=dev), 1.0,
                                       torch.zeros(8, device=dev), torch.zeros(3, device=dev), cu_draft=cu, gamma=5)
        torch.cuda.synchronize()
        return {"device_status": r["device_status"].cpu().numpy()}
    plain, chk = both(checked, call)
    assert int(plain["device_status"][0]) & _lib.SPEC_DEV_OFFSETS
    assert int(chk["device_status"][0]) & _lib.SPEC_DEV_OFFSETS
    assert int(chk["device_status"][0]) & _lib.SPEC_DEV_BOUNDS == 0


def test_trees(dev, checked):
    rng = np.random.default_rng(30)
    for parent in ([-1], [-1, 0, 0, 1, 2, -1], list(range(-1, 63))):
        N = len(parent)
        t32 = rng.normal(0, 1, (5 * (N + 1), 300)).astype(np.float32)
        t32[:, 7] = 5.0
        tok = np.where(rng.random((5, N)) < 0.85, 7, rng.integers(0, 300, (5, N))).astype(np.int32)
        w = synth.TreeWorkload(B=5, N=N, V=300, dtype=synth.BF16, parent=np.array(parent, np.int32),
                               target=synth.storage(t32, synth.BF16), node_tokens=tok)
        same(*both(checked, lambda: run_tree(w, dev)))
    w = synth.make_tree(6, 3001, synth.BF16, seed=5)
    same(*both(checked, lambda: run_tree(w, dev, offset=3)))


@pytest.mark.parametrize("K,V,dtype,stochastic", [(3, 32000, synth.BF16, True), (4, 5001, synth.F32, True),
                                                  (3, 50257, synth.BF16, True), (2, 4096, synth.BF16, False)])
def test_multi_draft(dev, checked, K, V, dtype, stochastic):
    w = synth.make_multi(4, K, 3, V, dtype, 0.8, seed=K * 100 + V % 97)

    def call():
        res = api.spec_verify_multi(to_dev(w.target, dev), to_dev(w.draft, dev), to_dev(w.tokens, dev), K, w.T,
                                    stochastic=stochastic, u_accept=to_dev(w.u_accept, dev),
                                    u_sample=to_dev(w.u_sample, dev))
        torch.cuda.synchronize()
        return {k: v.cpu().numpy() for k, v in res.items()}
    same(*both(checked, call))


def test_longest_drafts_and_largest_tables(dev, checked):
    w = handmade(2, 128, 600, synth.F32, seed=21)
    same(*both(checked, lambda: run_stochastic(w, dev)))
    w = handmade(2, 2, 1500000, synth.F32, T=1.0, seed=3)     # slice table read from global memory
    same(*both(checked, lambda: run_stochastic(w, dev)))


def test_zero_residual_second_pass(dev, checked):
    """The sampler's second pass over p (a rejection on identical rows) on aligned and
    staged rows."""
    for V in (50000, 50001):
        z = np.full((1, V), -200.0, np.float32)
        z[:, [3, 1000, V - 1]] = 0.0
        same_row = synth.storage(z, synth.BF16)[0]
        rng = np.random.default_rng(V)
        t = synth.storage(rng.normal(0, 2, (2 * 3, V)).astype(np.float32), synth.BF16)
        d = synth.storage(rng.normal(0, 2, (2 * 2, V)).astype(np.float32), synth.BF16)
        t[0], d[0], t[3 + 1], d[2 + 1] = same_row, same_row, same_row, same_row
        w = synth.StochasticWorkload(B=2, V=V, dtype=synth.BF16, T=1.0, gammas=np.full(2, 2, np.int32),
                                     cu_draft=np.array([0, 2, 4], np.int32), target=t, draft=d,
                                     tokens=rng.integers(0, V, 4).astype(np.int32),
                                     u_accept=np.array([1.5, 0.0, 0.0, 1.5], np.float32),
                                     u_sample=np.array([0.2, 0.7], np.float32))
        same(*both(checked, lambda: run_stochastic(w, dev)))


def test_static_scratch(dev, checked):
    w = handmade(6, 4, 20000, synth.BF16, T=0.9, seed=77)

    def call():
        t, d = put(w.target, dev), put(w.draft, dev)
        res = api.spec_verify_stochastic_static(t, d, to_dev(w.tokens, dev), w.T, to_dev(w.u_accept, dev),
                                                to_dev(w.u_sample, dev), gamma=4)
        torch.cuda.synchronize()
        return {k: v.cpu().numpy() for k, v in res.items()}
    same(*both(checked, call))
