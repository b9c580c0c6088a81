"""GPU parity: the CUDA library, called through the C ABI, against the fp64 oracle.

Tolerances: accepted counts and tokens bit-exact in greedy and tree modes, and in
stochastic mode except the sequences the oracle flags (a decision within 1e-5 of its
boundary); p(x), q(x), alpha and NKL within 1e-4 relative of fp64 (NKL also within an
absolute 2e-6 near zero)."""
import numpy as np
import pytest
import scipy.stats
import torch

from oracle import oracle as O
from speculative_decoding_token_temp_gb300 import _lib, api, synth

import oracle_pool
from gpu_util import (compare_greedy, compare_nkl, compare_stochastic, compare_tree, handmade, run_greedy,
                      run_nkl, run_stochastic, run_tree, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


_CACHE = {}


def workload(cfg):
    if cfg.name not in _CACHE:
        _CACHE[cfg.name] = cfg.make()
    return _CACHE[cfg.name]


# ---------------------------------------------------------------- the five workloads

def test_tiny_B1_g4_V1000_f32(dev):
    w = workload(synth.TINY)
    res = run_stochastic(w, dev)
    compare_stochastic(w, res, range(w.B))
    assert res["device_status"][0] == 0
    compare_greedy(w, run_greedy(w, dev), range(w.B))
    compare_nkl(w, run_nkl(w, dev), range(w.B))


@pytest.mark.parametrize("T", [0.6, 1.0])
def test_B64_g5_V32000_bf16_all_sequences(dev, T):
    w = synth.MID.make(T=T)
    res = run_stochastic(w, dev)
    n, flagged, mismatched = compare_stochastic(w, res, range(w.B))
    _report(f"B=64 stochastic T={T}", w, n, flagged, mismatched)
    assert res["device_status"][0] == 0
    compare_greedy(w, run_greedy(w, dev), range(w.B))
    compare_nkl(w, run_nkl(w, dev), range(w.B))


def _oracle(kind, w, key=None, **kw):
    """The oracle over every sequence of w, on every host core, cached per workload."""
    k = (w.name, w.B, w.V, w.T, w.dtype, kind, key)
    if k not in _ORACLE:
        _ORACLE[k] = oracle_pool.oracle_batch(kind, w, **kw)
    return _ORACLE[k]


_ORACLE = {}


def _report(label, w, n, flagged, mismatched):
    """One line per workload: sequences compared, band-flagged by the oracle (a decision
    within 1e-5 of its boundary), and differing (at most max(1, 1e-4 of the rows))."""
    rows = int(w.total_target)
    print(f"PARITY {label}: {n} sequences ({rows} target rows) compared, {flagged} band-flagged by the oracle "
          f"({flagged / max(rows, 1):.2e} of rows), {mismatched} differ (budget max(1, 1e-4 of rows) = "
          f"{max(1, int(1e-4 * rows))})")


def test_headline_B256_g8_V128256_all_sequences(dev):
    """Every sequence of the headline batch against the oracle: the stochastic decisions
    (count and tokens bit-exact except flagged sequences, at most max(1, 1e-4 of the rows)
    of them differing), p(x), q(x), alpha, NKL and its mask, and the fused greedy outputs;
    the standalone greedy call; properties that hold at any size."""
    w = workload(synth.HEADLINE)
    res = run_stochastic(w, dev)
    assert res["device_status"][0] == 0
    n_cmp, flagged, mismatched = compare_stochastic(w, res, range(w.B), ref=_oracle("stochastic", w))
    _report("headline stochastic", w, n_cmp, flagged, mismatched)
    g = run_greedy(w, dev)
    compare_greedy(w, g, range(w.B), ref=_oracle("greedy", w))
    assert np.array_equal(g["n_accepted"], res["greedy_n"])
    assert np.array_equal(g["out_tokens"], res["greedy_tokens"])
    n = res["n_accepted"]
    assert np.all((n >= 0) & (n <= 8))
    out = res["out_tokens"].reshape(w.B, 9)
    for b in range(w.B):
        assert np.all(out[b, :n[b]] == w.tokens[b * 8:b * 8 + n[b]])
        assert 0 <= out[b, n[b]] < w.V and np.all(out[b, n[b] + 1:] == -1)
    assert np.all(res["alpha"] <= 1.0) and np.all(res["alpha"] > 0)
    assert np.all(res["nkl"] >= -NKL_FLOOR)


NKL_FLOOR = 1e-6


def test_headline_nkl_standalone_all_pairs(dev):
    """spec_nkl on all 2048 (target, draft) row pairs of the headline batch."""
    w = workload(synth.HEADLINE)
    res = run_nkl(w, dev)
    assert res["device_status"][0] == 0
    compare_nkl(w, res, range(w.B), ref=_oracle("nkl", w))


def test_tree_B32_N12_V128256_all_sequences(dev):
    w = synth.TREE.make()
    res = run_tree(w, dev)
    assert res["device_status"][0] == 0
    compare_tree(w, res, range(w.B))


def test_ragged_B512_V152064_all_sequences(dev):
    """Every sequence of the ragged batch (gamma_b ~ U{1..16}, packed): stochastic with its
    fused NKL and greedy outputs, and the standalone greedy call."""
    w = workload(synth.RAGGED)
    assert not w.dense
    res = run_stochastic(w, dev)
    assert res["device_status"][0] == 0
    n_cmp, flagged, mismatched = compare_stochastic(w, res, range(w.B), ref=_oracle("stochastic", w))
    _report("ragged stochastic", w, n_cmp, flagged, mismatched)
    compare_greedy(w, run_greedy(w, dev), range(w.B), ref=_oracle("greedy", w))
    n = res["n_accepted"]
    assert np.all((n >= 0) & (n <= w.gammas))


def _live_rows(R, V, live, dtype):
    """R rows whose only live tokens (logit 0) are `live`; every other logit is -200, so
    that exp((-200 - 0) / T) underflows in fp32 and the rows' softmax is exact on both
    sides: 1/len(live) at the live tokens."""
    z = np.full((R, V), -200.0, np.float32)
    z[:, live] = 0.0
    return synth.storage(z, dtype)


@pytest.mark.parametrize("V,dtype", [(50000, synth.BF16), (50001, synth.BF16), (30000, synth.F32)])
def test_zero_residual_draws_from_p(dev, V, dtype):
    """Reading R6 on the GPU: a rejection whose residual max(0, p - q) is zero everywhere
    (identical target and draft rows) takes the sampler's second pass, which draws from p
    of the same row. Identical rows give alpha = 1, so a uniform above 1 forces the
    rejection (accept iff u <= alpha); the live tokens make the draw exact on both sides.
    V = 50001 (rows off the 16-byte grid) takes the staged sampler."""
    live = [3, 1000, 20000, V - 17, V - 1]
    B, g = 6, 3
    rng = np.random.default_rng(V)
    t = rng.normal(0, 2, (B * (g + 1), V)).astype(np.float32)
    d = rng.normal(0, 2, (B * g, V)).astype(np.float32)
    t_st, d_st = synth.storage(t, dtype), synth.storage(d, dtype)
    u_acc = np.zeros(B * g, np.float32)                      # u = 0 accepts every other position
    rej = [b % g for b in range(B)]                          # the rejected position of sequence b
    same = _live_rows(1, V, live, dtype)[0]
    tokens = rng.integers(0, V, B * g).astype(np.int32)
    for b in range(B):
        i = rej[b]
        t_st[b * (g + 1) + i] = same
        d_st[b * g + i] = same
        u_acc[b * g + i] = 1.5
    u_smp = np.array([0.1, 0.3, 0.5, 0.7, 0.9, 0.55], np.float32)
    w = synth.StochasticWorkload(B=B, V=V, dtype=dtype, T=1.0, gammas=np.full(B, g, np.int32),
                                 cu_draft=np.arange(B + 1, dtype=np.int32) * g, target=t_st, draft=d_st,
                                 tokens=tokens, u_accept=u_acc, u_sample=u_smp, name=f"zero residual V={V}")
    res = run_stochastic(w, dev)
    assert res["device_status"][0] == 0
    ref = O.verify_stochastic(w.target, w.draft, w.tokens, w.cu_draft, w.T, w.u_accept, w.u_sample, w.dtype)
    for b in range(B):
        r = ref[b]
        assert ("zero_residual", rej[b]) in r["flags"]
        want_y = live[int(u_smp[b] * len(live))]
        assert r["tokens"][rej[b]] == want_y                   # the oracle draws from p of that row
        assert int(res["n_accepted"][b]) == r["n"] == rej[b]
        t0 = b * (g + 1)
        assert list(res["out_tokens"][t0:t0 + g + 1]) == list(r["tokens"]), b


# ---------------------------------------------------------------- edge cases

@pytest.mark.parametrize("V", [1, 2, 7, 8, 9, 4095, 4096, 4097, 40000])
@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
def test_odd_vocab_sizes(dev, V, dtype):
    w = handmade(3, 3, V, dtype, T=0.8, seed=V)
    res = run_stochastic(w, dev)
    compare_stochastic(w, res, range(w.B))
    compare_greedy(w, run_greedy(w, dev), range(w.B))
    compare_nkl(w, run_nkl(w, dev), range(w.B))


# ---------------------------------------------------------------- rows off the 16-byte grid (phased and staged paths)

@pytest.mark.parametrize("offset", [0, 1, (0, 3), (5, 2)])
@pytest.mark.parametrize("V", [3 * 4096, 3 * 4096 + 37])
@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
def test_off_grid_offsets(dev, offset, V, dtype):
    """Base pointers shifted by whole elements (target and draft alike: the phased path when
    the rows are whole 16-byte blocks; apart: the staged path), and row lengths off the
    16-byte grid: several stages per tile and a ragged last stage, in every mode."""
    if offset == 0 and V % 8 == 0:
        pytest.skip("the aligned path")
    w = handmade(4, 5, V, dtype, T=0.7, seed=11 + V % 7)
    res = run_stochastic(w, dev, offset=offset)
    assert res["device_status"][0] == 0
    compare_stochastic(w, res, range(w.B))
    compare_nkl(w, run_nkl(w, dev, offset=offset), range(w.B))
    ot = offset[0] if isinstance(offset, tuple) else offset
    compare_greedy(w, run_greedy(w, dev, offset=ot), range(w.B))


def test_off_grid_ties_and_flat_rows(dev):
    """Lowest index of a tied maximum when the tied entries share one thread's strided
    group, sit in different groups, or fill a whole (flat) row."""
    V = 3000
    t = np.zeros((3, V), dtype=np.float32)
    t[0, [1256, 1000, 2900]] = 3.0       # 1000 and 1256 are one thread's elements, 256 apart
    t[2, [2999, 2998, 2742]] = 1.0       # 2742 = 2998 - 256: lowest is 2742
    d = np.zeros((2, V), dtype=np.float32)
    for dtype in (synth.F32, synth.BF16):
        w = synth.StochasticWorkload(B=1, V=V, dtype=dtype, T=1.0, gammas=np.array([2], np.int32),
                                     cu_draft=np.array([0, 2], np.int32), target=synth.storage(t, dtype),
                                     draft=synth.storage(d, dtype), tokens=np.array([1000, 0], np.int32),
                                     u_accept=np.array([0.1, 0.2], np.float32),
                                     u_sample=np.array([0.3], np.float32))
        for off in (1, 3):
            res = run_greedy(w, dev, offset=off)
            assert res["n_accepted"][0] == 2 and list(res["out_tokens"]) == [1000, 0, 2742]
            compare_stochastic(w, run_stochastic(w, dev, offset=off), [0])


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
@pytest.mark.parametrize("V", [13, 4101, 4104, 70003, 70008])
def test_rows_at_every_phase(dev, V, dtype):
    """Rows at every element phase of the 16-byte grid, through the greedy, stochastic and
    NKL calls (both buffers shifted alike: phased vector tiles when the row is a whole
    number of 16-byte blocks, else the staged path). Maxima sit in the partial blocks at
    the ends of the vocabulary chunks (the first and last elements of a row; ties at every
    multiple of 8, where chunks start, or at every 8j + 7, where they end, from a third of
    the row on) and tie with maxima inside the chunks, so the lowest index must come out
    of the element-by-element edge folds and the chunk merge."""
    rng = np.random.default_rng(V)
    R = 9
    t = rng.normal(0.0, 1.0, (R, V)).astype(np.float32)
    d = rng.normal(0.0, 1.0, (R - 1, V)).astype(np.float32)
    m0 = V // 3
    plant = [
        [0, V // 2],                                  # a tie: the first element wins
        [V - 1],                                      # the last element alone
        [V // 2, V - 1],                              # a tie with the last element: the middle wins
        [min(1, V - 1), min(2, V - 1)],               # a tie inside the head block
        [j for j in range(0, V, 8) if j >= m0],       # chunk starts
        [j for j in range(7, V, 8) if j >= m0],       # chunk ends
        [],                                           # a flat row: index 0
        [V // 2 + 1, V // 2],
        [V - 3, V - 2, V - 1],
    ]
    for i, idx in enumerate(plant):
        if i == 6:
            t[i] = 0.0
        t[i, idx] = 9.0
    t64 = O.widen(synth.storage(t, dtype), dtype)
    expect = [int(np.argmax(t64[i])) for i in range(R)]
    tokens = np.array(expect[:R - 1], np.int32)  # every draft the target's argmax: all must match
    w = synth.StochasticWorkload(B=1, V=V, dtype=dtype, T=1.0, gammas=np.array([R - 1], np.int32),
                                 cu_draft=np.array([0, R - 1], np.int32), target=synth.storage(t, dtype),
                                 draft=synth.storage(d, dtype), tokens=tokens,
                                 u_accept=np.full(R - 1, 0.5, np.float32), u_sample=np.array([0.5], np.float32))
    for off in range(8 if dtype == synth.BF16 else 4):
        res = run_greedy(w, dev, offset=off)
        assert res["device_status"][0] == 0
        assert int(res["n_accepted"][0]) == R - 1, off
        assert list(res["out_tokens"][:R]) == expect, off
        compare_greedy(w, res, [0])
        rs = run_stochastic(w, dev, offset=off)
        assert rs["device_status"][0] == 0
        assert list(rs["greedy_tokens"][:R]) == expect, off
        compare_stochastic(w, rs, [0])
        compare_nkl(w, run_nkl(w, dev, offset=off), [0])


@pytest.mark.parametrize("V,dtype,offset", [(3001, synth.BF16, 0), (128256, synth.BF16, 3), (5001, synth.F32, 1)])
def test_off_grid_tree(dev, V, dtype, offset):
    """The tree call on rows off the 16-byte grid (an odd vocabulary, a shifted buffer):
    the argmax of every node's row, its lowest index on ties, the deepest accepted path."""
    w = synth.make_tree(12, V, dtype, seed=V % 1000 + offset)
    res = run_tree(w, dev, offset=offset)
    assert res["device_status"][0] == 0
    compare_tree(w, res, range(w.B))
    assert np.any(res["accept_len"] > 1)


def test_off_grid_nkl_positions(dev):
    """The position-adaptive NKL mask on an odd vocabulary (staged pairs)."""
    w = synth.make_stochastic(12, 50257, synth.BF16, 0.8, seed=88, gamma_range=(1, 6), agreement=0.8)
    pos = np.random.default_rng(88).integers(1, 3000, w.B).astype(np.int32)
    compare_nkl(w, run_nkl(w, dev, positions=pos), range(w.B), positions=pos)
    res = run_stochastic(w, dev, options={"position": pos, "min_block_len": 2})
    compare_stochastic(w, res, range(w.B), positions=pos, min_block_len=2)


def test_off_grid_headline_shape(dev):
    """The headline batch (B=256, gamma=8, V=128256, bf16) with the logits one element off
    the 16-byte grid (phased tiles and sampler): every sequence against the oracle."""
    w = workload(synth.HEADLINE)
    res = run_stochastic(w, dev, offset=1)
    assert res["device_status"][0] == 0
    n_cmp, flagged, mismatched = compare_stochastic(w, res, range(w.B), ref=_oracle("stochastic", w))
    _report("headline stochastic, logits one element off the 16-byte grid", w, n_cmp, flagged, mismatched)
    g = run_greedy(w, dev, offset=1)
    compare_greedy(w, g, range(w.B), ref=_oracle("greedy", w))
    assert np.array_equal(g["n_accepted"], res["greedy_n"])
    aligned = run_stochastic(w, dev)
    # the two paths sum in different orders: decisions agree except at a boundary tie
    assert np.mean(aligned["n_accepted"] == res["n_accepted"]) > 0.99
    np.testing.assert_allclose(res["alpha"], aligned["alpha"], rtol=1e-4)


def test_off_grid_odd_vocabulary(dev):
    """A vocabulary whose bf16 rows are not a multiple of 16 bytes (V = 50257): every row
    has its own phase, target and draft rows of one position differ in phase."""
    w = synth.make_stochastic(64, 50257, synth.BF16, 0.8, seed=27, gamma=5, name="odd_vocab_B64_g5_V50257")
    res = run_stochastic(w, dev)
    assert res["device_status"][0] == 0
    n_cmp, flagged, mismatched = compare_stochastic(w, res, range(w.B), ref=_oracle("stochastic", w))
    _report("V=50257 stochastic (staged pairs)", w, n_cmp, flagged, mismatched)
    compare_greedy(w, run_greedy(w, dev), range(w.B), ref=_oracle("greedy", w))
    compare_nkl(w, run_nkl(w, dev), range(w.B), ref=_oracle("nkl", w))


def test_gamma_zero_and_one(dev):
    for g in (0, 1):
        w = handmade(5, g, 3000, synth.BF16, seed=20 + g)
        res = run_stochastic(w, dev)
        compare_stochastic(w, res, range(w.B))
        if g == 0:
            assert np.all(res["n_accepted"] == 0)


def test_max_gamma(dev):
    w = handmade(2, 128, 600, synth.F32, seed=21)
    res = run_stochastic(w, dev)
    compare_stochastic(w, res, range(w.B))


def test_identical_rows_accept_all(dev):
    """Invariant (a) on the GPU: q == p gives alpha == 1 and n == gamma; NKL == 0."""
    w = handmade(6, 4, 5000, synth.BF16, seed=22, draft_equals_target=True)
    w.u_accept[:] = np.float32(1.0) - np.float32(2.0 ** -24)
    res = run_stochastic(w, dev)
    assert np.all(res["n_accepted"] == 4)
    assert np.all(res["alpha"] == 1.0)
    assert np.all(np.abs(res["nkl"]) <= NKL_FLOOR)
    compare_stochastic(w, res, range(w.B))


def test_the_drafter_accepts_nothing(dev):
    w = handmade(16, 4, 32000, synth.BF16, seed=23, the_token=17)
    res = run_stochastic(w, dev)
    compare_stochastic(w, res, range(w.B))
    assert np.allclose(res["alpha"], res["p_x"], rtol=1e-3)
    assert res["n_accepted"].sum() == 0


def test_ties_and_flat_rows(dev):
    V = 64
    t = np.zeros((3, V), dtype=np.float32)
    t[0, [5, 9, 40]] = 3.0          # tie: lowest index 5
    t[2, [63, 62]] = 1.0            # tie at the end: 62
    d = np.zeros((2, V), dtype=np.float32)
    w = synth.StochasticWorkload(B=1, V=V, dtype=synth.F32, T=1.0, gammas=np.array([2], np.int32),
                                 cu_draft=np.array([0, 2], np.int32), target=t, draft=d,
                                 tokens=np.array([5, 0], np.int32), u_accept=np.array([0.1, 0.2], np.float32),
                                 u_sample=np.array([0.3], np.float32))
    res = run_greedy(w, dev)
    assert res["n_accepted"][0] == 2 and list(res["out_tokens"]) == [5, 0, 62]
    res = run_stochastic(w, dev)
    compare_stochastic(w, res, [0])


def test_nonfinite_and_token_range_are_reported(dev):
    w = handmade(4, 3, 2048, synth.F32, seed=24)
    w.target[1 * 4 + 2, 100] = np.inf          # sequence 1
    w.draft[2 * 3 + 0, 7] = np.nan             # sequence 2
    w.tokens[3 * 3 + 1] = 2048                 # sequence 3
    res = run_stochastic(w, dev)
    assert res["device_status"][0] == (_lib.SPEC_DEV_NONFINITE | _lib.SPEC_DEV_TOKEN_RANGE)
    assert list(res["n_accepted"][1:]) == [-1, -1, -1]
    assert np.all(res["out_tokens"][4:] == -1)
    assert np.all(np.isnan(res["alpha"][3:]))
    compare_stochastic(w, res, [0])            # the clean sequence is unaffected
    g = run_greedy(w, dev)
    assert g["device_status"][0] & _lib.SPEC_DEV_NONFINITE and g["n_accepted"][1] == -1
    w2 = handmade(2, 2, 512, synth.F32, seed=25)
    w2.target[2, 3] = -np.inf                  # the bonus row of sequence 0
    r2 = run_stochastic(w2, dev)
    assert r2["device_status"][0] == _lib.SPEC_DEV_NONFINITE and r2["n_accepted"][0] == -1
    nk = run_nkl(w2, dev)
    assert nk["device_status"][0] == 0         # the bonus row is not part of any NKL pair


def test_ragged_with_empty_sequences_and_bad_offsets(dev):
    w = synth.make_stochastic(9, 3000, synth.BF16, 0.8, seed=26, gamma_range=(0, 5), agreement=0.7)
    res = run_stochastic(w, dev)
    compare_stochastic(w, res, range(w.B))
    compare_greedy(w, run_greedy(w, dev), range(w.B))
    compare_nkl(w, run_nkl(w, dev), range(w.B))
    # non-monotone offsets are reported, with every access kept in bounds
    cu = torch.tensor([0, 5, 3, 8], dtype=torch.int32, device=dev)
    t = torch.zeros(11, 64, dtype=torch.bfloat16, device=dev)
    d = torch.zeros(8, 64, dtype=torch.bfloat16, device=dev)
    r = api.spec_verify_stochastic(t, d, torch.zeros(8, dtype=torch.int32, device=dev), 1.0,
                                   torch.zeros(8, device=dev), torch.zeros(3, device=dev), cu_draft=cu, gamma=5)
    torch.cuda.synchronize()
    assert int(r["device_status"][0]) & _lib.SPEC_DEV_OFFSETS


def test_tree_shapes(dev):
    rng = np.random.default_rng(30)
    for parent in ([-1], [-1, 0, 1, 2, 3], [-1, 0, 0, 1, 2, -1], list(range(-1, 63))):
        N = len(parent)
        B, V = 7, 300
        t32 = rng.normal(0, 1, (B * (N + 1), V)).astype(np.float32)
        t32[:, 7] = 5.0                           # makes many nodes match
        tok = np.where(rng.random((B, N)) < 0.85, 7, rng.integers(0, V, (B, N))).astype(np.int32)
        w = synth.TreeWorkload(B=B, N=N, V=V, dtype=synth.BF16, parent=np.array(parent, np.int32),
                               target=synth.storage(t32, synth.BF16), node_tokens=tok)
        compare_tree(w, run_tree(w, dev), range(B))


def test_output_distribution_is_the_target(dev):
    """Losslessness on the GPU: many sequences share one row pair and differ only in
    their uniforms; the emitted first token must follow p (chi-square)."""
    V, B, T = 6, 200000, 0.9
    rng = np.random.default_rng(31)
    zt = rng.normal(0, 1.5, (2, V)).astype(np.float32)
    zd = rng.normal(0, 1.5, (1, V)).astype(np.float32)
    q = np.exp(zd[0] / T) / np.exp(zd[0] / T).sum()
    x = rng.choice(V, size=B, p=q / q.sum()).astype(np.int32)    # drafts drawn from q
    w = synth.StochasticWorkload(B=B, V=V, dtype=synth.F32, T=T, gammas=np.ones(B, np.int32),
                                 cu_draft=np.arange(B + 1, dtype=np.int32), target=np.tile(zt, (B, 1)),
                                 draft=np.tile(zd, (B, 1)), tokens=x,
                                 u_accept=rng.random(B, dtype=np.float32), u_sample=rng.random(B, dtype=np.float32))
    res = run_stochastic(w, dev)
    first = res["out_tokens"].reshape(B, 2)[:, 0]
    p = np.exp(zt[0].astype(np.float64) / T)
    p /= p.sum()
    counts = np.bincount(first, minlength=V)
    stat, pval = scipy.stats.chisquare(counts, p * B)
    assert pval > 1e-4, (counts, p * B)


def test_large_vocab(dev):
    w = handmade(2, 2, 1 << 20, synth.BF16, T=0.7, seed=32)
    res = run_stochastic(w, dev)
    compare_stochastic(w, res, range(w.B))


@pytest.mark.parametrize("V,dtype", [(160000, synth.F32), (300000, synth.BF16), (1500000, synth.F32)])
def test_large_vocab_crossing(dev, V, dtype):
    """Large vocabularies. At 1.5M f32 tokens the slice-mass table (11728 entries) is
    longer than the 11264 entries the crossing search stages in shared memory, so the
    search reads it from global memory."""
    w = handmade(3, 2, V, dtype, T=1.0, seed=V % 997)
    res = run_stochastic(w, dev)
    compare_stochastic(w, res, range(w.B))


def _draw_in_band(w, b, n, y, T):
    """The drawn token has positive mass under the oracle's draw distribution of row n
    (residual, its p fallback, or the bonus p) and sits at the oracle's inverse-CDF
    crossing up to the flag band: C(y-1)/Z <= u + band and C(y)/Z >= u - band."""
    g = int(w.gammas[b])
    t0, d0 = w.target_base(b), w.draft_base(b)
    lp = O.log_softmax_T(O.widen(w.target[t0 + n], w.dtype), T)
    p = np.exp(lp)
    if n < g:
        q = np.exp(O.log_softmax_T(O.widen(w.draft[d0 + n], w.dtype), T))
        wt = O.residual(p, q)
        if float(np.sum(wt)) <= 1e-30:
            wt = p
    else:
        wt = p
    u = float(w.u_sample[b])
    C = np.cumsum(wt)
    Z = float(C[-1])
    before = float(C[y - 1]) if y > 0 else 0.0
    return wt[y] > 0 and before / Z <= u + O.FLAG_BAND and float(C[y]) / Z >= u - O.FLAG_BAND


@pytest.mark.parametrize("u", [0.0, 0.5, 0.99999994])
@pytest.mark.parametrize("V,dtype", [(50000, synth.BF16), (160000, synth.F32)])
def test_draw_at_cdf_ends(dev, u, V, dtype):
    """u = 0 takes the first token with mass, u just below 1 the last one. Exact where
    the oracle does not flag the draw, in band everywhere."""
    w = handmade(4, 2, V, dtype, T=0.9, seed=61)
    w.u_sample[:] = np.float32(u)
    res = run_stochastic(w, dev)
    compare_stochastic(w, res, range(w.B))
    for b in range(w.B):
        n = int(res["n_accepted"][b])
        y = int(res["out_tokens"][w.target_base(b) + n])
        assert _draw_in_band(w, b, n, y, w.T), (b, n, y)


def test_accept_at_u_equal_to_alpha(dev):
    """Reading R4 on the device: a draft is accepted when u <= alpha, so u set to the call's
    own alpha at a sequence's first rejected position turns it into an acceptance, and u one
    float above alpha keeps the rejection. A property of the device's comparison: both runs
    read the alpha the first call returned, no oracle value."""
    w = handmade(24, 6, 5000, synth.BF16, T=0.8, seed=62)
    first = run_stochastic(w, dev)
    n0 = first["n_accepted"].astype(int)
    alpha = first["alpha"]
    rejected = [b for b in range(w.B) if n0[b] < 6 and alpha[6 * b + n0[b]] < 1.0]
    assert len(rejected) >= 5
    at = w.u_accept.copy()
    above = w.u_accept.copy()
    for b in rejected:
        a = np.float32(alpha[6 * b + n0[b]])
        at[6 * b + n0[b]] = a
        above[6 * b + n0[b]] = np.nextafter(a, np.float32(np.inf), dtype=np.float32)
    w.u_accept[:] = at
    eq = run_stochastic(w, dev)
    w.u_accept[:] = above
    gt = run_stochastic(w, dev)
    for b in rejected:
        i = 6 * b + n0[b]
        assert eq["alpha"][i] == alpha[i] and gt["alpha"][i] == alpha[i], b
        assert int(eq["n_accepted"][b]) > n0[b], (b, n0[b], int(eq["n_accepted"][b]))
        assert int(gt["n_accepted"][b]) == n0[b], (b, n0[b], int(gt["n_accepted"][b]))


def test_back_to_back_calls_on_shared_buffers(dev):
    """Calls queued on one stream with no synchronisation between them, all on one
    workspace, each preceded by torch kernels that overwrite the input buffers the previous
    call read: every call sees its own inputs, and tickets and records are re-armed between
    calls of any mode (kernels of adjacent calls may be resident at the same time)."""
    ws = [handmade(6, 4, 20000, synth.BF16, T=0.9, seed=70 + k) for k in range(6)]
    src = [dict(t=to_dev(w.target, dev), d=to_dev(w.draft, dev), tok=to_dev(w.tokens, dev),
                ua=to_dev(w.u_accept, dev), us=to_dev(w.u_sample, dev)) for w in ws]
    buf = {k: torch.empty_like(v) for k, v in src[0].items()}
    work = torch.empty(64 << 20, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    modes = ["stochastic", "stochastic", "greedy", "nkl", "stochastic", "stochastic"]
    outs = []
    for k, mode in enumerate(modes):
        for name, v in src[k].items():
            buf[name].copy_(v)
        if mode == "stochastic":
            outs.append(api.spec_verify_stochastic(buf["t"], buf["d"], buf["tok"], ws[k].T, buf["ua"], buf["us"],
                                                   gamma=4, workspace=work))
        elif mode == "greedy":
            outs.append(api.spec_verify_greedy(buf["t"], buf["tok"], gamma=4, workspace=work))
        else:
            outs.append(api.spec_nkl(buf["t"], buf["d"], ws[k].T, gamma=4, workspace=work))
    torch.cuda.synchronize()
    for k, mode in enumerate(modes):
        res = {name: v.cpu().numpy() for name, v in outs[k].items()}
        assert res["device_status"][0] == 0, (k, mode)
        if mode == "stochastic":
            compare_stochastic(ws[k], res, range(ws[k].B))
        elif mode == "greedy":
            compare_greedy(ws[k], res, range(ws[k].B))
        else:
            compare_nkl(ws[k], res, range(ws[k].B))


def test_repeat_calls_reuse_workspace(dev):
    """Tickets are re-armed by every call: two calls on one workspace give the same result,
    also after a call with a different geometry."""
    w = handmade(8, 3, 5000, synth.BF16, seed=33)
    a = run_stochastic(w, dev)
    run_stochastic(handmade(3, 5, 700, synth.F32, seed=34), dev)
    b = run_stochastic(w, dev)
    for k in ("n_accepted", "out_tokens", "alpha", "nkl", "greedy_tokens"):
        assert np.array_equal(a[k], b[k]), k
