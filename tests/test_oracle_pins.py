"""Pins for the fp64 oracle: closed forms, invariants, brute force and the values the
pages print. No GPU. Each check is chosen so that a plausible slip in the oracle (a
swapped p/q, T multiplied instead of divided, a wrong row index, '<' for '<=', a
non-strict CDF comparison, log2 for ln) makes at least one of them fail."""
import json
import math
import os

import numpy as np
import pytest
import scipy.special as sps
import scipy.stats

from oracle import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- widening

def test_widen_bf16_is_exact_ieee():
    bits = np.array([0x3F80, 0xC040, 0x7F7F, 0x0001, 0x8000, 0x4049], dtype=np.uint16)
    want = [1.0, -3.0, 3.3895313892515355e38, 2.0 ** -133, -0.0, 3.140625]
    got = O.widen(bits, "bf16")
    assert list(got) == want
    assert math.copysign(1.0, got[4]) == -1.0


# ---------------------------------------------------------------- softmax at temperature T

def test_two_point_softmax_is_sigmoid_of_scaled_gap():
    a, T = 1.7, 0.6
    lp = O.log_softmax_T(np.array([0.0, a]), T)
    assert abs(math.exp(lp[1]) - 1.0 / (1.0 + math.exp(-a / T))) < 1e-15


def test_uniform_row_and_shift_invariance():
    V = 1000
    lp = O.log_softmax_T(np.full(V, 2.5), 0.7)
    assert np.allclose(lp, -math.log(V), atol=1e-14, rtol=0)
    rng = np.random.default_rng(5)
    z = rng.normal(0, 3, 4096)
    assert np.allclose(O.log_softmax_T(z, 0.8), O.log_softmax_T(z + 11.0, 0.8), atol=1e-12, rtol=0)


def test_softmax_matches_scipy_and_sums_to_one():
    rng = np.random.default_rng(6)
    z = rng.normal(0, 3, (3, 128256))
    for T in (0.6, 1.0, 1.7):
        p = O.softmax_T(z, T)
        assert np.allclose(p.sum(axis=1), 1.0, atol=1e-12, rtol=0)
        assert np.allclose(p, sps.softmax(z / T, axis=1), rtol=1e-12, atol=1e-300)


# ---------------------------------------------------------------- acceptance

def test_acceptance_prob_closed_form():
    assert O.acceptance_prob(math.log(0.25), math.log(0.5)) == pytest.approx(0.5, abs=1e-15)
    assert O.acceptance_prob(math.log(0.5), math.log(0.25)) == 1.0


def test_first_rejection_uses_less_or_equal():
    assert O.first_rejection(np.array([0.5, 0.5, 0.5]), np.array([0.5, 0.5, 0.5])) == 3
    assert O.first_rejection(np.array([0.1, 0.2, 0.9]), np.array([0.5, 0.5, 0.5])) == 2
    assert O.first_rejection(np.array([0.6]), np.array([0.5])) == 0
    assert O.first_rejection(np.array([]), np.array([])) == 0


def _rows(rng, g, V, scale=3.0):
    return rng.normal(0, scale, (g + 1, V))


def test_identical_rows_accept_everything():
    """Invariant (a): q == p gives alpha == 1 at every position and n == gamma for any u < 1."""
    rng = np.random.default_rng(7)
    for V, g in ((2, 1), (8, 3), (1000, 5), (32000, 4)):
        t = _rows(rng, g, V)
        d = t[:g].copy()
        tok = rng.integers(0, V, g)
        u = np.full(g, np.float32(1.0) - np.float32(2.0 ** -24), dtype=np.float64)
        r = O.verify_stochastic_sequence(t, d, tok, 0.9, u, 0.3)
        assert np.all(r["alpha"] == 1.0)
        assert r["n"] == g
        assert np.all(r["nkl"] == 0.0) or np.all(np.abs(r["nkl"]) < 1e-15)
        assert list(r["tokens"][:g]) == list(tok)


def test_the_drafter_gets_no_acceptance():
    """The 'Chain of Draft' article's degenerate drafter (always the same token):
    q(x) ~ 1 so alpha = p(x), tiny at V = 32000; with seeded u every sequence stops at 0."""
    want = gold("cod_the_drafter.json")["acceptance_rate"]
    rng = np.random.default_rng(8)
    V, g, the = 32000, 4, 17
    accepted = 0
    for _ in range(64):
        t = _rows(rng, g, V)
        d = rng.normal(0, 3, (g, V))
        d[:, the] = 60.0
        u = rng.random(g).astype(np.float32).astype(np.float64)
        r = O.verify_stochastic_sequence(t, d, np.full(g, the), 1.0, u, float(rng.random()))
        assert np.allclose(r["alpha"], r["p_x"], rtol=1e-9)
        accepted += r["n"]
    assert accepted / (64 * g) == want


# ---------------------------------------------------------------- inverse CDF

def test_inverse_cdf_hand_cases():
    w = np.array([0.0, 1.0, 0.0, 3.0])
    assert O.inverse_cdf(w, 0.0)[0] == 1          # a zero-mass token is never drawn
    assert O.inverse_cdf(w, 0.2499)[0] == 1
    assert O.inverse_cdf(w, 0.25)[0] == 3         # strict '>': C(1) = 1 is not > 1
    assert O.inverse_cdf(w, 0.99999)[0] == 3
    y, Z, c0, c1 = O.inverse_cdf(w, 0.5)
    assert (y, Z, c0, c1) == (3, 4.0, 1.0, 4.0)


def test_bonus_two_token_closed_form():
    """V = 2, everything accepted: the bonus token is 1 iff u_sample >= p_gamma(0)."""
    zt = np.array([[0.3, -0.4], [1.1, 0.2]])
    p0 = sps.softmax(zt[1] / 0.8)[0]
    for us, want in ((p0 - 1e-9, 0), (p0 + 1e-9, 1), (0.0, 0), (0.999, 1)):
        r = O.verify_stochastic_sequence(zt, zt[:1].copy(), np.array([1]), 0.8, np.array([0.0]), us)
        assert r["n"] == 1 and r["tokens"][1] == want


# ---------------------------------------------------------------- losslessness by enumeration

def _measure(fn, lo=0.0, hi=1.0, iters=60):
    """Length of the set of u in [lo, hi) where fn(u) is True, for fn monotone (True then False)."""
    if not fn(lo):
        return 0.0
    if fn(np.nextafter(hi, 0)):
        return hi - lo
    a, b = lo, hi
    for _ in range(iters):
        m = 0.5 * (a + b)
        if fn(m):
            a = m
        else:
            b = m
    return a - lo


def _sampler_masses(call, V):
    """Masses of u_sample mapping to each token: the map is monotone non-decreasing in u,
    so the breakpoints are found by bisection."""
    masses = np.zeros(V)
    for v in range(V):
        masses[v] = _measure(lambda u: call(u) <= v) - (_measure(lambda u: call(u) <= v - 1) if v else 0.0)
    return masses


@pytest.mark.parametrize("V,T", [(2, 1.0), (3, 0.5), (5, 1.3), (8, 0.7), (8, 2.0)])
def test_output_marginal_equals_target_distribution(V, T):
    """Invariant (b): draw x ~ q, accept with the oracle's own rule, else draw from the
    oracle's residual sampler; the emitted token's law must be p within 1e-12."""
    rng = np.random.default_rng(100 + V)
    zt = rng.normal(0, 2, (2, V))
    zd = rng.normal(0, 2, (1, V))
    p = sps.softmax(zt[0] / T)
    q = sps.softmax(zd[0] / T)

    def n_for(x, u):
        return O.verify_stochastic_sequence(zt, zd, np.array([x]), T, np.array([u]), 0.5)["n"]

    acc = np.array([_measure(lambda u, x=x: n_for(x, u) >= 1) for x in range(V)])
    # the correction does not depend on which x was rejected; take the draft token
    # with the lowest acceptance so that a rejection is reachable
    xr = int(np.argmin(acc))
    assert acc[xr] < 1.0
    res = _sampler_masses(lambda us: O.verify_stochastic_sequence(
        zt, zd, np.array([xr]), T, np.array([np.nextafter(1.0, 0)]), us)["tokens"][0], V)
    emitted = q * acc + np.sum(q * (1.0 - acc)) * res
    assert np.allclose(emitted, p, atol=1e-12, rtol=0)
    assert np.allclose(acc, np.minimum(1.0, p / q), atol=1e-12, rtol=0)


def test_second_position_and_bonus_use_their_own_rows():
    """gamma = 2: given the first draft accepted, the second emitted token follows p_1,
    and when both are accepted the third follows p_2 (the bonus row)."""
    V, T = 6, 0.9
    rng = np.random.default_rng(11)
    zt = rng.normal(0, 2, (3, V))
    zd = rng.normal(0, 2, (2, V))
    p1 = sps.softmax(zt[1] / T)
    p2 = sps.softmax(zt[2] / T)
    q1 = sps.softmax(zd[1] / T)
    x0 = 0

    def run(x1, u1, us):
        return O.verify_stochastic_sequence(zt, zd, np.array([x0, x1]), T, np.array([0.0, u1]), us)

    acc1 = np.array([_measure(lambda u, x=x: run(x, u, 0.5)["n"] == 2) for x in range(V)])
    xr = int(np.argmin(acc1))
    res = _sampler_masses(lambda us: run(xr, np.nextafter(1.0, 0), us)["tokens"][1], V)
    second = q1 * acc1 + np.sum(q1 * (1 - acc1)) * res
    assert np.allclose(second, p1, atol=1e-12, rtol=0)
    xa = int(np.argmax(acc1))
    bonus = _sampler_masses(lambda us: run(xa, 0.0, us)["tokens"][2], V)
    assert np.allclose(bonus, p2, atol=1e-12, rtol=0)


def test_worked_example_three_accepted_one_corrected():
    ex = gold("sps_worked_example.json")
    g = ex["drafted"]
    rng = np.random.default_rng(12)
    V = 50
    t = rng.normal(0, 2, (g + 1, V))
    d = t[:g].copy()
    d[3] = rng.normal(0, 2, V)                 # the 4th draft row disagrees with the target
    q3 = sps.softmax(d[3])
    p3 = sps.softmax(t[3])
    x3 = int(np.argmax(q3 / p3))               # a token the target under-weights: alpha < 1
    tok = np.array([5, 9, 7, x3])
    u = np.array([0.3, 0.7, 0.99, 0.999999])
    r = O.verify_stochastic_sequence(t, d, tok, 1.0, u, 0.42)
    assert r["alpha"][3] < 0.999999
    assert r["n"] == ex["accepted"]
    valid = int(np.sum(r["tokens"] >= 0))
    assert valid == ex["emitted"] == ex["accepted"] + ex["corrected"]
    assert list(r["tokens"][:3]) == [5, 9, 7]
    w = np.maximum(0, p3 - q3)
    assert w[r["tokens"][3]] > 0                # the correction comes from the residual's support


# ---------------------------------------------------------------- greedy

def test_greedy_accepts_target_argmax_drafts():
    """Invariant (c)."""
    rng = np.random.default_rng(13)
    t = rng.normal(0, 3, (6, 777))
    am = [int(np.argmax(r)) for r in t]
    r = O.verify_greedy_sequence(t, np.array(am[:5]))
    assert r["n"] == 5 and list(r["tokens"]) == am


def test_greedy_first_mismatch_and_ties():
    t = np.array([[3.0, 5.0, 5.0, 1.0], [0.0, 0.0, 0.0, 0.0], [1.0, 2.0, 9.0, 9.0]])
    r = O.verify_greedy_sequence(t, np.array([1, 0]))
    assert r["n"] == 2 and list(r["tokens"]) == [1, 0, 2]
    r = O.verify_greedy_sequence(t, np.array([2, 0]))
    assert r["n"] == 0 and list(r["tokens"]) == [1, -1, -1]
    r = O.verify_greedy_sequence(t, np.array([1, 3]))
    assert r["n"] == 1 and list(r["tokens"]) == [1, 0, -1]


# ---------------------------------------------------------------- tree

def _tree_brute(t_rows, tok, parent):
    """Walk every root-to-leaf chain, keep the longest prefix whose tokens each equal the
    argmax of the row before them; best = deepest end node, lowest index on ties."""
    N = len(parent)
    children = {j: [k for k in range(N) if parent[k] == j] for j in range(-1, N)}
    chains = []

    def walk(j, acc):
        acc = acc + [j]
        if not children[j]:
            chains.append(acc)
        for c in children[j]:
            walk(c, acc)

    for r in children[-1]:
        walk(r, [])
    ends = []
    for ch in chains:
        row = 0
        good = []
        for j in ch:
            if int(tok[j]) == int(np.argmax(t_rows[row])):
                good.append(j)
                row = j + 1
            else:
                break
        if good:
            ends.append((len(good), good[-1], good))
    if not ends:
        return 0, [], int(np.argmax(t_rows[0]))
    best = min(ends, key=lambda e: (-e[0], e[1]))
    return best[0], best[2], int(np.argmax(t_rows[best[1] + 1]))


@pytest.mark.parametrize("seed", range(12))
def test_tree_matches_brute_force(seed):
    parent = [-1, -1, -1, 0, 1, 2, 3, 4, 5, 6, 7, 8]
    assert len(parent) == gold("pd_tree_shape.json")["max_nodes"]
    assert sum(1 for p in parent if p < 0) == gold("pd_tree_shape.json")["root_candidates"]
    rng = np.random.default_rng(seed)
    V = 9
    t = rng.normal(0, 1, (13, V))
    am = np.argmax(t, axis=1)
    tok = rng.integers(0, V, 12)
    for j in range(12):                          # force matches at random
        if rng.random() < 0.6:
            tok[j] = am[0 if parent[j] < 0 else parent[j] + 1]
    r = O.verify_tree_sequence(t, tok, parent)
    L, path, corr = _tree_brute(t, tok, parent)
    assert r["len"] == L
    assert list(r["path"][:L]) == path and np.all(r["path"][L:] == -1)
    assert list(r["tokens"][:L]) == [int(tok[j]) for j in path]
    assert r["tokens"][L] == corr and np.all(r["tokens"][L + 1:] == -1)


def test_tree_branching_shapes_and_ties():
    parent = [-1, 0, 0, 1, 2, -1]               # two branches of equal depth under root 0
    t = np.zeros((7, 4))
    t[0, 2] = 1; t[1, 1] = 1; t[2, 3] = 1; t[3, 0] = 1
    tok = np.array([2, 1, 1, 3, 0, 0])          # nodes 3 and 4 both accepted at depth 3: lowest wins
    r = O.verify_tree_sequence(t, tok, parent)
    L, path, corr = _tree_brute(t, tok, parent)
    assert (r["len"], list(r["path"][:L])) == (L, path) == (3, [0, 1, 3])
    tok2 = np.array([2, 1, 1, 0, 1, 0])         # only depth-2 nodes 1 and 2 accepted: lowest wins
    r = O.verify_tree_sequence(t, tok2, parent)
    assert r["len"] == 2 and list(r["path"][:2]) == [0, 1] and r["tokens"][2] == int(np.argmax(t[2]))


def test_chain_tree_reduces_to_greedy():
    rng = np.random.default_rng(21)
    for _ in range(20):
        V, N = 11, 6
        t = rng.normal(0, 1, (N + 1, V))
        am = np.argmax(t, axis=1)
        tok = np.where(rng.random(N) < 0.7, am[:N], rng.integers(0, V, N))
        tr = O.verify_tree_sequence(t, tok, [-1, 0, 1, 2, 3, 4])
        gr = O.verify_greedy_sequence(t, tok)
        assert tr["len"] == gr["n"]
        assert list(tr["tokens"]) == list(gr["tokens"])


# ---------------------------------------------------------------- NKL

def test_nkl_zero_on_identical_rows_and_nonnegative():
    """Invariant (d)."""
    rng = np.random.default_rng(31)
    z = rng.normal(0, 3, 5000)
    assert abs(O.nkl_pair(z, z.copy(), 0.6)[0]) < 1e-15
    for _ in range(20):
        a, b = rng.normal(0, 3, 300), rng.normal(0, 3, 300)
        assert O.nkl_pair(a, b, 0.6)[0] >= 0.0


def test_nkl_one_token_vocabulary_is_zero():
    assert O.nkl_pair(np.array([3.0]), np.array([-7.0]), 0.5) == (0.0, 0.0)


def test_nkl_two_point_and_direction():
    """KL(q || p) with q the DRAFT row, natural log, divided by ln V: against scipy's
    relative entropy, which is not symmetric, so a swapped direction fails."""
    zt = np.array([0.0, 1.2])
    zd = np.array([0.0, -0.9])
    T = 0.7
    p = sps.softmax(zt / T)
    q = sps.softmax(zd / T)
    want = scipy.stats.entropy(q, p) / math.log(2)
    assert O.nkl_pair(zt, zd, T)[0] == pytest.approx(want, rel=1e-12)
    assert abs(scipy.stats.entropy(p, q) / math.log(2) - want) > 1e-3


def test_nkl_scale_is_log_vocab():
    """Against a uniform target a one-hot draft has KL = ln V, so NKL -> 1; at the page's
    128k vocabulary ln V ~ 11.76, the 'about 12' the page quotes."""
    c = gold("cod_nkl_constants.json")
    V = c["vocab_size"]
    assert abs(math.log(V) - c["page_kl_scale_about"]) < 0.5
    assert math.log(V) == pytest.approx(11.7618, abs=1e-4)
    zt = np.zeros(V)
    zd = np.zeros(V)
    zd[123] = 2000.0
    nkl, nkl_eps = O.nkl_pair(zt, zd, 1.0)
    assert nkl == pytest.approx(1.0, abs=1e-12)
    assert abs(nkl_eps - nkl) < 1e-6


def test_nkl_mask_threshold_and_eps_form():
    c = gold("cod_nkl_constants.json")
    rng = np.random.default_rng(33)
    V, g = 4000, 3
    t = rng.normal(0, 3, (g + 1, V))
    d = 0.9 * t[:g] + rng.normal(0, 1, (g, V))
    r = O.verify_stochastic_sequence(t, d, np.zeros(g, dtype=int), 0.6, np.zeros(g), 0.5, c["delta"])
    assert np.all(r["mask"] == (r["nkl"] < c["delta"]))
    assert np.all(np.abs(r["nkl_eps"] - r["nkl"]) <= 1e-4 * r["nkl"])


# ---------------------------------------------------------------- position-adaptive delta

def test_position_delta_printed_values():
    c = gold("cod_position_delta.json")
    for pos, val in c["printed"].items():
        got = O.position_delta(int(pos), c["delta_base"], c["alpha"], c["delta_max"])
        if pos in c["page_inconsistent"]:
            assert abs(got - val) > 0.03          # the page's 0.192 fits neither log form
        else:
            assert got == pytest.approx(val, abs=1e-12)
    assert O.position_delta(10 ** 9) == c["delta_max"]


# ---------------------------------------------------------------- error semantics

def test_errors_mark_the_whole_sequence():
    rng = np.random.default_rng(41)
    t = rng.normal(0, 1, (4, 10))
    d = rng.normal(0, 1, (3, 10))
    bad = t.copy()
    bad[3, 4] = np.inf
    r = O.verify_stochastic_sequence(bad, d, np.array([1, 2, 3]), 1.0, np.zeros(3), 0.5)
    assert r["n"] == -1 and r["err"] == O.ERR_NONFINITE and np.all(r["tokens"] == -1)
    assert np.all(np.isnan(r["alpha"]))
    r = O.verify_stochastic_sequence(t, d, np.array([1, 10, 3]), 1.0, np.zeros(3), 0.5)
    assert r["n"] == -1 and r["err"] == O.ERR_TOKEN_RANGE
    r = O.verify_greedy_sequence(t, np.array([-1, 2, 3]))
    assert r["n"] == -1 and r["err"] == O.ERR_TOKEN_RANGE


# ---------------------------------------------------------------- separate temperatures (R19)

@pytest.mark.parametrize("V,Tt,Td", [(3, 0.8, 0.4), (6, 0.7, 0.3), (8, 0.9, 0.5), (5, 1.0, 2.0)])
def test_separate_temperatures_emit_the_target_distribution(V, Tt, Td):
    """Drafts drawn from q at T_d, verified against p at T_t: the emitted token's law is
    softmax(z_t / T_t) within 1e-12, and the acceptance is min(1, p/q) with q at T_d."""
    rng = np.random.default_rng(200 + V)
    zt = rng.normal(0, 2, (2, V))
    zd = rng.normal(0, 2, (1, V))
    p = sps.softmax(zt[0] / Tt)
    q = sps.softmax(zd[0] / Td)

    def run(x, u, us):
        return O.verify_stochastic_sequence(zt, zd, np.array([x]), Tt, np.array([u]), us, T_draft=Td)

    acc = np.array([_measure(lambda u, x=x: run(x, u, 0.5)["n"] >= 1) for x in range(V)])
    assert np.allclose(acc, np.minimum(1.0, p / q), atol=1e-12, rtol=0)
    xr = int(np.argmin(acc))
    assert acc[xr] < 1.0
    res = _sampler_masses(lambda us: run(xr, np.nextafter(1.0, 0), us)["tokens"][0], V)
    emitted = q * acc + np.sum(q * (1.0 - acc)) * res
    assert np.allclose(emitted, p, atol=1e-12, rtol=0)


def test_separate_temperatures_nkl_at_the_target_temperature():
    """p(x) and q(x) use their own temperatures; NKL scales both rows by T_t ([CoD] 3.2)."""
    rng = np.random.default_rng(17)
    V, g, Tt, Td = 50, 3, 0.8, 0.4
    t = rng.normal(0, 2, (g + 1, V))
    d = rng.normal(0, 2, (g, V))
    x = np.array([3, 7, 11])
    r = O.verify_stochastic_sequence(t, d, x, Tt, np.full(g, 0.5), 0.5, T_draft=Td)
    for i in range(g):
        assert r["p_x"][i] == pytest.approx(sps.softmax(t[i] / Tt)[x[i]], rel=1e-12)
        assert r["q_x"][i] == pytest.approx(sps.softmax(d[i] / Td)[x[i]], rel=1e-12)
        want = scipy.stats.entropy(sps.softmax(d[i] / Tt), sps.softmax(t[i] / Tt)) / math.log(V)
        assert r["nkl"][i] == pytest.approx(want, rel=1e-9)
    same = O.verify_stochastic_sequence(t, d, x, Tt, np.full(g, 0.5), 0.5)
    assert np.allclose(same["nkl"], r["nkl"], rtol=0, atol=0)


# ---------------------------------------------------------------- position-adaptive mask (R18)

def _two_point_rows(nkl):
    """A (target, draft) row pair over V = 2 with KL(q || p) / ln 2 = nkl: q uniform,
    p = (a, 1 - a) with a(1 - a) = exp(-2 (nkl ln 2 + ln 2))."""
    prod = math.exp(-2.0 * (nkl * math.log(2) + math.log(2)))
    a = (1.0 - math.sqrt(1.0 - 4.0 * prod)) / 2.0
    return np.array([math.log(a), math.log(1.0 - a)]), np.array([0.0, 0.0])


def test_position_mask_follows_the_printed_thresholds():
    """NKL 0.156 lies between delta(1) = 0.15 and delta(2) = 0.162: the first draft (at
    position 1) is masked out and the second (position 2) in. NKL 0.2 is out at position 1
    and in at position 1024 (delta 0.27, the page's printed value)."""
    zt, zd = _two_point_rows(0.156)
    t = np.stack([zt, zt, zt])
    d = np.stack([zd, zd])
    r = O.verify_stochastic_sequence(t, d, np.array([0, 0]), 1.0, np.zeros(2), 0.5, 0.15, position=1)
    assert r["nkl"] == pytest.approx([0.156, 0.156], abs=1e-12)
    assert list(r["mask"]) == [0, 1]
    assert list(O.verify_stochastic_sequence(t, d, np.array([0, 0]), 1.0, np.zeros(2), 0.5, 0.15)["mask"]) == [0, 0]
    zt, zd = _two_point_rows(0.2)
    t = np.stack([zt, zt])
    d = zd[None]
    lo = O.verify_stochastic_sequence(t, d, np.array([0]), 1.0, np.zeros(1), 0.5, 0.15, position=1)
    hi = O.verify_stochastic_sequence(t, d, np.array([0]), 1.0, np.zeros(1), 0.5, 0.15, position=1024)
    assert lo["mask"][0] == 0 and hi["mask"][0] == 1
    rows = O.nkl_rows(np.stack([zt, zt]), zd[None], np.array([0, 1]), 1.0, "f32", 0.15, positions=np.array([1024]))
    assert rows[0]["mask"][0] == 1
    bad = O.verify_stochastic_sequence(t, d, np.array([0]), 1.0, np.zeros(1), 0.5, 0.15, position=0)
    assert bad["mask"][0] == 0 and bad["nkl"][0] == pytest.approx(0.2, abs=1e-12)


# ---------------------------------------------------------------- block-accept (R20)

def _block_accept_page_loops(d, t, min_len):
    """The page's search written out: every (start, end) window of length >= min_len whose
    draft and target slices are equal; a strictly longer one replaces the best."""
    g = len(d)
    max_len, best_start = 0, 0
    for start in range(g):
        for end in range(start + min_len, g + 1):
            if list(d[start:end]) == list(t[start:end]) and end - start > max_len:
                max_len, best_start = end - start, start
    if max_len >= min_len and max_len > 0:
        e = best_start + max_len
        return e, list(d[:e]) + list(t[e:])
    return 0, list(t)


@pytest.mark.parametrize("seed", range(40))
def test_block_accept_matches_the_page_search(seed):
    rng = np.random.default_rng(300 + seed)
    g = int(rng.integers(0, 13))
    t = rng.integers(0, 3, g)
    d = np.where(rng.random(g) < 0.7, t, rng.integers(0, 3, g))
    for min_len in (1, 2, 3, 4):
        e, toks = O.block_accept(d, t, min_len)
        we, wt = _block_accept_page_loops(d, t, min_len)
        assert e == we and list(toks) == wt, (list(d), list(t), min_len)


def test_block_accept_hand_cases():
    assert O.block_accept([1, 2, 3, 4, 5], [1, 9, 3, 4, 5], 3)[0] == 5       # the run 3,4,5 ends the block
    e, toks = O.block_accept([7, 2, 3, 4, 8, 8], [1, 2, 3, 4, 5, 6], 3)
    assert e == 4 and list(toks) == [7, 2, 3, 4, 5, 6]                       # the draft before the run is kept
    e, toks = O.block_accept([1, 2, 9, 4, 5], [1, 2, 3, 4, 5], 3)
    assert e == 0 and list(toks) == [1, 2, 3, 4, 5]                          # two runs of 2: fallback
    assert O.block_accept([5, 5, 0, 5, 5, 5, 0, 5, 5, 5], [5] * 10, 3)[0] == 6  # ties: the earlier run
    t = np.array([[0.0, 1.0, 0.0], [2.0, 0.0, 0.0], [0.0, 0.0, 3.0], [1.0, 0.0, 0.0]])
    r = O.verify_greedy_sequence(t, np.array([1, 0, 2]), min_block_len=3)
    assert r["block_n"] == 3 and list(r["block_tokens"]) == [1, 0, 2]


# ---------------------------------------------------------------- acceptance statistics (R21)

def test_acceptance_summary_against_numpy():
    rng = np.random.default_rng(44)
    recs = [(int(rng.integers(0, 10)), int(rng.integers(-1, 9)), int(rng.integers(0, 9))) for _ in range(500)]
    recs = [(bk, min(n, g), g) for bk, n, g in recs]
    s = O.acceptance_summary(recs, 9, 4)
    keep = [(n, g) for bk, n, g in recs if 5 < bk <= 9 and g > 0 and n >= 0]
    rates = np.array([n / g for n, g in keep])
    assert s["rounds"] == len(keep) and s["accepted"] == sum(n for n, _ in keep)
    assert s["mean_accepted"] == pytest.approx(np.mean([n for n, _ in keep]), rel=1e-12)
    assert s["arsd"] == pytest.approx(np.std(rates), rel=1e-9)
    h = O.acceptance_summary([(0, 2, 4), (0, 4, 4), (1, 3, 4)], 0, 1)
    assert h["rounds"] == 2 and h["mean_accepted"] == 3.0 and h["arsd"] == pytest.approx(0.25, abs=1e-15)


# ---------------------------------------------------------------- multi-draft (R22)

def test_pairwise_nkl_against_scipy():
    rng = np.random.default_rng(51)
    K, V, T = 4, 300, 0.7
    d = rng.normal(0, 2, (K, V))
    M = O.pairwise_nkl(d, T)
    for a in range(K):
        assert M[a, a] == 0.0
        for b in range(K):
            if a != b:
                want = scipy.stats.entropy(sps.softmax(d[a] / T), sps.softmax(d[b] / T)) / math.log(V)
                assert M[a, b] == pytest.approx(want, rel=1e-9)
    assert not np.allclose(M, M.T)                        # KL is not symmetric: both directions kept
    same = O.pairwise_nkl(np.stack([d[0]] * 3), T)
    assert np.all(np.abs(same) < 1e-12)
    assert O.consensus_divergence(same) == (True, False)


def test_consensus_and_divergence_flags():
    M = np.full((3, 3), 0.5)
    np.fill_diagonal(M, 0.0)
    assert O.consensus_divergence(M) == (False, True)
    M[0, 2] = 0.05
    assert O.consensus_divergence(M) == (False, False)    # one direction alone is not consensus
    M[2, 0] = 0.09
    assert O.consensus_divergence(M) == (True, False)
    M = np.full((2, 2), 0.15)
    np.fill_diagonal(M, 0.0)
    assert O.consensus_divergence(M) == (False, False)    # 0.15 is not above 0.15
    M[0, 1] = M[1, 0] = 0.1
    assert O.consensus_divergence(M)[0] is False          # 0.1 is not below 0.1


def test_multi_draft_keeps_the_longest_accepted_candidate():
    """Greedy groups of K = 3 candidates with known argmax rows: accepted counts 0, 2, 2
    -> candidate 1 (the lower index of the tie) and its tokens."""
    V, g, K = 5, 3, 3
    rows_t, rows_d, toks = [], [], []
    am = [1, 2, 3, 4]
    for k, n in enumerate([0, 2, 2]):
        t = np.zeros((g + 1, V))
        for i in range(g + 1):
            t[i, am[i]] = 5.0
        rows_t.append(t)
        rows_d.append(np.zeros((g, V)) + k)
        toks.append([am[i] if i < n else (am[i] + 1) % V for i in range(g)])
    target = np.concatenate(rows_t).astype(np.float32)
    draft = np.concatenate(rows_d).astype(np.float32)
    tokens = np.array(toks, dtype=np.int64).reshape(-1)
    r = O.verify_multi(target, draft, tokens, 1, K, g, 1.0, "f32", stochastic=False)[0]
    assert [c["n"] for c in r["cand"]] == [0, 2, 2]
    assert r["best_k"] == 1 and r["best_n"] == 2
    assert list(r["best_tokens"]) == [1, 2, 3, -1]       # the target argmax replaces the mismatch
    assert np.all(np.abs(r["pair_nkl"]) < 1e-12) and np.all(r["consensus"] == 1)   # constant rows: identical q


# ---------------------------------------------------------------- vocabulary shards (R23)

@pytest.mark.parametrize("seed", range(6))
def test_shard_merge_equals_the_whole_row(seed):
    rng = np.random.default_rng(600 + seed)
    V, T = int(rng.integers(2, 3000)), float(rng.uniform(0.3, 1.5))
    zt = np.round(rng.normal(0, 3, V), 1)              # rounded: ties of the maximum across shards occur
    zd = 0.9 * zt + rng.normal(0, 1, V)
    cuts = sorted(set(int(c) for c in rng.integers(1, V, int(rng.integers(0, 5))))) if V > 1 else []
    bounds = [0] + cuts + [V]
    parts = [O.shard_stats(zt[a:b], zd[a:b], T, a) for a, b in zip(bounds, bounds[1:])]
    left = parts[0]
    for p in parts[1:]:
        left = O.merge_stats(left, p)
    right = parts[-1]
    for p in reversed(parts[:-1]):
        right = O.merge_stats(p, right)
    for st in (left, right):
        out = O.stats_outputs(st, V)
        assert out["argmax"] == int(np.argmax(zt))                     # lowest index among ties
        assert out["lse_t"] == pytest.approx(float(zt[0] / T - O.log_softmax_T(zt, T)[0]), rel=1e-12)
        assert out["lse_d"] == pytest.approx(float(zd[0] / T - O.log_softmax_T(zd, T)[0]), rel=1e-12)
        assert out["nkl"] == pytest.approx(O.nkl_pair(zt, zd, T)[0], rel=1e-9, abs=1e-13)


def test_sharded_draw_equals_the_whole_row():
    rng = np.random.default_rng(61)
    for _ in range(200):
        V = int(rng.integers(1, 60))
        w = np.where(rng.random(V) < 0.5, 0.0, rng.random(V))
        if not np.any(w > 0):
            w[int(rng.integers(0, V))] = 1.0
        u = float(rng.random())
        cuts = sorted(set(int(c) for c in rng.integers(1, V, 3))) if V > 1 else []
        bounds = [0] + cuts + [V]
        y, Z = O.sharded_draw([w[a:b] for a, b in zip(bounds, bounds[1:])], u)
        y0, Z0, c0, c1 = O.inverse_cdf(w, u)
        assert Z == pytest.approx(Z0, rel=1e-12)
        if abs(c0 / Z0 - u) > 1e-9 and abs(c1 / Z0 - u) > 1e-9:    # away from a boundary: exactly the token
            assert y == y0
        assert w[y] > 0


# ---------------------------------------------------------------- R6: a rejection that meets Z = 0

def test_zero_residual_draws_from_p_of_the_rejected_row():
    """R6. Identical target and draft rows give alpha = 1 and max(0, p - q) = 0 exactly; a
    uniform above 1 forces the rejection all the same (accept iff u <= alpha), so the
    residual has Z = 0 and the correction comes from p of the rejected position's own
    target row. V = 2 closed form: y = 1 iff u_sample >= sigmoid((z0 - z1) / T) of that
    row. The next target row and the bonus row lean the other way, so drawing from either
    (or reading the wrong position) changes y."""
    T = 0.9
    same = np.array([2.0, 0.0])                  # p0 = sigmoid(2 / T) = 0.902
    other = np.array([0.0, 2.0])                 # p0 = 0.098
    for n_rej in (0, 1):
        t = np.stack([other, other, other])
        t[n_rej] = same
        d = t[:2].copy()                          # draft rows equal to the target rows: alpha = 1
        u = np.array([0.0, 0.0])
        u[n_rej] = 1.5
        p0 = 1.0 / (1.0 + math.exp(-2.0 / T))
        for us in (0.05, 0.5, p0 - 1e-6, p0 + 1e-6, 0.99):
            r = O.verify_stochastic_sequence(t, d, np.array([1, 0]), T, u, us)
            assert r["alpha"][n_rej] == 1.0
            assert r["n"] == n_rej
            assert ("zero_residual", n_rej) in r["flags"] and r["flag"]
            assert r["tokens"][n_rej] == (1 if us >= p0 else 0), (n_rej, us)
            assert list(r["tokens"][:n_rej]) == [1, 0][:n_rej] and np.all(r["tokens"][n_rej + 1:] == -1)


def test_zero_residual_inverse_cdf_over_p_matches_scipy():
    """R6 with a longer row: the correction after a rejection on identical rows is the
    inverse CDF of scipy's softmax of that row at T, for uniforms away from its steps."""
    rng = np.random.default_rng(91)
    V, T = 7, 0.7
    row = rng.normal(0, 1.5, V)
    t = np.stack([row, rng.normal(0, 1.5, V)])
    p = sps.softmax(row / T)
    C = np.cumsum(p)
    for us in rng.random(40):
        if np.min(np.abs(C - us)) < 1e-9:
            continue
        r = O.verify_stochastic_sequence(t, row[None, :].copy(), np.array([3]), T, np.array([2.0]), float(us))
        assert r["n"] == 0 and r["tokens"][0] == int(np.argmax(C > us))


# ---------------------------------------------------------------- batch drivers over the packed layout

def _packed_ragged(seed, gammas, V):
    """A packed batch built by concatenating per-sequence arrays, so each sequence's rows
    are known without the layout's index arithmetic."""
    rng = np.random.default_rng(seed)
    per = []
    for g in gammas:
        t = rng.normal(0, 2, (g + 1, V)).astype(np.float32)
        d = (0.9 * t[:g] + rng.normal(0, 1, (g, V))).astype(np.float32)
        tok = rng.integers(0, V, g).astype(np.int32)
        amax = np.argmax(t[:g], axis=1) if g else np.zeros(0, np.int64)
        tok = np.where(rng.random(g) < 0.6, amax, tok).astype(np.int32)   # greedy runs of matches
        per.append((t, d, tok, rng.random(g).astype(np.float32), np.float32(rng.random())))
    target = np.concatenate([p[0] for p in per])
    draft = np.concatenate([p[1] for p in per]) if sum(gammas) else np.zeros((0, V), np.float32)
    tokens = np.concatenate([p[2] for p in per])
    u_acc = np.concatenate([p[3] for p in per])
    u_smp = np.array([p[4] for p in per], np.float32)
    cu = np.zeros(len(gammas) + 1, np.int32)
    cu[1:] = np.cumsum(gammas)
    return per, target, draft, tokens, u_acc, u_smp, cu


def _same(a, b):
    if isinstance(a, np.ndarray) or isinstance(b, np.ndarray):
        return np.array_equal(np.asarray(a), np.asarray(b), equal_nan=True)
    return a == b


def test_packed_drivers_index_every_sequence():
    """verify_stochastic, verify_greedy and nkl_rows on a ragged batch with empty sequences
    (first, middle and last) give, for every sequence, exactly the per-sequence functions'
    results on that sequence's own arrays: a slip in the target base cu[b] + b, the draft
    base cu[b] or the per-sequence uniform fails here."""
    gammas = [0, 3, 5, 0, 1, 4, 2, 0]
    V, T = 23, 0.8
    per, target, draft, tokens, u_acc, u_smp, cu = _packed_ragged(5, gammas, V)
    pos = np.arange(1, len(gammas) + 1, dtype=np.int32) * 7
    st = O.verify_stochastic(target, draft, tokens, cu, T, u_acc, u_smp, "f32", positions=pos, min_block_len=2)
    gr = O.verify_greedy(target, tokens, cu, "f32", min_block_len=2)
    nk = O.nkl_rows(target, draft, cu, T, "f32", positions=pos)
    assert sorted(st) == sorted(gr) == sorted(nk) == list(range(len(gammas)))
    for b, (t, d, tok, ua, us) in enumerate(per):
        t64, d64 = t.astype(np.float64), d.astype(np.float64)
        ref = O.verify_stochastic_sequence(t64, d64, tok, T, ua.astype(np.float64), float(us), position=int(pos[b]),
                                           min_block_len=2)
        for k in ("n", "tokens", "p_x", "q_x", "alpha", "nkl", "mask", "greedy_n", "greedy_tokens", "block_n",
                  "block_tokens", "flags"):
            assert _same(st[b][k], ref[k]), (b, k)
        gref = O.verify_greedy_sequence(t64, tok, min_block_len=2)
        for k in ("n", "tokens", "block_n", "block_tokens"):
            assert _same(gr[b][k], gref[k]), (b, k)
        want = [O.nkl_pair(t64[i], d64[i], T)[0] for i in range(len(tok))]
        assert np.array_equal(nk[b]["nkl"], np.array(want)), b
        thr = [O.position_delta(int(pos[b]) + i) for i in range(len(tok))]
        assert list(nk[b]["mask"]) == [1 if a < th else 0 for a, th in zip(want, thr)], b
    # the uniform each sequence draws with is its own: sequence b's u_sample drives its draw
    assert len({float(x) for x in u_smp}) == len(gammas)


def test_packed_tree_driver_indexes_every_sequence():
    """verify_tree over B packed trees equals verify_tree_sequence on each tree's own
    N + 1 rows (a slip in the row base b * (N + 1) or in the node-token row fails)."""
    rng = np.random.default_rng(6)
    parent = [-1, -1, 0, 1, 2, 2, 4]
    N, V, B = len(parent), 11, 5
    rows = [rng.normal(0, 1, (N + 1, V)).astype(np.float32) for _ in range(B)]
    for r in rows:
        r[:, 3] += 2.5                             # most argmaxes at token 3: deep accepted paths
    node = np.where(rng.random((B, N)) < 0.8, 3, rng.integers(0, V, (B, N))).astype(np.int32)
    res = O.verify_tree(np.concatenate(rows), node, parent, "f32")
    deepest = 0
    for b in range(B):
        ref = O.verify_tree_sequence(rows[b].astype(np.float64), node[b], parent)
        assert res[b]["len"] == ref["len"]
        assert np.array_equal(res[b]["path"], ref["path"]) and np.array_equal(res[b]["tokens"], ref["tokens"])
        deepest = max(deepest, ref["len"])
    assert deepest >= 3
