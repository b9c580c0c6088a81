"""Oracle: a plain fp64 CPU restatement of batched draft-token verification.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT. Only the tests, the package-level
smoke check and the benchmark's CPU-baseline / reference legs may import this
module. The CUDA library never calls it, and the two share no code, header,
table or helper; they meet only on the arrays of the seeded input generator.

Everything is computed in float64 from the exact widening of the stored logits
(bf16 bit patterns or fp32), one sequence at a time, in the order the pages give
the steps. Library primitives (max, sum, exp, log, cumsum, argmax) are the only
building blocks; there is no blocking, fusion or reordering beyond them.

Sources (page title, then section):
  [SpS] speculative-sampling article "大模型推理的投机采样：Draft 小模型辅助与验证加速",
        section "核心算法数学原理：无损拒绝采样" -- alpha = min(1, p(x)/q(x)); a draft
        token is accepted when a uniform r <= alpha; on rejection a new token is drawn
        from max(0, p - q)/norm and drafting stops there; section "核心实现" -- the target
        is evaluated on the last gamma+1 positions (one row per draft plus one more).
  [CoD] "Chain of Draft" article, section 3.2 (compute_nkl) -- both rows are softmaxed
        at one temperature, KL(draft || target) is summed over the vocabulary and
        divided by log(vocab size); drafts with NKL below delta = 0.15 are kept.
  [MTP] Gemma 4 multi-token-prediction drafter article, section 2.3 -- greedy
        verification: d_i is accepted while it equals the argmax of target row i; at
        the first mismatch r the target's own token replaces d_r; section 4.1 gives
        the same loop as pseudo-code.
  [PD]  Parallel Drafting article, section 2.2 -- the P-EAGLE draft tree (three root
        candidates, at most 12 nodes), verified by the longest accepted path.

Readings taken where the pages are silent, garbled or disagree:
  R1  bonus token: when all gamma drafts are accepted, one more token is drawn from
      target row gamma (the (gamma+1)-th row the pages slice out), by the same
      inverse-CDF rule as the correction.
  R2  correction on rejection follows [SpS]'s stated residual math, not the argmax
      shortcut in the same page's sample code.
  R3  no 1e-8 floor on q(x) (the sample code's max(1e-8, q)); q(x) > 0 for finite
      logits. Rows with q(x) < 1e-8 are flagged.
  R4  comparison: accept iff u <= alpha (u == alpha is accepted).
  R5  "norm" is Z = sum_v max(0, p_v - q_v).
  R6  if a rejection meets Z == 0 (only rounding can cause it), the correction is
      drawn from p at that position; the row is flagged.
  R7  inverse CDF in ascending token order with a strict ">": y = min{v : C(v) > u*Z},
      so a zero-mass token is never drawn; if rounding leaves u*Z >= C(V-1) the last
      token with positive mass is taken.
  R8  one u_sample per sequence serves either the correction or the bonus token.
  R9  one temperature T for target and draft ([CoD] 3.2: temperatures must match).
  R10 greedy argmax on the raw logits (T does not matter), ties to the lowest index.
  R11 NKL = KL(q || p) / ln V with q the draft distribution; natural log.
  R12 NKL is reported as the raw ratio, unclamped (KL(q||p) can exceed ln V).
  R13 accept mask = NKL < delta (strict).
  R14 the exact KL is the definition; the page's epsilon-guarded form
      sum q (log(q + 1e-12) - log(p + 1e-12)) is reported beside it.
  R15 tree: node j is accepted iff its token equals the argmax of its parent's row
      and its parent is accepted (roots compare against the parent row, row 0); the
      pick is the accepted node of greatest depth, ties to the lowest node index;
      the correction is the argmax of the picked node's row (row 0 if none).
  R17 a one-token vocabulary (V = 1): both rows are the same point mass, KL = 0, and
      the ratio 0 / ln 1 is taken as 0.
  R16 errors: a non-finite logit in any row a sequence uses, or a draft / node token
      outside [0, V), makes that sequence an error: its count is -1 and all its
      outputs are -1 (integers) or NaN (reals). For the standalone NKL call the
      error is per row pair.
  R18 position-adaptive threshold ([CoD] 4.3): delta_pos = min(delta_max,
      delta_base * (1 + a * log2(pos))) with pos the 1-based position of the token in
      the generated text (draft i of a sequence whose first draft sits at position P
      has pos = P + i); the page's printed values fit log2(pos), not log2(pos + 1).
      A first position below 1 has no threshold: every mask entry of that sequence
      is 0 (the other outputs do not depend on positions).
  R19 separate temperatures ([PD] 4.4: draft 0.3-0.5, target 0.7-0.9): p is
      softmax(z_t / T_t), q is softmax(z_d / T_d) -- the distribution the drafts were
      drawn from -- for p(x), q(x), alpha and the residual. NKL keeps [CoD] 3.2's rule
      that both rows are scaled by one temperature, the target's: KL(softmax(z_d / T_t)
      || softmax(z_t / T_t)) / ln V.
  R20 block-accept ([CoD] 3.3): the longest run of consecutive positions where the
      draft token equals the target's token (the argmax of the target row, R10) counts
      if it is at least min_len long (3 on the page); among equally long runs the
      earliest wins. Its end e is the number of draft tokens kept: the output is the
      draft tokens before e followed by the target's tokens from e on (gamma tokens in
      all); without such a run the output is the target's tokens and e = 0.
  R21 acceptance statistics ([MTP] 5.1: the acceptance rate is the accepted draft
      tokens per speculative round, total accepted / rounds; [PD] 5.2: ARSD, the
      standard deviation of the acceptance rate in a one-minute window, to be watched
      beside P99): a round is one sequence with gamma_b > 0 in one
      call; its acceptance rate is n_b / gamma_b; mean accepted = sum n_b / rounds;
      ARSD = the population standard deviation of the rates of the rounds in the
      window. The window is the caller's last W time buckets (a bucket is any
      monotone label the caller chooses, e.g. whole seconds).

  R22 multi-draft ([MTP] 6.2: several drafters each propose a draft, the target
      verifies all of them and the longest accepted path is kept; [CoD] 4.4: the
      pairwise NKL matrix of the drafts, consensus below 0.1, divergence above 0.15;
      the page's comparison operators are lost): a group holds K candidate
      sequences verified independently (greedy or stochastic); the kept candidate is
      the one with the most accepted drafts, the lowest index among equals (with
      stochastic verification this choice is not distribution-preserving; the page
      asks for it as stated). At draft position i the matrix is
      M[a][b] = KL(q_a || q_b) / ln V between the candidates' draft rows i at the one
      temperature T. Consensus at i: some pair a != b is below the consensus
      threshold in both directions; divergence at i: every entry off the diagonal is
      above the divergence threshold.

  R23 a row split over vocabulary shards (logits sharded over tensor-parallel ranks; the
      pages do not treat it): every statistic is a maximum, a log-sum-exp or a sum, so
      per-shard statistics merge associatively (sums moved to the larger maximum, the
      argmax by value then lowest index); the inverse-CDF draw takes the shard whose
      exclusive prefix of shard masses passes u * Z and that shard's own running sum.

Parity pins for every function: tests/test_oracle_pins.py.
"""
from __future__ import annotations

import math

import numpy as np

FLAG_BAND = 1e-5          # decisions closer than this to a boundary are flagged
NKL_EPS = 1e-12           # the guard in [CoD]'s compute_nkl code

ERR_TOKEN_RANGE = 1
ERR_NONFINITE = 2
ERR_OFFSETS = 4


# ---------------------------------------------------------------------------
# input widening (bit patterns -> exact float64)

def widen(raw: np.ndarray, dtype: str) -> np.ndarray:
    """Stored logits -> float64. bf16 is the high half of an IEEE fp32, so the
    widening is exact: shift the 16 stored bits into the top of a 32-bit word."""
    if dtype == "bf16":
        return (np.asarray(raw).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    if dtype == "f32":
        return np.asarray(raw, dtype=np.float32).astype(np.float64)
    raise ValueError(dtype)


# ---------------------------------------------------------------------------
# [CoD] 3.2 step 1: temperature-scaled softmax, here in log form

def log_softmax_T(z: np.ndarray, T: float) -> np.ndarray:
    """log softmax(z / T) over the last axis, two-pass (max, then log-sum-exp)."""
    s = z / T
    m = np.max(s, axis=-1, keepdims=True)
    lse = m + np.log(np.sum(np.exp(s - m), axis=-1, keepdims=True))
    return s - lse


def softmax_T(z: np.ndarray, T: float) -> np.ndarray:
    return np.exp(log_softmax_T(z, T))


# ---------------------------------------------------------------------------
# [SpS] acceptance, first rejection, residual, inverse CDF

def acceptance_prob(log_p_x: float, log_q_x: float) -> float:
    """alpha = min(1, p(x)/q(x)), evaluated as exp(min(0, log p(x) - log q(x)))."""
    return math.exp(min(0.0, log_p_x - log_q_x))


def first_rejection(u: np.ndarray, alpha: np.ndarray) -> int:
    """Number of leading accepted drafts: the first i with not (u_i <= alpha_i), else gamma (R4)."""
    for i in range(len(alpha)):
        if not (u[i] <= alpha[i]):
            return i
    return len(alpha)


def residual(p: np.ndarray, q: np.ndarray) -> np.ndarray:
    """max(0, p - q) over the vocabulary (unnormalised; R5)."""
    return np.maximum(0.0, p - q)


def inverse_cdf(w: np.ndarray, u: float):
    """Draw from the (unnormalised) weights w with the uniform u (R7).

    Returns (token, Z, C_before, C_at): Z = sum w, C = running sum in token order,
    token = min{v : C(v) > u*Z}; C_before = C(token-1) (0 for token 0), C_at = C(token)."""
    Z = float(np.sum(w))
    C = np.cumsum(w)
    target = u * Z
    hit = np.nonzero(C > target)[0]
    if hit.size:
        y = int(hit[0])
    else:
        y = int(np.nonzero(w > 0)[0][-1])
    c_before = float(C[y - 1]) if y > 0 else 0.0
    return y, Z, c_before, float(C[y])


# ---------------------------------------------------------------------------
# [CoD] 3.2: NKL

def nkl_pair(zt: np.ndarray, zd: np.ndarray, T: float):
    """(NKL, NKL_eps) for one (target row, draft row) pair, NKL = KL(q || p) / ln V.

    KL(q||p) = sum_v q_v (log q_v - log p_v) with q = softmax(zd/T), p = softmax(zt/T)."""
    V = zt.shape[-1]
    lp = log_softmax_T(zt, T)
    lq = log_softmax_T(zd, T)
    q = np.exp(lq)
    p = np.exp(lp)
    kl = float(np.sum(q * (lq - lp)))
    kl_eps = float(np.sum(q * (np.log(q + NKL_EPS) - np.log(p + NKL_EPS))))
    if V == 1:                                   # R17
        return 0.0, 0.0
    lnV = math.log(V)
    return kl / lnV, kl_eps / lnV


# ---------------------------------------------------------------------------
# one sequence, stochastic

def verify_stochastic_sequence(t_rows: np.ndarray, d_rows: np.ndarray, tokens: np.ndarray, T: float,
                               u_accept: np.ndarray, u_sample: float, nkl_delta: float = 0.15, *,
                               T_draft: float | None = None, position: int | None = None,
                               delta_alpha: float = 0.08, delta_max: float = 0.3, min_block_len: int = 0) -> dict:
    """Stochastic verification of one sequence ([SpS]; bonus token R1).

    t_rows: float64 [gamma+1, V]; d_rows: float64 [gamma, V]; tokens int [gamma].
    T_draft: the drafts' temperature when it differs from the target's (R19).
    position: 1-based position of the first draft; the NKL mask then compares against
    the position-adaptive threshold (R18). min_block_len > 0 adds the block-accept
    outputs (R20) computed from the target's argmax tokens."""
    g = d_rows.shape[0]
    V = t_rows.shape[1]
    out = {"n": -1, "tokens": np.full(g + 1, -1, dtype=np.int64),
           "p_x": np.full(g, np.nan), "q_x": np.full(g, np.nan), "alpha": np.full(g, np.nan),
           "nkl": np.full(g, np.nan), "nkl_eps": np.full(g, np.nan), "mask": np.zeros(g, dtype=np.uint8),
           "greedy_n": -1, "greedy_tokens": np.full(g + 1, -1, dtype=np.int64),
           "err": 0, "flag": False, "flags": []}
    if not (np.all(np.isfinite(t_rows)) and np.all(np.isfinite(d_rows))):
        out["err"] |= ERR_NONFINITE
    if np.any((tokens < 0) | (tokens >= V)):
        out["err"] |= ERR_TOKEN_RANGE
    if out["err"]:
        return out

    # temperature-scaled log-probabilities of every row (one T for both, R9, unless the
    # drafts were drawn at their own temperature, R19)
    Td = T if T_draft is None else T_draft
    lp = log_softmax_T(t_rows, T)          # [g+1, V]
    lq = log_softmax_T(d_rows, Td)         # [g, V]

    # gather at the drafted tokens, acceptance probability
    for i in range(g):
        x = int(tokens[i])
        out["p_x"][i] = math.exp(lp[i, x])
        out["q_x"][i] = math.exp(lq[i, x])
        out["alpha"][i] = acceptance_prob(lp[i, x], lq[i, x])
        if out["q_x"][i] < 1e-8:
            out["flags"].append(("q_below_1e-8", i))
        out["nkl"][i], out["nkl_eps"][i] = nkl_pair(t_rows[i], d_rows[i], T)   # both rows at T (R19)
        if position is not None and position < 1:
            out["mask"][i] = 0
        else:
            delta = nkl_delta if position is None else position_delta(position + i, nkl_delta, delta_alpha,
                                                                      delta_max)
            out["mask"][i] = 1 if out["nkl"][i] < delta else 0

    # first rejection
    n = first_rejection(u_accept, out["alpha"])
    for i in range(min(n + 1, g)):
        if abs(float(u_accept[i]) - out["alpha"][i]) < FLAG_BAND:
            out["flags"].append(("accept_band", i))

    # correction (residual) or bonus token
    if n < g:
        p = np.exp(lp[n])
        q = np.exp(lq[n])
        w = residual(p, q)
        if float(np.sum(w)) <= 1e-30:                     # R6
            out["flags"].append(("zero_residual", n))
            w = p
    else:
        w = np.exp(lp[g])
    y, Z, c0, c1 = inverse_cdf(w, float(u_sample))
    if abs(c0 / Z - u_sample) < FLAG_BAND or abs(c1 / Z - u_sample) < FLAG_BAND:
        out["flags"].append(("cdf_band", n))

    out["n"] = n
    out["tokens"][:n] = tokens[:n]
    out["tokens"][n] = y

    # greedy mode on the same rows (R10)
    gn, gtok = greedy_sequence_core(t_rows, tokens)
    out["greedy_n"], out["greedy_tokens"] = gn, gtok
    if min_block_len > 0:
        out["block_n"], out["block_tokens"] = block_accept(tokens, np.argmax(t_rows[:g], axis=1), min_block_len)
    out["flag"] = bool(out["flags"])
    return out


# ---------------------------------------------------------------------------
# greedy

def greedy_sequence_core(t_rows: np.ndarray, tokens: np.ndarray):
    """[MTP] 2.3: accept while d_i == argmax(target row i); at the first mismatch n the
    target's argmax replaces d_n; if all match, the argmax of row gamma follows."""
    g = len(tokens)
    amax = np.argmax(t_rows, axis=1)            # first maximal index = lowest-index tie-break
    n = g
    for i in range(g):
        if int(tokens[i]) != int(amax[i]):
            n = i
            break
    toks = np.full(g + 1, -1, dtype=np.int64)
    toks[:n] = tokens[:n]
    toks[n] = amax[n]
    return n, toks


def verify_greedy_sequence(t_rows: np.ndarray, tokens: np.ndarray, min_block_len: int = 0) -> dict:
    g = len(tokens)
    V = t_rows.shape[1]
    err = 0
    if not np.all(np.isfinite(t_rows)):
        err |= ERR_NONFINITE
    if np.any((tokens < 0) | (tokens >= V)):
        err |= ERR_TOKEN_RANGE
    if err:
        return {"n": -1, "tokens": np.full(g + 1, -1, dtype=np.int64), "err": err,
                "block_n": -1, "block_tokens": np.full(g, -1, dtype=np.int64)}
    n, toks = greedy_sequence_core(t_rows, tokens)
    res = {"n": n, "tokens": toks, "err": 0}
    if min_block_len > 0:
        res["block_n"], res["block_tokens"] = block_accept(tokens, np.argmax(t_rows[:g], axis=1), min_block_len)
    return res


# ---------------------------------------------------------------------------
# [CoD] 3.3 block-accept (R20)

def block_accept(draft_tokens, target_tokens, min_len: int = 3):
    """(e, tokens): the longest run of consecutive positions with draft == target, if it is
    at least min_len long (the earliest of equally long runs), keeps the draft tokens up
    to its end e; the target's tokens fill the rest. Without such a run: (0, target)."""
    d = [int(x) for x in draft_tokens]
    t = [int(x) for x in target_tokens]
    g = len(d)
    best_len, best_start = 0, 0
    run = 0
    for i in range(g):
        run = run + 1 if d[i] == t[i] else 0
        if run > best_len:                    # a strictly longer run; ties keep the earlier
            best_len, best_start = run, i - run + 1
    if best_len < min_len:
        return 0, np.array(t, dtype=np.int64)
    e = best_start + best_len
    return e, np.array(d[:e] + t[e:], dtype=np.int64)


# ---------------------------------------------------------------------------
# tree

def tree_depths(parent) -> list:
    depth = []
    for j, pj in enumerate(parent):
        depth.append(1 if pj < 0 else depth[pj] + 1)
    return depth


def verify_tree_sequence(t_rows: np.ndarray, node_tokens: np.ndarray, parent) -> dict:
    """[PD] 2.2 tree, read as R15. t_rows [N+1, V]: row 0 is the parent position,
    row j+1 scores the token that follows node j."""
    N = len(parent)
    V = t_rows.shape[1]
    depth = tree_depths(parent)
    Dmax = max(depth) if N else 0
    res = {"len": -1, "path": np.full(Dmax, -1, dtype=np.int64),
           "tokens": np.full(Dmax + 1, -1, dtype=np.int64), "err": 0}
    if not np.all(np.isfinite(t_rows)):
        res["err"] |= ERR_NONFINITE
    if np.any((node_tokens < 0) | (node_tokens >= V)):
        res["err"] |= ERR_TOKEN_RANGE
    if res["err"]:
        return res
    amax = np.argmax(t_rows, axis=1)
    ok = [False] * N
    for j in range(N):
        prow = 0 if parent[j] < 0 else parent[j] + 1
        ok[j] = int(node_tokens[j]) == int(amax[prow]) and (parent[j] < 0 or ok[parent[j]])
    pick, best = -1, 0
    for j in range(N):
        if ok[j] and depth[j] > best:
            pick, best = j, depth[j]
    chain = []
    k = pick
    while k >= 0:
        chain.append(k)
        k = parent[k]
    chain.reverse()
    res["len"] = best
    res["path"][:best] = chain
    res["tokens"][:best] = [int(node_tokens[j]) for j in chain]
    res["tokens"][best] = int(amax[pick + 1]) if pick >= 0 else int(amax[0])
    return res


# ---------------------------------------------------------------------------
# batch drivers over the packed layout (target rows of sequence b start at
# cu_draft[b] + b, draft rows at cu_draft[b])

def verify_stochastic(target_raw, draft_raw, tokens, cu_draft, T, u_accept, u_sample, dtype,
                      nkl_delta=0.15, seqs=None, *, T_draft=None, positions=None, delta_alpha=0.08,
                      delta_max=0.3, min_block_len=0) -> dict:
    """Run verify_stochastic_sequence over sequences `seqs` (default: all). positions:
    per-sequence 1-based position of the first draft (R18), or None."""
    B = len(cu_draft) - 1
    seqs = range(B) if seqs is None else seqs
    res = {}
    for b in seqs:
        d0, d1 = int(cu_draft[b]), int(cu_draft[b + 1])
        t0 = d0 + b
        g = d1 - d0
        t_rows = widen(target_raw[t0:t0 + g + 1], dtype)
        d_rows = widen(draft_raw[d0:d1], dtype)
        res[b] = verify_stochastic_sequence(t_rows, d_rows, np.asarray(tokens[d0:d1]), T,
                                            np.asarray(u_accept[d0:d1], dtype=np.float64),
                                            float(u_sample[b]), nkl_delta, T_draft=T_draft,
                                            position=None if positions is None else int(positions[b]),
                                            delta_alpha=delta_alpha, delta_max=delta_max,
                                            min_block_len=min_block_len)
    return res


def verify_greedy(target_raw, tokens, cu_draft, dtype, seqs=None, min_block_len=0) -> dict:
    B = len(cu_draft) - 1
    seqs = range(B) if seqs is None else seqs
    res = {}
    for b in seqs:
        d0, d1 = int(cu_draft[b]), int(cu_draft[b + 1])
        t0 = d0 + b
        res[b] = verify_greedy_sequence(widen(target_raw[t0:t0 + (d1 - d0) + 1], dtype),
                                        np.asarray(tokens[d0:d1]), min_block_len)
    return res


def verify_tree(target_raw, node_tokens, parent, dtype, seqs=None) -> dict:
    N = len(parent)
    B = node_tokens.shape[0]
    seqs = range(B) if seqs is None else seqs
    res = {}
    for b in seqs:
        rows = widen(target_raw[b * (N + 1):(b + 1) * (N + 1)], dtype)
        res[b] = verify_tree_sequence(rows, np.asarray(node_tokens[b]), list(parent))
    return res


def nkl_rows(target_raw, draft_raw, cu_draft, T, dtype, delta=0.15, seqs=None, *, positions=None,
             delta_alpha=0.08, delta_max=0.3) -> dict:
    """Standalone NKL over every (target row i, draft row i) pair of the chosen sequences,
    per-row errors (R16); positions: as in verify_stochastic (R18)."""
    B = len(cu_draft) - 1
    seqs = range(B) if seqs is None else seqs
    res = {}
    for b in seqs:
        d0, d1 = int(cu_draft[b]), int(cu_draft[b + 1])
        t0 = d0 + b
        vals, eps, mask = [], [], []
        for i in range(d1 - d0):
            zt = widen(target_raw[t0 + i], dtype)
            zd = widen(draft_raw[d0 + i], dtype)
            if not (np.all(np.isfinite(zt)) and np.all(np.isfinite(zd))):
                vals.append(np.nan), eps.append(np.nan), mask.append(0)
                continue
            a, e = nkl_pair(zt, zd, T)
            if positions is not None and int(positions[b]) < 1:
                vals.append(a), eps.append(e), mask.append(0)
                continue
            dl = delta if positions is None else position_delta(int(positions[b]) + i, delta, delta_alpha, delta_max)
            vals.append(a), eps.append(e), mask.append(1 if a < dl else 0)
        res[b] = {"nkl": np.array(vals), "nkl_eps": np.array(eps), "mask": np.array(mask, dtype=np.uint8)}
    return res


def position_delta(pos: int, delta_base: float = 0.15, a: float = 0.08, delta_max: float = 0.3) -> float:
    """[CoD] 4.3 position-adaptive threshold, read with log2(pos), pos 1-based, capped at
    delta_max: the page's printed values at pos 1 (0.15) and 1024 (0.27) fit log2(pos),
    not the log2(pos + 1) its formula shows; its 0.192 at pos 128 fits neither."""
    return min(delta_max, delta_base * (1.0 + a * math.log2(pos)))


# ---------------------------------------------------------------------------
# acceptance statistics (R21)

def acceptance_summary(records, bucket_now: int, window: int) -> dict:
    """records: iterable of (bucket, n_b, gamma_b) per verified sequence. Over the rounds
    whose bucket lies in (bucket_now - window, bucket_now] and whose gamma_b > 0: rounds,
    accepted = sum n_b, drafted = sum gamma_b, mean accepted per round, mean rate, and
    ARSD = the population standard deviation of the rates n_b / gamma_b (two passes)."""
    rates, acc, drafted = [], 0, 0
    for bucket, n, g in records:
        if bucket_now - window < bucket <= bucket_now and g > 0 and n >= 0:
            rates.append(n / g)
            acc += n
            drafted += g
    R = len(rates)
    if R == 0:
        return {"rounds": 0, "accepted": 0, "drafted": 0, "mean_accepted": 0.0, "mean_rate": 0.0, "arsd": 0.0}
    mean = sum(rates) / R
    var = sum((r - mean) ** 2 for r in rates) / R
    return {"rounds": R, "accepted": acc, "drafted": drafted, "mean_accepted": acc / R, "mean_rate": mean,
            "arsd": math.sqrt(var)}


# ---------------------------------------------------------------------------
# multi-draft verification (R22)

def pairwise_nkl(d_rows: np.ndarray, T: float) -> np.ndarray:
    """M[a][b] = KL(q_a || q_b) / ln V for the K draft rows d_rows [K, V] at temperature T
    (q_k = softmax(d_rows[k] / T)); zero diagonal."""
    K = d_rows.shape[0]
    M = np.zeros((K, K))
    for a in range(K):
        for b in range(K):
            if a != b:
                M[a, b] = nkl_pair(d_rows[b], d_rows[a], T)[0]    # nkl_pair(target=p, draft=q)
    return M


def consensus_divergence(M: np.ndarray, c_thr: float = 0.1, d_thr: float = 0.15):
    K = M.shape[0]
    off = [(a, b) for a in range(K) for b in range(K) if a != b]
    cons = any(M[a, b] < c_thr and M[b, a] < c_thr for a, b in off)
    div = all(M[a, b] > d_thr for a, b in off)
    return cons, div


def verify_multi(target_raw, draft_raw, tokens, G: int, K: int, gamma: int, T: float, dtype, stochastic: bool,
                 u_accept=None, u_sample=None, c_thr=0.1, d_thr=0.15, groups=None) -> dict:
    """Groups of K candidate sequences (sequence g*K + k, dense gamma drafts each, laid out
    like verify_stochastic's dense batches). Per group: the candidates' results, the kept
    candidate (most accepted drafts, lowest index among equals), its tokens, and per draft
    position the pairwise NKL matrix with the consensus and divergence flags."""
    groups = range(G) if groups is None else groups
    res = {}
    for g in groups:
        seqs = [g * K + k for k in range(K)]
        cu = np.arange(G * K + 1, dtype=np.int64) * gamma
        if stochastic:
            r = verify_stochastic(target_raw, draft_raw, tokens, cu, T, u_accept, u_sample, dtype, seqs=seqs)
            cand = [{"n": r[b]["n"], "tokens": r[b]["tokens"], "flag": r[b]["flag"]} for b in seqs]
        else:
            r = verify_greedy(target_raw, tokens, cu, dtype, seqs=seqs)
            cand = [{"n": r[b]["n"], "tokens": r[b]["tokens"], "flag": False} for b in seqs]
        ns = [c["n"] for c in cand]
        best = int(np.argmax(ns))                      # first maximal index
        mats, cons, div = [], [], []
        for i in range(gamma):
            rows = np.stack([widen(draft_raw[(g * K + k) * gamma + i], dtype) for k in range(K)])
            M = pairwise_nkl(rows, T)
            c, d = consensus_divergence(M, c_thr, d_thr)
            mats.append(M), cons.append(c), div.append(d)
        res[g] = {"cand": cand, "best_k": best if ns[best] >= 0 else -1, "best_n": ns[best],
                  "best_tokens": cand[best]["tokens"], "pair_nkl": np.array(mats).reshape(gamma, K, K),
                  "consensus": np.array(cons, dtype=np.uint8), "divergence": np.array(div, dtype=np.uint8)}
    return res


# ---------------------------------------------------------------------------
# the same definitions over a partition of the vocabulary (shards of a row, e.g. logits
# split over tensor-parallel ranks): every statistic above is a log-sum-exp, a maximum or
# a sum, so per-shard statistics combine associatively into the full row's

def shard_stats(z_t: np.ndarray, z_d: np.ndarray, T: float, v0: int) -> dict:
    """Statistics of one shard [v0, v0 + len) of a (target row, draft row) pair at T:
    target maximum m_t of z_t / T and S_t = sum exp(z_t / T - m_t); the lowest global index
    of the raw target maximum; draft m_d, S_d likewise; K = sum exp(z_d / T - m_d) *
    (z_d - z_t) / T."""
    st, sd = z_t / T, z_d / T
    m_t, m_d = float(np.max(st)), float(np.max(sd))
    e_d = np.exp(sd - m_d)
    return {"m_t": m_t, "S_t": float(np.sum(np.exp(st - m_t))), "amax_v": float(np.max(z_t)),
            "amax_i": v0 + int(np.argmax(z_t)), "m_d": m_d, "S_d": float(np.sum(e_d)),
            "K": float(np.sum(e_d * (sd - st)))}


def merge_stats(a: dict, b: dict) -> dict:
    """Associative combination of two shards' statistics (sums moved to the larger maximum;
    argmax by value, then the lower index)."""
    m_t = max(a["m_t"], b["m_t"])
    m_d = max(a["m_d"], b["m_d"])
    fa, fb = math.exp(a["m_d"] - m_d), math.exp(b["m_d"] - m_d)
    if a["amax_v"] > b["amax_v"] or (a["amax_v"] == b["amax_v"] and a["amax_i"] < b["amax_i"]):
        av, ai = a["amax_v"], a["amax_i"]
    else:
        av, ai = b["amax_v"], b["amax_i"]
    return {"m_t": m_t, "S_t": a["S_t"] * math.exp(a["m_t"] - m_t) + b["S_t"] * math.exp(b["m_t"] - m_t),
            "amax_v": av, "amax_i": ai, "m_d": m_d, "S_d": a["S_d"] * fa + b["S_d"] * fb,
            "K": a["K"] * fa + b["K"] * fb}


def stats_outputs(st: dict, V: int) -> dict:
    """Full-row quantities from merged statistics: lse_t, lse_d (of z / T, lse = m + ln S),
    the argmax, and NKL with KL(q || p) = K / S_d - lse_d + lse_t."""
    lse_t = st["m_t"] + math.log(st["S_t"])
    lse_d = st["m_d"] + math.log(st["S_d"])
    kl = st["K"] / st["S_d"] - lse_d + lse_t
    return {"lse_t": lse_t, "lse_d": lse_d, "argmax": st["amax_i"], "nkl": 0.0 if V == 1 else kl / math.log(V)}


def sharded_draw(weights_per_shard, u: float):
    """Inverse-CDF draw over a row split into shards (token order = shard order): Z_s per
    shard, an exclusive scan picks the shard whose range passes u * Z, and that shard's
    own running sum finds the token. Returns (global token, Z)."""
    Zs = [float(np.sum(w)) for w in weights_per_shard]
    Z = float(sum(Zs))
    target = u * Z
    base, off = 0.0, 0
    for s, w in enumerate(weights_per_shard):
        if base + Zs[s] > target or s == len(weights_per_shard) - 1:
            C = base + np.cumsum(w)
            hit = np.nonzero(C > target)[0]
            if hit.size:
                return off + int(hit[0]), Z
            nz = np.nonzero(w > 0)[0]
            return off + (int(nz[-1]) if nz.size else len(w) - 1), Z
        base += Zs[s]
        off += len(w)
    return off - 1, Z
