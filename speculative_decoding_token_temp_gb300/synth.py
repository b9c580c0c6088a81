"""Seeded synthetic workloads for batched draft-token verification.

This module holds random draws and the fp32 -> bf16 rounding of the drawn
logits, nothing else: no softmax, no acceptance rule, no residual and no
inverse-CDF sampling. The fp64 oracle and the CUDA library are both fed the
identical arrays it returns, so it is the one piece the two sides share.

Recipe (the workload shape the speculative-decoding pages describe: a target
forward over the gamma drafted positions plus one, and a drafter whose rows
agree with the target's most of the time):

  target row  z_t = 3 * N(0, 1) per token, plus 8 on one uniformly drawn "peak" token
  draft row   z_d = 0.9 * (z_t without its +8) + N(0, 1), plus 0.9 * 8 on the draft's peak;
              the draft's peak is the target's peak with probability `agreement`
              (0.8; 0.7 for the ragged multi-token-head shape), else a uniform token
  draft token a sample from softmax(z_d / T) taken with the Gumbel-max construction
              argmax_v (z_d[v] / T + G_v), G_v = -log E_v, E_v ~ Exp(1); the rows are
              first rounded to the storage dtype so that the token is a sample of the
              very distribution the verifier sees
  uniforms    u_accept[sum gamma_b] and u_sample[B], fp32 in [0, 1)
  rounding    logits are drawn in fp32 and, for bf16 workloads, rounded to bf16
              (round to nearest, ties to even)

Layout (the library's packed layout): target rows [sum_b (gamma_b + 1), V] with
sequence b's rows starting at cu_draft[b] + b; draft rows and tokens
[sum_b gamma_b, V] starting at cu_draft[b]. A dense batch is the special case
gamma_b = gamma for all b.

Every sequence draws from its own stream, numpy.random.default_rng([seed, b]),
so one sequence of a large workload can be regenerated alone.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

BF16 = "bf16"
F32 = "f32"

PEAK_BONUS = 8.0
TARGET_SIGMA = 3.0
DRAFT_SCALE = 0.9

# Tree shape of the P-EAGLE style draft tree used by the tree workload: three
# root candidates, each followed by a chain of three tokens (12 nodes), nodes
# numbered breadth-first so that every parent precedes its children.
TREE_PARENT = (-1, -1, -1, 0, 1, 2, 3, 4, 5, 6, 7, 8)


def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 array -> uint16 bf16 bit patterns, round to nearest even (finite inputs)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    b = b + (np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1)))
    return (b >> np.uint32(16)).astype(np.uint16)


def bf16_bits_as_f32(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> the fp32 values they encode (exact)."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def storage(x32: np.ndarray, dtype: str) -> np.ndarray:
    """Store fp32 logits in the workload's dtype (bf16 bits as uint16, or fp32)."""
    if dtype == BF16:
        return round_to_bf16_bits(x32)
    if dtype == F32:
        return np.ascontiguousarray(x32, dtype=np.float32)
    raise ValueError(f"unknown dtype {dtype!r}")


def stored_as_f32(a: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_bits_as_f32(a) if dtype == BF16 else a.astype(np.float32, copy=False)


@dataclass
class StochasticWorkload:
    """One batch for the stochastic / greedy / NKL calls (packed layout)."""
    B: int
    V: int
    dtype: str
    T: float
    gammas: np.ndarray          # int32 [B]
    cu_draft: np.ndarray        # int32 [B+1], prefix sums of gammas
    target: np.ndarray          # [sum(gamma+1), V] uint16 (bf16 bits) or float32
    draft: np.ndarray           # [sum(gamma), V]
    tokens: np.ndarray          # int32 [sum(gamma)]
    u_accept: np.ndarray        # float32 [sum(gamma)]
    u_sample: np.ndarray        # float32 [B]
    dense: bool = True
    name: str = ""

    @property
    def gamma_max(self) -> int:
        return int(self.gammas.max()) if self.B else 0

    @property
    def total_draft(self) -> int:
        return int(self.cu_draft[-1])

    @property
    def total_target(self) -> int:
        return self.total_draft + self.B

    def target_base(self, b: int) -> int:
        return int(self.cu_draft[b]) + b

    def draft_base(self, b: int) -> int:
        return int(self.cu_draft[b])

    def sequence(self, b: int):
        """(target rows [g+1, V], draft rows [g, V], tokens [g], u_accept [g], u_sample) of sequence b."""
        g = int(self.gammas[b])
        t0, d0 = self.target_base(b), self.draft_base(b)
        return (self.target[t0:t0 + g + 1], self.draft[d0:d0 + g], self.tokens[d0:d0 + g],
                self.u_accept[d0:d0 + g], float(self.u_sample[b]))

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == BF16 else 4


@dataclass
class TreeWorkload:
    """One batch for the tree call: per sequence the parent row plus one row per node."""
    B: int
    N: int
    V: int
    dtype: str
    parent: np.ndarray          # int32 [N], topologically ordered
    target: np.ndarray          # [B*(N+1), V]; row 0 of a sequence = parent row, row j+1 = node j
    node_tokens: np.ndarray     # int32 [B, N]
    name: str = ""

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == BF16 else 4


def _for_each(fn, n: int) -> None:
    """Run fn(0..n-1); sequences draw from independent streams, so the order and the
    thread count do not change the result (numpy releases the GIL in the bulk draws)."""
    workers = min(16, os.cpu_count() or 1, max(1, n))
    if workers == 1 or n < 4:
        for b in range(n):
            fn(b)
        return
    with ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(fn, range(n)))


def _draw_sequence(rng, gamma: int, V: int, dtype: str, T: float, agreement: float):
    """Target rows [gamma+1, V], draft rows [gamma, V] (storage dtype), tokens, u_accept."""
    base = rng.standard_normal((gamma + 1, V), dtype=np.float32)
    base *= np.float32(TARGET_SIGMA)
    peak_t = rng.integers(0, V, size=gamma + 1)
    noise = rng.standard_normal((gamma, V), dtype=np.float32)
    keep = rng.random(gamma) < agreement
    moved = rng.integers(0, V, size=gamma)
    peak_d = np.where(keep, peak_t[:gamma], moved)
    expo = rng.standard_exponential((gamma, V), dtype=np.float32)
    u_acc = rng.random(gamma, dtype=np.float32)

    draft32 = np.float32(DRAFT_SCALE) * base[:gamma] + noise
    draft32[np.arange(gamma), peak_d] += np.float32(DRAFT_SCALE * PEAK_BONUS)
    target32 = base
    target32[np.arange(gamma + 1), peak_t] += np.float32(PEAK_BONUS)

    t_st = storage(target32, dtype)
    d_st = storage(draft32, dtype)
    d_seen = stored_as_f32(d_st, dtype)
    gumbel = -np.log(np.maximum(expo, np.float32(np.finfo(np.float32).tiny)))
    tokens = np.argmax(d_seen / np.float32(T) + gumbel, axis=1).astype(np.int32)
    return t_st, d_st, tokens, u_acc


def sequence_data(seed: int, b: int, gamma: int, V: int, dtype: str, T: float, agreement: float):
    """Sequence b of a make_stochastic batch with this seed, on its own (its random stream
    depends only on (seed, b)): target rows, draft rows, tokens, u_accept, u_sample."""
    rng = np.random.default_rng([seed, b])
    t_st, d_st, tok, ua = _draw_sequence(rng, gamma, V, dtype, T, agreement)
    return t_st, d_st, tok, ua, rng.random(dtype=np.float32)


def make_stochastic(B: int, V: int, dtype: str, T: float, seed: int, gamma: int | None = None,
                    gamma_range: tuple[int, int] | None = None, agreement: float = 0.8,
                    name: str = "") -> StochasticWorkload:
    """Dense batch (gamma given) or ragged batch (gamma_b ~ U{lo..hi}, gamma_range given)."""
    if (gamma is None) == (gamma_range is None):
        raise ValueError("give exactly one of gamma / gamma_range")
    if gamma is not None:
        gammas = np.full(B, gamma, dtype=np.int32)
        dense = True
    else:
        lo, hi = gamma_range
        gammas = np.random.default_rng([seed, 0x6A77]).integers(lo, hi + 1, size=B).astype(np.int32)
        dense = False
    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(gammas)
    tot_d = int(cu[-1])
    sdt = np.uint16 if dtype == BF16 else np.float32
    target = np.empty((tot_d + B, V), dtype=sdt)
    draft = np.empty((tot_d, V), dtype=sdt)
    tokens = np.empty(tot_d, dtype=np.int32)
    u_acc = np.empty(tot_d, dtype=np.float32)
    u_smp = np.empty(B, dtype=np.float32)
    def one(b):
        g = int(gammas[b])
        t_st, d_st, tok, ua, us = sequence_data(seed, b, g, V, dtype, T, agreement)
        t0, d0 = int(cu[b]) + b, int(cu[b])
        target[t0:t0 + g + 1] = t_st
        draft[d0:d0 + g] = d_st
        tokens[d0:d0 + g] = tok
        u_acc[d0:d0 + g] = ua
        u_smp[b] = us

    _for_each(one, B)
    return StochasticWorkload(B=B, V=V, dtype=dtype, T=float(T), gammas=gammas, cu_draft=cu,
                              target=target, draft=draft, tokens=tokens, u_accept=u_acc,
                              u_sample=u_smp, dense=dense, name=name)


def make_multi(G: int, K: int, gamma: int, V: int, dtype: str, T: float, seed: int,
               spreads=(0.02, 0.3, 1.5)) -> StochasticWorkload:
    """Multi-draft groups: G groups of K candidate sequences (candidate k of group g is
    sequence g*K + k of the dense batch returned). The candidates of a group share a
    context: their target rows are one base plus a small per-candidate perturbation, and
    their draft rows one shared draft plus per-candidate noise of standard deviation
    spreads[g % len(spreads)] -- small spreads give candidates that agree, large ones
    candidates that diverge. Draft tokens are Gumbel-max samples of softmax(draft / T)."""
    B = G * K
    sdt = np.uint16 if dtype == BF16 else np.float32
    target = np.empty((B * (gamma + 1), V), dtype=sdt)
    draft = np.empty((B * gamma, V), dtype=sdt)
    tokens = np.empty(B * gamma, dtype=np.int32)
    u_acc = np.empty(B * gamma, dtype=np.float32)
    u_smp = np.empty(B, dtype=np.float32)

    def one(g):
        rng = np.random.default_rng([seed, g])
        spread = np.float32(spreads[g % len(spreads)])
        base = rng.standard_normal((gamma + 1, V), dtype=np.float32) * np.float32(TARGET_SIGMA)
        peak_t = rng.integers(0, V, size=gamma + 1)
        base[np.arange(gamma + 1), peak_t] += np.float32(PEAK_BONUS)
        shared = np.float32(DRAFT_SCALE) * base[:gamma] + rng.standard_normal((gamma, V), dtype=np.float32)
        for k in range(K):
            b = g * K + k
            t32 = base + np.float32(0.1) * rng.standard_normal((gamma + 1, V), dtype=np.float32)
            d32 = shared + spread * rng.standard_normal((gamma, V), dtype=np.float32)
            expo = rng.standard_exponential((gamma, V), dtype=np.float32)
            target[b * (gamma + 1):(b + 1) * (gamma + 1)] = storage(t32, dtype)
            d_st = storage(d32, dtype)
            draft[b * gamma:(b + 1) * gamma] = d_st
            gumbel = -np.log(np.maximum(expo, np.float32(np.finfo(np.float32).tiny)))
            tokens[b * gamma:(b + 1) * gamma] = np.argmax(stored_as_f32(d_st, dtype) / np.float32(T) + gumbel, axis=1)
            u_acc[b * gamma:(b + 1) * gamma] = rng.random(gamma, dtype=np.float32)
            u_smp[b] = rng.random(dtype=np.float32)

    _for_each(one, G)
    gammas = np.full(B, gamma, dtype=np.int32)
    cu = np.arange(B + 1, dtype=np.int32) * gamma
    return StochasticWorkload(B=B, V=V, dtype=dtype, T=float(T), gammas=gammas, cu_draft=cu, target=target,
                              draft=draft, tokens=tokens, u_accept=u_acc, u_sample=u_smp, dense=True,
                              name=f"multi G={G} K={K}")


def make_tree(B: int, V: int, dtype: str, seed: int, parent=TREE_PARENT, agreement: float = 0.8,
              name: str = "") -> TreeWorkload:
    """Tree batch: a draft row is drawn beside every target row; root candidates are the
    three largest distinct entries of the parent row's draft, every other node is the
    argmax of the draft row drawn beside its parent's row. The draft rows are then dropped."""
    parent = np.asarray(parent, dtype=np.int32)
    N = int(parent.shape[0])
    roots = [j for j in range(N) if parent[j] < 0]
    sdt = np.uint16 if dtype == BF16 else np.float32
    target = np.empty((B * (N + 1), V), dtype=sdt)
    node_tokens = np.empty((B, N), dtype=np.int32)
    def one(b):
        rng = np.random.default_rng([seed, b])
        base = rng.standard_normal((N + 1, V), dtype=np.float32)
        base *= np.float32(TARGET_SIGMA)
        peak_t = rng.integers(0, V, size=N + 1)
        noise = rng.standard_normal((N + 1, V), dtype=np.float32)
        keep = rng.random(N + 1) < agreement
        moved = rng.integers(0, V, size=N + 1)
        peak_d = np.where(keep, peak_t, moved)
        d32 = np.float32(DRAFT_SCALE) * base + noise
        d32[np.arange(N + 1), peak_d] += np.float32(DRAFT_SCALE * PEAK_BONUS)
        base[np.arange(N + 1), peak_t] += np.float32(PEAK_BONUS)
        target[b * (N + 1):(b + 1) * (N + 1)] = storage(base, dtype)
        d_seen = stored_as_f32(storage(d32, dtype), dtype)
        order = np.argsort(-d_seen[0], kind="stable")
        for k, j in enumerate(roots):
            node_tokens[b, j] = order[k]
        for j in range(N):
            if parent[j] >= 0:
                node_tokens[b, j] = int(np.argmax(d_seen[parent[j] + 1]))

    _for_each(one, B)
    return TreeWorkload(B=B, N=N, V=V, dtype=dtype, parent=parent, target=target,
                        node_tokens=node_tokens, name=name)


@dataclass
class Config:
    name: str
    kind: str                    # "stochastic" or "tree"
    B: int
    V: int
    dtype: str
    T: tuple = (1.0,)
    gamma: int | None = None
    gamma_range: tuple | None = None
    agreement: float = 0.8
    seed: int = 0
    extra: dict = field(default_factory=dict)

    def make(self, T: float | None = None, seed: int | None = None, B: int | None = None, V: int | None = None):
        s = self.seed if seed is None else seed
        nb = self.B if B is None else B
        nv = self.V if V is None else V
        if self.kind == "tree":
            return make_tree(nb, nv, self.dtype, s, name=self.name)
        return make_stochastic(nb, nv, self.dtype, self.T[0] if T is None else T, s,
                               gamma=self.gamma, gamma_range=self.gamma_range,
                               agreement=self.agreement, name=self.name)


# The five workloads: a tiny fp32 case, a mid-size bf16 case at two temperatures,
# the B=256 / gamma=8 / V=128256 headline, the 12-node tree, and the ragged
# multi-token-head batch with gamma_b ~ U{1..16} over a 152064-token vocabulary.
TINY = Config("tiny_B1_g4_V1000_f32", "stochastic", B=1, V=1000, dtype=F32, T=(1.0,), gamma=4, seed=0)
MID = Config("B64_g5_V32000_bf16", "stochastic", B=64, V=32000, dtype=BF16, T=(0.6, 1.0), gamma=5, seed=1)
HEADLINE = Config("B256_g8_V128256_bf16", "stochastic", B=256, V=128256, dtype=BF16, T=(0.6,), gamma=8, seed=2)
TREE = Config("tree_B32_N12_V128256_bf16", "tree", B=32, V=128256, dtype=BF16, seed=3)
RAGGED = Config("ragged_B512_g1-16_V152064_bf16", "stochastic", B=512, V=152064, dtype=BF16, T=(0.8,),
                gamma_range=(1, 16), agreement=0.7, seed=4)
WORKLOADS = {c.name: c for c in (TINY, MID, HEADLINE, TREE, RAGGED)}
