// Tile kernel and per-sequence finalisation (see kernels.cuh for the pipeline).
#pragma once

#include "kernels.cuh"
#include "kernels_sample.cuh"

namespace sv {

__global__ void prologue_kernel(const __grid_constant__ ProParams p) {
  // Launched programmatically after whatever precedes the call on the stream: the tile
  // kernel may be scheduled at once, but nothing here touches memory before the
  // preceding work has completed.
  griddep_launch();
  griddep_wait();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < p.nzero2) p.zero2[b] = 0u;
  if (b == 0 && in_ext(p.cntA + p.B, sizeof(unsigned), p.x_ws, p.status)) {
    p.cntA[p.B] = 0u;
    if (p.stats != nullptr && p.stats->bucket != p.bucket) {
      // a new time bucket takes over the slot (every finaliser of this call runs after
      // the prologue has completed, and every earlier call has completed)
      p.stats->rounds = p.stats->accepted = p.stats->drafted = 0;
      p.stats->rate_fx = p.stats->rate2_fx = 0;
      p.stats->bucket = p.bucket;
    }
  }
  if (b >= p.B) return;
  if (!in_ext(p.cntA + b, sizeof(unsigned), p.x_ws, p.status) || !in_ext(p.cntB + b, sizeof(unsigned), p.x_ws, p.status) ||
      !in_ext(p.rec + b, sizeof(SeqRec), p.x_ws, p.status))
    return;
  p.cntA[b] = 0u;
  p.cntB[b] = 0u;
  SeqRec q;
  q.state = REC_PENDING;
  q.n = -1;
  q.t_row = -1;
  q.d_row = -1;
  q.lt2 = 0.f;
  q.ld2 = 0.f;
  q.us = 0.f;
  q.mode = 0;
  p.rec[b] = q;
  if (p.cu != nullptr) {
    const int c0 = __ldg(p.cu + b), c1 = __ldg(p.cu + b + 1);
    const bool own = c1 >= c0 && c1 - c0 <= p.gamma && c0 >= 0 && c1 <= p.total_draft;  // its rows are in range
    const bool bad = !own || (b == 0 && c0 != 0) || (b == p.B - 1 && c1 != p.total_draft);
    if (bad) atomicOr(p.status, SPEC_DEV_OFFSETS);
    // the row -> sequence table the tiles look themselves up in: rows [c0 + hb b, c1 + hb (b+1))
    // (with offsets out of order a row may keep an older entry: the tile's own checks of
    // the offsets then report it)
    if (own && p.row_seq != nullptr) {
      const int r1 = min(c1 + p.hb * (b + 1), p.total_rows);
      for (int r = c0 + p.hb * b; r < r1; ++r)
        if (in_ext(p.row_seq + r, sizeof(int32_t), p.x_ws, p.status)) p.row_seq[r] = b;
    }
  }
}

// A stochastic tile has made its last write (its partial, or its sequence's record): the
// sampler stops waiting for records that are still pending once every tile has counted
// itself (a batch whose offsets failed the prologue's check leaves some unpublished).
template <int MODE>
__device__ __forceinline__ void tile_done(const RowsParams& p) {
  if constexpr (is_stoch(MODE)) red_add_release_gpu(p.cnt + p.B, 1u);
}

// Publishes a sequence record to the sampler, which may already be polling it: the
// payload (with the state still pending), then the state word with release semantics, so a
// reader that acquires the state sees the payload.
__device__ __forceinline__ void publish_rec(SeqRec* dst, SeqRec q) {
  const int state = q.state;
  q.state = REC_PENDING;
  *dst = q;
  st_release_gpu(&dst->state, state);
}

// ---------------------------------------------------------------------------
// policy epilogues

// NKL threshold of draft i of sequence b: delta, or with positions the position-adaptive
// min(dmax, delta * (1 + dalpha * log2(pos))), pos = position[b] + i, 1-based ([CoD] 4.3).
// Negative (every mask 0) when position[b] < 1.
__device__ __forceinline__ float nkl_threshold(const RowsParams& p, int b, int i) {
  if (p.position == nullptr) return p.delta;
  const long long P = (long long)p.position[b];
  if (P < 1) return -1.f;
  return fminf(p.dmax, p.delta * (1.f + p.dalpha * log2f((float)(P + i))));
}

// Block-accept ([CoD] 3.3): the end of the longest run of at least min_block consecutive
// positions whose draft equals the target argmax (the earliest of equally long runs), or
// 0 without one.
template <class RS>
__device__ __forceinline__ int block_end(const int32_t* tok, const RS* rs, int gb, int min_block) {
  int best = 0, start = 0, run = 0;
  for (int i = 0; i < gb; ++i) {
    run = (tok[i] == rs[i].tidx) ? run + 1 : 0;
    if (run > best) {
      best = run;
      start = i - run + 1;
    }
  }
  return best >= min_block ? start + best : 0;
}

// One round of acceptance statistics: n of gamma drafts accepted (gamma > 0). The rates
// are rounded to multiples of 2^-32 so the sums are exact integers.
__device__ __forceinline__ void add_round(spec_stats_slot* st, int n, int gamma) {
  auto* a = reinterpret_cast<unsigned long long*>(st);
  const unsigned long long un = (unsigned long long)n, ug = (unsigned long long)gamma;
  atomicAdd(a + 1, 1ull);
  atomicAdd(a + 2, un);
  atomicAdd(a + 3, ug);
  atomicAdd(a + 4, (((un << 33) / ug) + 1ull) >> 1);
  atomicAdd(a + 5, ((((un * un) << 33) / (ug * ug)) + 1ull) >> 1);
}

// Block-accept outputs and acceptance statistics of a decided sequence (n of gb drafts
// accepted; rs[i].tidx is the target argmax of position i). Called by every thread.
template <class SY, class RS>
__device__ __forceinline__ void policy_epilogue(const RowsParams& p, int b, int gb, int db, int n, const RS* rs) {
  if (p.min_block > 0) {
    __shared__ int s_e;
    if (threadIdx.x == 0) s_e = block_end(p.tokens + db, rs, gb, p.min_block);
    SY::sync();
    const int e = s_e;
    for (int k = threadIdx.x; k < gb; k += SY::NT) p.block_tok[db + k] = (k < e) ? p.tokens[db + k] : rs[k].tidx;
    if (threadIdx.x == 0) p.block_n[b] = e;
  }
  if (p.stats != nullptr && gb > 0 && threadIdx.x == 0) add_round(p.stats, n, gb);
}

// ---------------------------------------------------------------------------
// finalisation, run by the last tile of a sequence

template <typename E, int MODE, class SY>
__device__ __noinline__ void finalize(const RowsParams& p, int b, int gb, int row0, int c0) {
  constexpr int HB = (MODE == M_NKL) ? 0 : 1;
  constexpr int NT = SY::NT, NW = SY::NT / 32;
  __shared__ RowStat rs[kMaxRows];
  __shared__ int s_tok[MODE == M_TREE ? SPEC_MAX_TREE_NODES : 1], s_par[MODE == M_TREE ? SPEC_MAX_TREE_NODES : 1];
  __shared__ int s_n, s_gn;
  __shared__ unsigned s_err;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int R = gb + HB;
  const float c = p.c;
  const size_t V = (size_t)p.V;
  if (tid == 0) {
    s_n = gb;
    s_gn = gb;
    s_err = 0u;
  }
  const int tb = c0 + b * HB;  // first target row of the sequence (NKL: c0 + b, set below)
  const int db = c0;           // first draft row / token / u_accept entry
  const E* target = static_cast<const E*>(p.target);
  const E* draft = static_cast<const E*>(p.draft);
  // Draft position i is owned by thread NT - gb + i (the last warps, while the rows merge
  // from the first): its token and, stochastic, its uniform and z(x) of both rows are read
  // there, the dependent loads of z(x) in flight beside the merge's reads.
  static_assert(NT > SPEC_MAX_GAMMA, "one draft position per thread");
  const int i_own = tid - (NT - gb);  // this thread's draft position, or < 0
  int px = 0;
  float pu = 0.f, pzt = 0.f, pzd = 0.f, pus = 0.f;
  // bounds-checked build: every output of the sequence lies in [tb, tb + gb] of the target-row
  // outputs and [db, db + gb) of the per-draft ones, its records at index b
  if (!in_idx(b, p.B, p.status) || !in_idx(db + gb - 1 + HB, p.total_draft + HB, p.status) ||
      !in_idx(tb + gb - 1 + HB, p.out_rows, p.status))
    return;
  if constexpr (MODE != M_TREE && MODE != M_NKL) {
    if (is_stoch(MODE) && tid == 0) pus = p.u_sample[b];  // for the sampler's record
    if (i_own >= 0) {
      px = p.tokens[db + i_own];
      if constexpr (is_stoch(MODE)) {
        pu = p.u_accept[db + i_own];
        if (px >= 0 && px < p.V) {
          const E* at = target + (size_t)(tb + i_own) * V + px;
          const E* ad = draft + (size_t)(db + i_own) * V + px;
          if (in_ext(at, sizeof(E), p.x_target, p.status)) pzt = elem_at<E>(at, 0);
          if (in_ext(ad, sizeof(E), p.x_draft, p.status)) pzd = elem_at<E>(ad, 0);
        }
      }
    }
  }
  if constexpr (MODE == M_TREE) {
    // the node tokens and parents go to shared memory from the last warps (node j: thread
    // NT - N + j), in flight while the first warps merge the rows
    static_assert(NT >= SPEC_MAX_TREE_NODES, "one node per thread");
    const int j = tid - (NT - p.N);
    if (j >= 0) {
      s_tok[j] = in_idx((long long)b * p.N + j, (long long)p.B * p.N, p.status) ? p.node_tokens[(size_t)b * p.N + j] : -1;
      s_par[j] = p.parent[j];
    }
  }
  // The partial 16-byte blocks at the chunks' ends of stochastic row ii (rows off the grid,
  // or of a length that is not a whole number of blocks), which its tiles left out, for the
  // merge.
  auto edges_of = [&](int ii) {
    constexpr int VEC = 16 / (int)sizeof(E);
    if constexpr (!is_stoch(MODE)) return RowEdges<E>();  // the other modes' tiles fold them
    const int r = row0 + ii;
    const E* trow = target + ((MODE == M_NKL) ? (size_t)r + b : (size_t)r) * V;
    const int ph = (int)(((uintptr_t)trow & 15u) / sizeof(E));
    RowEdges<E> ed;
    if (ph == 0 && p.V % VEC == 0) return ed;  // chunk lengths are whole vectors: none
    const bool pair = (MODE == M_NKL) || (is_stoch(MODE) && ii < gb);
    ed.t = trow;
    ed.d = pair ? draft + ((MODE == M_NKL) ? (size_t)r : (size_t)(r - b)) * V : nullptr;
    ed.ph = ph;
    ed.V = p.V;
    ed.ce = p.chunk_elems;
    ed.sums = MODE != M_GREEDY && MODE != M_TREE;
    ed.sept = MODE == M_STOCH2;
    ed.xt = &p.x_target;
    ed.xd = &p.x_draft;
    ed.status = p.status;
    return ed;
  };
  if (p.nchunks <= 16) {
    // two rows per warp (one per half-warp): one round of partial reads for up to 2 NW rows
    const int half = lane >> 4;
    for (int i = 2 * warp; i < R; i += 2 * NW) {
      const int ii = min(i + half, R - 1);
      const Partial* pr = p.part + (size_t)(row0 + ii) * p.nchunks;
      const bool okp = in_ext(pr, sizeof(Partial) * p.nchunks, p.x_ws, p.status);
      const RowStat r = merge_row<16, E>(okp ? pr : p.part, okp ? p.nchunks : 0, c, p.cd, edges_of(ii));
      if ((lane & 15) == 0 && i + half < R) rs[i + half] = r;
    }
  } else {
    for (int i = warp; i < R; i += NW) {
      const Partial* pr = p.part + (size_t)(row0 + i) * p.nchunks;
      const bool okp = in_ext(pr, sizeof(Partial) * p.nchunks, p.x_ws, p.status);
      const RowStat r = merge_row<32, E>(okp ? pr : p.part, okp ? p.nchunks : 0, c, p.cd, edges_of(i));
      if (lane == 0) rs[i] = r;
    }
  }
  SY::sync();

  if constexpr (MODE == M_TREE) {
    // The first warp decides the (at most 64-node) tree: lane l holds nodes l and l + 32.
    // A node is accepted when its token is its parent row's argmax and its parent is
    // accepted; acceptance and depth settle from the roots down, one shuffle round per
    // level (after round r every node of depth <= r + 1 is final).
    if (warp == 0) {
      const int N = p.N, D = p.depth;
      int32_t* path = p.path_nodes + (size_t)b * D;
      int32_t* out = p.out_tok + (size_t)b * (D + 1);
      int err = 0;
      for (int r = lane; r <= N; r += 32)
        if (rs[r].bad) err |= (int)SPEC_DEV_NONFINITE;
      for (int j = lane; j < N; j += 32) {
        const int x = s_tok[j];
        if (x < 0 || x >= p.V) err |= (int)SPEC_DEV_TOKEN_RANGE;
      }
      err = warp_or<32>(err);
      if (err) {
        if (lane == 0) {
          atomicOr(p.status, (unsigned)err);
          p.accept_len[b] = -1;
        }
        for (int k = lane; k < D; k += 32) path[k] = -1;
        for (int k = lane; k <= D; k += 32) out[k] = -1;
        return;
      }
      int par[2], match[2], acc[2], dep[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int j = lane + 32 * h;
        const bool valid = j < N;
        par[h] = valid ? s_par[j] : -1;
        match[h] = valid && s_tok[j] == rs[par[h] < 0 ? 0 : par[h] + 1].tidx;
        acc[h] = match[h] && par[h] < 0;
        dep[h] = valid ? 1 : 0;
      }
      for (int it = 1; it < D; ++it) {
        const int a0 = acc[0], a1 = acc[1], d0 = dep[0], d1 = dep[1];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int q = par[h] < 0 ? 0 : par[h];
          const int sa0 = __shfl_sync(kFull, a0, q & 31), sa1 = __shfl_sync(kFull, a1, q & 31);
          const int sd0 = __shfl_sync(kFull, d0, q & 31), sd1 = __shfl_sync(kFull, d1, q & 31);
          if (par[h] >= 0) {
            acc[h] = match[h] && ((q >> 5) ? sa1 : sa0);
            dep[h] = ((q >> 5) ? sd1 : sd0) + 1;
          }
        }
      }
      // the deepest accepted node, ties to the lowest index: the largest (depth, -node)
      int key = -1;
#pragma unroll
      for (int h = 0; h < 2; ++h)
        if (acc[h]) key = max(key, (dep[h] << 7) | (127 - (lane + 32 * h)));
      key = __reduce_max_sync(kFull, key);
      const int best = key >= 0 ? key >> 7 : 0, pick = key >= 0 ? 127 - (key & 127) : -1;
      for (int d = best + lane; d < D; d += 32) path[d] = -1;
      for (int d = best + 1 + lane; d <= D; d += 32) out[d] = -1;
      if (lane == 0) {
        p.accept_len[b] = best;
        int k = pick;
        for (int d = best - 1; d >= 0; --d) {
          path[d] = k;
          out[d] = s_tok[k];
          k = s_par[k];
        }
        out[best] = rs[pick + 1].tidx;  // pick == -1 gives row 0
      }
    }
    return;
  } else if constexpr (MODE == M_NKL) {
    const int tbn = c0 + b;
    for (int i = tid; i < gb; i += NT) {
      const RowStat r = rs[i];
      float v = __int_as_float(0x7fc00000);
      uint8_t m = 0;
      if (r.bad) {
        atomicOr(p.status, SPEC_DEV_NONFINITE);
      } else {
        v = row_nkl(r, p.invT, p.inv_lnV);
        m = v < nkl_threshold(p, b, i) ? 1 : 0;
      }
      p.nkl[db + i] = v;
      if (p.mask) p.mask[db + i] = m;
    }
    if (tid == 0 && p.position != nullptr && p.position[b] < 1) atomicOr(p.status, SPEC_DEV_POSITION);
    (void)tbn;
    return;
  } else {
  // stochastic and greedy: validate the sequence first
  {
    unsigned e = (tid < R && rs[tid].bad) ? SPEC_DEV_NONFINITE : 0u;  // R <= SPEC_MAX_GAMMA + 1 <= NT
    if (i_own >= 0 && (px < 0 || px >= p.V)) e |= SPEC_DEV_TOKEN_RANGE;
    if (e) atomicOr(&s_err, e);
  }
  SY::sync();
  if (s_err) {
    if (tid == 0) atomicOr(p.status, s_err);
    for (int k = tid; k <= gb; k += NT) {
      p.out_tok[tb + k] = -1;
      if (is_stoch(MODE) && p.g_tok) p.g_tok[tb + k] = -1;
      if (p.block_tok != nullptr && k < gb) p.block_tok[db + k] = -1;
      if (is_stoch(MODE) && k < gb) {
        const float qnan = __int_as_float(0x7fc00000);
        if (p.p_x) p.p_x[db + k] = qnan;
        if (p.q_x) p.q_x[db + k] = qnan;
        if (p.alpha) p.alpha[db + k] = qnan;
        if (p.nkl) p.nkl[db + k] = qnan;
        if (p.mask) p.mask[db + k] = 0;
      }
    }
    if (tid == 0) {
      p.n_acc[b] = -1;
      if (p.block_n != nullptr) p.block_n[b] = -1;
      if (is_stoch(MODE)) {
        if (p.g_n) p.g_n[b] = -1;
        SeqRec q;
        q.state = REC_SKIP;
        q.n = -1;
        q.t_row = q.d_row = -1;
        q.lt2 = q.ld2 = q.us = 0.f;
        q.mode = 0;
        publish_rec(p.rec + b, q);
      }
    }
    return;
  }

  if constexpr (MODE == M_GREEDY) {
    if (i_own >= 0 && px != rs[i_own].tidx) atomicMin(&s_gn, i_own);
    SY::sync();
    const int n = s_gn;
    if (i_own >= 0) p.out_tok[tb + i_own] = (i_own < n) ? px : (i_own == n ? rs[n].tidx : -1);
    if (tid == 0) {
      p.out_tok[tb + gb] = (n == gb) ? rs[gb].tidx : -1;  // the bonus position
      p.n_acc[b] = n;
    }
    policy_epilogue<SY>(p, b, gb, db, n, rs);
    return;
  } else {
  // stochastic
  float lp2 = 0.f, lq2 = 0.f, a = 0.f;
  if (i_own >= 0) {
    const RowStat& r = rs[i_own];
    lp2 = (pzt - r.tm) * c - log2f(r.ts);     // log2 p(x)
    lq2 = (pzd - r.dm) * p.cd - log2f(r.ds);  // log2 q(x), at the draft's temperature
    a = exp2f(fminf(0.f, lp2 - lq2));
    if (!(pu <= a)) atomicMin(&s_n, i_own);
    if (px != r.tidx) atomicMin(&s_gn, i_own);
  }
  SY::sync();
  const int n = s_n, gn = s_gn;
  if (tid == 0) {
    // the sampler waits on this record: published before any other output of the sequence,
    // so that the fence orders only the record's payload
    SeqRec q;
    q.state = REC_READY;
    q.n = n;
    q.t_row = tb + n;
    q.d_row = (n < gb) ? db + n : -1;
    q.lt2 = rs[n].tm * c + log2f(rs[n].ts);
    q.ld2 = (n < gb) ? rs[n].dm * p.cd + log2f(rs[n].ds) : 0.f;
    q.us = pus;
    q.mode = (n < gb) ? S_RESID : S_P;
    publish_rec(p.rec + b, q);
  }
  if (i_own >= 0) {
    const int i = i_own;
    if (p.p_x) p.p_x[db + i] = exp2f(lp2);
    if (p.q_x) p.q_x[db + i] = exp2f(lq2);
    if (p.alpha) p.alpha[db + i] = a;
    if (p.nkl || p.mask) {
      const float v = row_nkl<MODE == M_STOCH2>(rs[i], p.invT, p.inv_lnV);  // both rows at the target's T
      if (p.nkl) p.nkl[db + i] = v;
      if (p.mask) p.mask[db + i] = v < nkl_threshold(p, b, i) ? 1 : 0;
    }
  }
  if (i_own >= 0) {
    const int k = i_own;
    if (k != n) p.out_tok[tb + k] = (k < n) ? px : -1;
    if (p.g_tok) p.g_tok[tb + k] = (k < gn) ? px : (k == gn ? rs[gn].tidx : -1);
  }
  if (tid == 0) {
    // the bonus position: the sampler's token when every draft is accepted
    if (n != gb) p.out_tok[tb + gb] = -1;
    if (p.g_tok) p.g_tok[tb + gb] = (gn == gb) ? rs[gb].tidx : -1;
    p.n_acc[b] = n;
    if (p.g_n) p.g_n[b] = gn;
    if (p.mask && p.position != nullptr && p.position[b] < 1) atomicOr(p.status, SPEC_DEV_POSITION);
  }
  policy_epilogue<SY>(p, b, gb, db, n, rs);
  }  // stochastic
  }  // stochastic and greedy
}

// ---------------------------------------------------------------------------
// tile kernel

// Two vectors of a stage as one 2*VEC-element group (va < vb, element bases va*VEC, vb*VEC).
template <typename E, int VEC>
__device__ __forceinline__ void unpack2(const uint4& a, const uint4& b, float (&f)[2 * VEC]) {
  float fa[VEC], fb[VEC];
  IO<E, VEC>::unpack(a, fa);
  IO<E, VEC>::unpack(b, fb);
#pragma unroll
  for (int k = 0; k < VEC; ++k) {
    f[k] = fa[k];
    f[VEC + k] = fb[k];
  }
}

// Vector path: every thread streams its own vectors through a private kCS-stage ring of
// cp.async copies in shared memory (lane-interleaved, so both the copies and the reads
// are bank-conflict free), waiting with cp.async.wait_group only -- no barriers, no
// registers held by loads in flight. A stage is kCV vectors per thread: for a pair the
// vectors v and v + 256 of the target and of the draft row, for a single row the vectors
// v, v + 256, v + 512, v + 768; each pair of vectors is folded in as one group.
// Argmax rows (KIND == K_ARGMAX) also keep, in `best`, the raw vectors of the group that
// holds the thread's maximum, so the tile end resolves its lowest index without
// re-reading the row.
// rot (0..7): vector v0 lies rot vectors past the start of its 128-byte line. Each stage's
// 256-vector block is then assigned rotated by rot (thread t takes offset (t - rot) mod 256),
// so that every warp but the first copies four whole lines instead of spreading its 32
// vectors over five.
template <typename E, int VEC, int MODE, int KIND>
__device__ __forceinline__ void stream_tile(const E* trow, const E* drow, int v0, int v1, int rot, float c, float cd,
                                            TAcc& ta, DAcc& da, unsigned char* smem, uint4 (&best)[2],
                                            const RowsParams& p) {
  constexpr bool IDX = is_stoch(MODE), SEPT = MODE == M_STOCH2;
  constexpr int PER = (KIND == K_PAIR) ? 2 * kThreads : 4 * kThreads;  // vectors of a row per stage
  constexpr unsigned SLOT = kCV * kThreads * 16;                         // bytes of one stage
  const int t = threadIdx.x;
  const uint32_t base = (uint32_t)__cvta_generic_to_shared(smem) + 16u * t;
  const int nst = (v1 - v0 + PER - 1) / PER;
  const int vt = v0 + ((t - rot) & (kThreads - 1));  // this thread's first vector in stage 0
  const E* tp = trow + (size_t)vt * VEC;
  const E* dp = drow + (size_t)vt * VEC;
  auto issue = [&](int k) {
    if (k < nst) {
      const uint32_t slot = base + (uint32_t)(k % kCS) * SLOT;
      const int v = vt + k * PER;
      const size_t off = (size_t)k * PER * VEC;
#pragma unroll
      for (int j = 0; j < kCV; ++j) {
        const int jv = (KIND == K_PAIR) ? (j & 1) : j;
        if (v + jv * kThreads < v1) {
          const E* src = ((KIND == K_PAIR && j >= 2) ? dp : tp) + off + (size_t)jv * kThreads * VEC;
          if (in_ext(src, 16, (KIND == K_PAIR && j >= 2) ? p.x_draft : p.x_target, p.status))
            cp_async16(slot + (uint32_t)(j * kThreads * 16), src);
        }
      }
    }
    cp_commit();
  };
#pragma unroll
  for (int k = 0; k < kCS - 1; ++k) issue(k);
  for (int k = 0; k < nst; ++k) {
    issue(k + kCS - 1);
    cp_wait<kCS - 1>();
    const uint4* q = reinterpret_cast<const uint4*>(smem + (size_t)(k % kCS) * SLOT) + t;
    const int va = vt + k * PER;
    if constexpr (KIND == K_PAIR) {
      const int vb = va + kThreads;
      if (vb < v1) {
        float ft[2 * VEC], fd[2 * VEC];
        unpack2<E, VEC>(q[0], q[kThreads], ft);
        unpack2<E, VEC>(q[2 * kThreads], q[3 * kThreads], fd);
        pair_update<2 * VEC, IDX, VEC, SEPT>(ta, da, ft, fd, va * VEC, c, cd);
      } else if (va < v1) {
        float ft[VEC], fd[VEC];
        IO<E, VEC>::unpack(q[0], ft);
        IO<E, VEC>::unpack(q[2 * kThreads], fd);
        pair_update<VEC, IDX, VEC, SEPT>(ta, da, ft, fd, va * VEC, c, cd);
      }
    } else {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int pa = va + 2 * h * kThreads, pb = pa + kThreads;
        if (pb < v1) {
          float ft[2 * VEC];
          const uint4 r0 = q[(2 * h) * kThreads], r1 = q[(2 * h + 1) * kThreads];
          unpack2<E, VEC>(r0, r1, ft);
          if constexpr (KIND == K_TSUM) {
            tsum_update<2 * VEC, VEC>(ta, ft, pa * VEC, c);
          } else {
            if (vmax_nan<2 * VEC>(ft) > ta.m) {
              best[0] = r0;
              best[1] = r1;
            }
            argmax_update<2 * VEC, VEC>(ta, ft, pa * VEC);
          }
        } else if (pa < v1) {
          float ft[VEC];
          const uint4 r0 = q[(2 * h) * kThreads];
          IO<E, VEC>::unpack(r0, ft);
          if constexpr (KIND == K_TSUM) {
            tsum_update<VEC>(ta, ft, pa * VEC, c);
          } else {
            if (vmax_nan<VEC>(ft) > ta.m) best[0] = best[1] = r0;  // a one-vector group: its first VEC
            argmax_update<VEC>(ta, ft, pa * VEC);
          }
        }
      }
    }
  }
  cp_wait<0>();
}

// Row pairs whose two rows sit at different offsets within the 16-byte grid (a vocabulary
// whose row is not a whole number of 16-byte blocks): the stream of stream_tile over the
// target's aligned vectors v in [v0, v1), and for each the draft's elements at the same
// row indices, which lie in the draft's aligned vectors w = v + dw and w + 1, shifted by S
// elements (dw * VEC + S = the draft's offset minus the target's, 0 < S < VEC; M whole
// words and the half-word permutation sel). Each lane
// copies its own w; after a warp barrier it takes w + 1 from the next lane's slot, and lane
// 31 copies its w + 1 itself into a small ring of its own (kShiftXSlot bytes per stage
// after the main ring). Lanes one vector past the end still copy their draft vector (the
// lane before needs it as its w + 1): it holds the last element of the last whole target
// vector, so it lies in the row. Two warp barriers per stage: before a slot is refilled
// (every lane has read it) and after the copies land (they are visible to the warp).
template <typename E, int VEC, int MODE, int M>
__device__ __forceinline__ void stream_tile_sh(const E* trv, const E* drv, int v0, int v1, int dw, unsigned sel,
                                               float c, float cd, TAcc& ta, DAcc& da, unsigned char* smem,
                                               const RowsParams& p) {
  constexpr bool IDX = is_stoch(MODE), SEPT = MODE == M_STOCH2;
  constexpr int PER = 2 * kThreads;            // vectors of a row per stage
  constexpr unsigned SLOT = kCV * kThreads * 16;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const uint32_t base = (uint32_t)__cvta_generic_to_shared(smem) + 16u * t;
  unsigned char* xring = smem + kCS * SLOT;
  const uint32_t xbase = (uint32_t)__cvta_generic_to_shared(xring) + (uint32_t)(warp * 32);
  const int nst = (v1 - v0 + PER - 1) / PER;
  const int vt = v0 + t;
  const E* tp = trv + (size_t)vt * VEC;
  const E* dp = drv + (ptrdiff_t)(vt + dw) * VEC;
  auto issue = [&](int k) {
    if (k < nst) {
      const uint32_t slot = base + (uint32_t)(k % kCS) * SLOT;
      const uint32_t xs = xbase + (uint32_t)(k % kCS) * kShiftXSlot;
      const int v = vt + k * PER;
      const size_t off = (size_t)k * PER * VEC;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int vh = v + h * kThreads;
        const size_t o = off + (size_t)h * kThreads * VEC;
        if (vh < v1 && in_ext(tp + o, 16, p.x_target, p.status)) cp_async16(slot + (uint32_t)(h * kThreads * 16), tp + o);
        if (vh <= v1 && in_ext(dp + o, 16, p.x_draft, p.status))
          cp_async16(slot + (uint32_t)((2 + h) * kThreads * 16), dp + o);
        if (lane == 31 && vh < v1 && in_ext(dp + o + VEC, 16, p.x_draft, p.status)) cp_async16(xs + 16u * h, dp + o + VEC);
      }
    }
    cp_commit();
  };
#pragma unroll
  for (int k = 0; k < kCS - 1; ++k) issue(k);
  for (int k = 0; k < nst; ++k) {
    __syncwarp();  // every lane has read the slot issue() refills (stage k - 1)
    issue(k + kCS - 1);
    cp_wait<kCS - 1>();
    __syncwarp();  // the lanes' copies of stage k are visible to the whole warp
    const uint4* q = reinterpret_cast<const uint4*>(smem + (size_t)(k % kCS) * SLOT) + t;
    const uint4* qx = reinterpret_cast<const uint4*>(xring + (size_t)(k % kCS) * kShiftXSlot) + warp * 2;
    const int va = vt + k * PER, vb = va + kThreads;
    if (MODE == M_NKL && vb < v1) {
      // NKL: both vectors of each row as one 2·VEC group, as the aligned tiles do
      float ft[2 * VEC], fd[2 * VEC];
      unpack2<E, VEC>(q[0], q[kThreads], ft);
      const uint4 n0 = lane < 31 ? q[2 * kThreads + 1] : qx[0];
      const uint4 n1 = lane < 31 ? q[3 * kThreads + 1] : qx[1];
      unpack2<E, VEC>(shift_vec<E, M>(q[2 * kThreads], n0, sel), shift_vec<E, M>(q[3 * kThreads], n1, sel), fd);
      pair_update<2 * VEC, IDX, VEC, SEPT>(ta, da, ft, fd, va * VEC, c, cd);
      continue;
    }
    // stochastic rows (and the NKL tile's last odd vector): one vector of each row at a time,
    // groups of VEC elements -- the argmax index and the shift's registers on top of a
    // two-vector group spilled at the 64-register limit
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int v = va + h * kThreads;
      if (v < v1) {
        float ft[VEC], fd[VEC];
        IO<E, VEC>::unpack(q[h * kThreads], ft);
        const uint4 n = lane < 31 ? q[(2 + h) * kThreads + 1] : qx[h];
        IO<E, VEC>::unpack(shift_vec<E, M>(q[(2 + h) * kThreads], n, sel), fd);
        pair_update<VEC, IDX, VEC, SEPT>(ta, da, ft, fd, v * VEC, c, cd);
      }
    }
  }
  cp_wait<0>();
}

// The shifted stream for the tile's shift s (0 < s < VEC): one instance per whole-word part
// of the shift (four for bf16, three for fp32), the half word a uniform runtime selector.
template <typename E, int VEC, int MODE>
__device__ __forceinline__ void stream_tile_shifted(int s, const E* trv, const E* drv, int v0, int v1, int dw, float c,
                                                    float cd, TAcc& ta, DAcc& da, unsigned char* smem,
                                                    const RowsParams& p) {
  if constexpr (VEC == 8) {
    const unsigned sel = (s & 1) ? 0x5432u : 0x3210u;
    switch (s >> 1) {
      case 0: stream_tile_sh<E, VEC, MODE, 0>(trv, drv, v0, v1, dw, sel, c, cd, ta, da, smem, p); break;
      case 1: stream_tile_sh<E, VEC, MODE, 1>(trv, drv, v0, v1, dw, sel, c, cd, ta, da, smem, p); break;
      case 2: stream_tile_sh<E, VEC, MODE, 2>(trv, drv, v0, v1, dw, sel, c, cd, ta, da, smem, p); break;
      default: stream_tile_sh<E, VEC, MODE, 3>(trv, drv, v0, v1, dw, sel, c, cd, ta, da, smem, p); break;
    }
  } else {
    switch (s) {
      case 1: stream_tile_sh<E, VEC, MODE, 1>(trv, drv, v0, v1, dw, 0u, c, cd, ta, da, smem, p); break;
      case 2: stream_tile_sh<E, VEC, MODE, 2>(trv, drv, v0, v1, dw, 0u, c, cd, ta, da, smem, p); break;
      default: stream_tile_sh<E, VEC, MODE, 3>(trv, drv, v0, v1, dw, 0u, c, cd, ta, da, smem, p); break;
    }
  }
}

// PH: rows at any element alignment, each tile applying its row's phase (the rows of a
// pair at one phase). SH (with PH): the rows of a pair may sit at different phases; a pair
// tile whose draft row is off its target row's phase takes the shifted stream.
template <typename E, int VEC, int MODE, bool PH = false, bool SH = false>
__global__ void __launch_bounds__(kThreads, 4) rows_kernel(const __grid_constant__ RowsParams p) {
  constexpr int HB = (MODE == M_NKL) ? 0 : 1;
  extern __shared__ __align__(128) unsigned char dsm[];
  // Nothing is read or written before the prologue -- and with it everything earlier on
  // the stream -- has completed. The stochastic sampler polls the per-sequence records
  // instead of waiting for this grid; it launches once every block has passed the
  // trigger, so after the prologue has re-armed the records.
  griddep_wait();
  griddep_launch();
  __shared__ int s_last;
  const int tile = blockIdx.x;
  const int r = tile / p.nchunks;
  const int chunk = tile - r * p.nchunks;
  int b, i, gb, c0;
  if (p.cu == nullptr) {
    const int R = p.gamma + HB;
    b = r / R;
    i = r - b * R;
    gb = p.gamma;
    c0 = b * p.gamma;
  } else {
    // the sequence owning row r, from the prologue's table (written before this grid's
    // griddepcontrol.wait returned); checked against the offsets below
    b = in_ext(p.row_seq + r, sizeof(int32_t), p.x_ws, p.status) ? __ldcg(p.row_seq + r) : -1;
    if (b < 0 || b >= p.B) {
      if (threadIdx.x == 0) {
        atomicOr(p.status, SPEC_DEV_OFFSETS);
        tile_done<MODE>(p);
      }
      return;
    }
    c0 = __ldg(p.cu + b);
    const int c1 = __ldg(p.cu + b + 1);
    gb = c1 - c0;
    i = r - (c0 + HB * b);
    if (gb < 0 || gb > p.gamma || c0 < 0 || c1 > p.total_draft || i < 0 || i >= gb + HB) {
      if (threadIdx.x == 0) {
        atomicOr(p.status, SPEC_DEV_OFFSETS);
        tile_done<MODE>(p);
      }
      return;
    }
  }
  const int kind = (MODE == M_NKL) ? K_PAIR : (is_stoch(MODE) ? (i < gb ? K_PAIR : K_TSUM) : K_ARGMAX);
  constexpr bool IDX = is_stoch(MODE), SEPT = MODE == M_STOCH2;
  const size_t V = (size_t)p.V;
  const size_t trow_i = (MODE == M_NKL) ? (size_t)r + b : (size_t)r;
  const size_t drow_i = (MODE == M_NKL) ? (size_t)r : (size_t)(r - b);
  const E* trow = static_cast<const E*>(p.target) + trow_i * V;
  const E* drow = static_cast<const E*>(p.draft) + ((kind == K_PAIR) ? drow_i * V : 0);
  const int e_begin = chunk * p.chunk_elems;
  const int e_end = min(e_begin + p.chunk_elems, p.V);
  // the draft's scale: the NKL call's is the target's (so the compiler keeps one register)
  const float c = p.c, cd = (MODE == M_NKL) ? p.c : p.cd;

  TAcc ta;
  DAcc da;
  init(ta);
  init(da);
  constexpr bool ARGMAX = MODE == M_GREEDY || MODE == M_TREE;
  static_assert(VEC > 1, "tiles stream 16-byte vectors");
  static_assert(!SH || (PH && !ARGMAX), "shifted pairs are phased pair tiles");
  // PH: the row's offset in elements within the 16-byte grid; indices are counted from the
  // aligned base until the partial is written
  {
    int ph = 0;
    uint4 best[2];
    // Rows at any element alignment (PH): the whole aligned 16-byte blocks of the chunk are
    // streamed as vectors of the aligned bases trv and drv (row element e is element
    // e + ph of trv, e + phd of drv). The elements of the partial blocks at the chunk's
    // ends: stochastic rows leave them to the row's merge in the finalisation (RowEdges),
    // so that their tiles carry no code for them (measured: the headline batch one element
    // off the grid, 192.1 -> 185.0 us); NKL, greedy and tree tiles fold them themselves
    // (TE), which measured faster for them (NKL 150.7 against 155.6 us).
    constexpr bool TE = PH && !is_stoch(MODE);
    if constexpr (PH) ph = (int)(((uintptr_t)trow & 15u) / sizeof(E));
    const int phd = (PH && kind == K_PAIR) ? (int)(((uintptr_t)drow & 15u) / sizeof(E)) : ph;
    const E* trv = trow - ph;
    const E* drv = drow - phd;
    // shifted pairs: the draft elements of target vector v lie in draft vectors v + dw and
    // v + dw + 1, from element sft on
    const int sft = (phd - ph + VEC) % VEC, dw = (phd - ph - sft) / VEC;
    const int vf0 = (e_begin + ph + VEC - 1) / VEC, vf1 = (e_end + ph) / VEC;
    // vectors between the start of vf0's 128-byte line and vf0 (the streams' rotation)
    const int rot = (int)((reinterpret_cast<uintptr_t>(trv + (size_t)vf0 * VEC) >> 4) & 7u);
    // TE: the partial blocks at the chunk's ends, head [e_begin, hend) and tail [tbeg, e_end),
    // fewer than VEC elements each: element j of the head is edge thread j's, element j of
    // the tail edge thread VEC + j's -- the block's last 2·VEC threads, whose share of a
    // tile's last stage is the smallest. Each copies the target block and the draft block
    // holding its element beside the ring and folds the element in after the stream. What
    // the fold needs -- the element's index from the aligned base and its draft position --
    // goes to shared memory beside the blocks, so that nothing of it is held in registers
    // through the stream.
    __shared__ uint4 s_edge[TE ? 2 * VEC : 1][2];  // [edge thread][target, draft]
    __shared__ int s_eidx[TE ? 2 * VEC : 1][2];    // [edge thread][e + ph or -1, (e + phd) % VEC]
    const int et = (int)threadIdx.x - (kThreads - 2 * VEC);  // edge thread index, if >= 0
    if (TE && et >= 0) {
      const int side = et / VEC;
      const int hend = min(e_end, vf0 * VEC - ph), tbeg = max(hend, vf1 * VEC - ph);
      int e = (side == 0 ? e_begin : tbeg) + et % VEC;
      if (e >= (side == 0 ? hend : e_end)) e = -1;
      s_eidx[et][0] = e >= 0 ? e + ph : -1;
      s_eidx[et][1] = (e + phd) % VEC;
      if (e >= 0) {
        const size_t tb = (size_t)((e + ph) / VEC) * VEC, db = (size_t)((e + phd) / VEC) * VEC;
        if (in_ext(trv + tb, 16, p.x_target, p.status))
          cp_async16((uint32_t)__cvta_generic_to_shared(&s_edge[et][0]), trv + tb);
        if (kind == K_PAIR && in_ext(drv + db, 16, p.x_draft, p.status))
          cp_async16((uint32_t)__cvta_generic_to_shared(&s_edge[et][1]), drv + db);
      }
    }
    // (the stream's last wait covers the edge copies too)
    if constexpr (ARGMAX) {
      stream_tile<E, VEC, MODE, K_ARGMAX>(trv, drv, vf0, vf1, rot, c, cd, ta, da, dsm, best, p);
      // the lowest index of the thread's maximum, from the raw vectors of its group
      if (ta.g0 >= 0) {
        float f[2 * VEC];
        unpack2<E, VEC>(best[0], best[1], f);
        int k = 2 * VEC - 1;
#pragma unroll
        for (int j = 2 * VEC - 2; j >= 0; --j)
          if (f[j] == ta.m) k = j;
        const int g = ta.g0 & ~1;  // the group's first vector; its second is kThreads vectors on
        ta.g0 = k < VEC ? g + k : g + kThreads * VEC + (k - VEC);
      }
    } else {
      if (kind == K_PAIR) {
        if (SH && sft != 0)
          stream_tile_shifted<E, VEC, MODE>(sft, trv, drv, vf0, vf1, dw, c, cd, ta, da, dsm, p);
        else
          stream_tile<E, VEC, MODE, K_PAIR>(trv, drv, vf0, vf1, rot, c, cd, ta, da, dsm, best, p);
      } else if constexpr (MODE != M_NKL) {
        stream_tile<E, VEC, MODE, K_TSUM>(trv, drv, vf0, vf1, rot, c, cd, ta, da, dsm, best, p);
      }
    }
    // (the thread's own shared-memory entries: no barrier needed)
    const int ea = (TE && et >= 0) ? s_eidx[et][0] : -1;  // e + ph
    if (ea >= 0) {
      const float x = sh_elem<E>(reinterpret_cast<const E*>(&s_edge[et][0]), ea % VEC);
      if constexpr (ARGMAX) {
        ta.hi = max_nan(ta.hi, x);
        ta.lo = fminf(ta.lo, x);
      } else {
        // the sums; the maximum and its index are kept apart (the recorded group stays
        // the one that holds the thread's maximum over whole vectors)
        const float m0 = ta.m;
        const int g0 = ta.g0;
        const float xt[1] = {x};
        const float xd[1] = {sh_elem<E>(reinterpret_cast<const E*>(&s_edge[et][1]), s_eidx[et][1])};
        pair_update<1, false, 0, SEPT>(ta, da, xt, xd, 0, c, cd);  // NKL: pairs only
        ta.m = m0;
        ta.g0 = g0;
      }
      // an edge element holding the thread's maximum carries its exact index (a head
      // element precedes every whole vector of the chunk: it wins ties)
      if (x > ta.m || (x == ta.m && ta.g0 >= 0 && ea < ta.g0)) {
        ta.m = x;
        ta.g0 = ARGMAX ? ea : exact_idx(ea);  // argmax rows hold resolved indices already
      }
    }
  }

  // the row's offset again (recomputed rather than held through the stream)
  const int ph2 = PH ? (int)(((uintptr_t)trow & 15u) / sizeof(E)) : 0;
  Partial part = reduce_tile<BlockSync, E, VEC, SEPT, ARGMAX>(kind, ta, da, c, trow - ph2, cd, &p.x_target, p.status);
  if constexpr (PH) {
    if (part.tidx != INT_MAX) part.tidx -= ph2;  // from the aligned base to the row
    // stochastic rows: a chunk without a whole block streamed nothing; its statistics are
    // empty, not non-finite (its elements are the merge's)
    if (is_stoch(MODE) && (e_end + ph2) / VEC <= (e_begin + ph2 + VEC - 1) / VEC) part.bad = 0;
  }
  if (threadIdx.x == 0) {
    float4* dst = reinterpret_cast<float4*>(p.part + tile);
    const bool okw = in_ext(dst, sizeof(Partial), p.x_ws, p.status) && in_ext(p.cnt + b, sizeof(unsigned), p.x_ws, p.status);
    if (okw) {
      __stcg(dst, make_float4(part.tm, part.ts, __int_as_float(part.tidx), __int_as_float(part.bad)));
      __stcg(dst + 1, make_float4(part.dm, part.ds, part.dk, part.ds2));
    }
    const unsigned total = (unsigned)((gb + HB) * p.nchunks);
    // release: this tile's partial before its ticket; acquire: the other tiles' partials
    // (read with ld.cg) before this block's reads
    const unsigned old = okw ? atom_add_acq_rel_gpu(p.cnt + b, 1u) : 0u;
    s_last = (okw && old + 1u == total) ? 1 : 0;
  }
  __syncthreads();
  if (!s_last) {
    if (threadIdx.x == 0) tile_done<MODE>(p);
    return;
  }
  finalize<E, MODE, BlockSync>(p, b, gb, r - i, c0);
  if constexpr (is_stoch(MODE)) {
    __syncthreads();  // the finaliser's writes, made by any thread, precede the count
    if (threadIdx.x == 0) tile_done<MODE>(p);
  }
}

// ---------------------------------------------------------------------------
// acceptance statistics summary: one thread per slot, then thread 0 combines the slots of
// the window (integer sums, so the order does not matter)

__global__ void __launch_bounds__(SPEC_STATS_SLOTS) summary_kernel(const spec_accept_stats* st, long long now,
                                                                  int window, double* out) {
  griddep_wait();  // the calls it summarises have completed
  __shared__ unsigned long long s[5][SPEC_STATS_SLOTS];
  const int t = threadIdx.x;
  const spec_stats_slot sl = st->slot[t];
  const bool in = sl.bucket > now - window && sl.bucket <= now;
  s[0][t] = in ? sl.rounds : 0ull;
  s[1][t] = in ? sl.accepted : 0ull;
  s[2][t] = in ? sl.drafted : 0ull;
  s[3][t] = in ? sl.rate_fx : 0ull;
  s[4][t] = in ? sl.rate2_fx : 0ull;
  __syncthreads();
  if (t == 0) {
    unsigned long long a[5] = {0ull, 0ull, 0ull, 0ull, 0ull};
    for (int k = 0; k < SPEC_STATS_SLOTS; ++k)
      for (int j = 0; j < 5; ++j) a[j] += s[j][k];
    const double R = (double)a[0];
    double mean_acc = 0.0, mean_rate = 0.0, arsd = 0.0;
    if (a[0] > 0) {
      const double unit = 1.0 / 4294967296.0;  // 2^-32
      mean_acc = (double)a[1] / R;
      mean_rate = (double)a[3] * unit / R;
      const double var = (double)a[4] * unit / R - mean_rate * mean_rate;
      arsd = var > 0.0 ? sqrt(var) : 0.0;
    }
    out[0] = R;
    out[1] = (double)a[1];
    out[2] = (double)a[2];
    out[3] = mean_acc;
    out[4] = mean_rate;
    out[5] = arsd;
  }
}

}  // namespace sv
