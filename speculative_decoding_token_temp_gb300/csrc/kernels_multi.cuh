// Multi-draft verification: the pairwise NKL matrix of K candidate drafts per position
// and the choice of the longest accepted candidate.
//
// A group holds K candidate sequences (sequence g*K + k of a dense batch, gamma drafts
// each), verified by the batch kernels like any other sequences. pair_kernel reads, for
// every (group, draft position, vocabulary chunk) tile, the K candidates' draft rows of
// that position together and accumulates per row a its reference and
// S_a = sum_v exp2((z_a,v - ref_a) * c), and per ordered pair (a, b)
// K_ab = sum_v exp2((z_a,v - ref_a) * c) (z_a,v - z_b,v). The last tile of a position
// (atomic ticket) merges the chunks and writes
// M[a][b] = KL(q_a || q_b) / ln V = ((K_ab / S_a - (ref_a - ref_b)) / T - ln(S_a / S_b)) / ln V
// with the consensus (some pair below c_thr both ways) and divergence (every entry above
// d_thr) flags. select_kernel keeps, per group, the candidate with the most accepted
// drafts (the lowest index among equals) and copies its tokens.
#pragma once

#include "kernels_rows.cuh"

namespace sv {

constexpr int kMaxCand = SPEC_MAX_CANDIDATES;

// per-tile partial: references, sums, ordered-pair KL sums (diagonal unused)
struct __align__(16) PairPartial {
  float ref[kMaxCand];
  float s[kMaxCand];
  float k[kMaxCand * kMaxCand];
};

struct PairParams {
  const void* draft;
  int V, gamma, K, G, nchunks, chunk_elems;
  float c, invT, inv_lnV, c_thr, d_thr;
  PairPartial* part;
  unsigned* cnt;  // [G * gamma] tickets, zeroed by the prologue
  float* pair_nkl;
  uint8_t* cons;
  uint8_t* div;
  uint32_t* status;
  Ext x_draft, x_ws;  // the draft rows and the workspace (bounds-checked build)
};

// The last tile of a (group, position): merge the chunks' partials (thread (a, j) owns
// S_a for j == K, else K_aj), then the K x K matrix and the flags. Every thread calls it.
template <int K>
__device__ __forceinline__ void pair_merge(const PairParams& p, int gi) {
  __shared__ float s_M[K], s_S[K], s_K[K * K], s_N[K * K];
  const float c = p.c;
  const PairPartial* pp = p.part + (size_t)gi * p.nchunks;
  if (!in_ext(pp, sizeof(PairPartial) * p.nchunks, p.x_ws, p.status) ||
      !in_idx((long long)gi, (long long)p.G * p.gamma, p.status))
    return;  // (every thread: the condition is uniform)
  if (threadIdx.x < K * (K + 1)) {
    const int a = threadIdx.x / (K + 1), j = threadIdx.x - a * (K + 1);
    float M = -INFINITY;
    for (int ch = 0; ch < p.nchunks; ++ch) M = fmaxf(M, __ldcg(&pp[ch].ref[a]));
    float t = 0.f;
    for (int ch = 0; ch < p.nchunks; ++ch) {
      const float r = __ldcg(&pp[ch].ref[a]);
      const float f = (r == -INFINITY) ? 0.f : ex2((r - M) * c);
      t += f * (j == K ? __ldcg(&pp[ch].s[a]) : __ldcg(&pp[ch].k[a * K + j]));
    }
    if (j == K) {
      s_S[a] = t;
      s_M[a] = M;
    } else {
      s_K[a * K + j] = t;
    }
  }
  __syncthreads();
  if (threadIdx.x < K * K) {
    const int a = threadIdx.x / K, b = threadIdx.x - a * K;
    float n = 0.f;
    if (a != b) {
      const float kl = (s_K[a * K + b] / s_S[a] - (s_M[a] - s_M[b])) * p.invT - logf(s_S[a] / s_S[b]);
      n = isfinite(kl) ? kl * p.inv_lnV : __int_as_float(0x7fc00000);
    }
    s_N[threadIdx.x] = n;
    if (p.pair_nkl) p.pair_nkl[(size_t)gi * K * K + threadIdx.x] = n;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    bool cons = false, div = true, bad = false;
    for (int a = 0; a < K; ++a)
      for (int b = 0; b < K; ++b) {
        if (a == b) continue;
        const float ab = s_N[a * K + b], ba = s_N[b * K + a];
        bad = bad || isnan(ab);
        cons = cons || (ab < p.c_thr && ba < p.c_thr);
        div = div && (ab > p.d_thr);
      }
    if (bad) atomicOr(p.status, SPEC_DEV_NONFINITE);
    if (p.cons) p.cons[gi] = cons ? 1 : 0;
    if (p.div) p.div[gi] = div ? 1 : 0;
  }
}

// Block reduction of the per-thread pairwise sums of one tile (per row a: reference mr,
// sum s; per ordered pair: kk) into the tile's PairPartial. Every thread calls it.
template <int K>
__device__ __forceinline__ void pair_partial_write(PairPartial* dst, const float (&mr)[K], const float (&s)[K],
                                                   const float (&kk)[K][K], float c, const PairParams& q) {
  __shared__ float s_red[kWarps][K + K * K];
  __shared__ float s_ref[kWarps][K];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int a = 0; a < K; ++a) {
    const float wm = warp_max(mr[a]);
    if (lane == 0) s_ref[warp][a] = wm;
  }
  __syncthreads();
  float DM[K];
#pragma unroll
  for (int a = 0; a < K; ++a) {
    DM[a] = s_ref[0][a];
    for (int w = 1; w < kWarps; ++w) DM[a] = fmaxf(DM[a], s_ref[w][a]);
    const float f = (mr[a] == -INFINITY) ? 0.f : ex2((mr[a] - DM[a]) * c);
    const float ws = warp_sum(s[a] * f);
    if (lane == 0) s_red[warp][a] = ws;
#pragma unroll
    for (int b = 0; b < K; ++b) {
      const float wk = warp_sum(kk[a][b] * f);
      if (lane == 0) s_red[warp][K + a * K + b] = wk;
    }
  }
  __syncthreads();
  const bool ok = in_ext(dst, sizeof(PairPartial), q.x_ws, q.status);
  if (ok && threadIdx.x < K + K * K) {
    float t = 0.f;
    for (int w = 0; w < kWarps; ++w) t += s_red[w][threadIdx.x];
    if (threadIdx.x < K)
      __stcg(&dst->s[threadIdx.x], t);
    else
      __stcg(&dst->k[threadIdx.x - K], t);
  }
  if (ok && threadIdx.x < K) __stcg(&dst->ref[threadIdx.x], DM[threadIdx.x]);
}

template <typename E, int VEC, int K>
__global__ void __launch_bounds__(kThreads, 2) pair_kernel(const __grid_constant__ PairParams p) {
  using io = IO<E, VEC>;
  using raw_t = typename io::raw_t;
  griddep_wait();  // earlier work on the stream (the verification, the prologue) has completed
  griddep_launch();
  __shared__ int s_last;
  const int tile = blockIdx.x;
  const int gi = tile / p.nchunks, chunk = tile - gi * p.nchunks;
  const int g = gi / p.gamma, i = gi - g * p.gamma;
  const size_t V = (size_t)p.V;
  const E* rows[K];
#pragma unroll
  for (int a = 0; a < K; ++a)
    rows[a] = static_cast<const E*>(p.draft) + ((size_t)(g * K + a) * p.gamma + i) * V;
  const int e_begin = chunk * p.chunk_elems;
  const int e_end = min(e_begin + p.chunk_elems, p.V);
  const int v1 = e_end / VEC;
  const float c = p.c;

  float mr[K], mth[K], nmc[K], s[K], kk[K][K];
#pragma unroll
  for (int a = 0; a < K; ++a) {
    mr[a] = -INFINITY;
    mth[a] = -INFINITY;
    nmc[a] = 0.f;
    s[a] = 0.f;
#pragma unroll
    for (int b = 0; b < K; ++b) kk[a][b] = 0.f;
  }
  auto fold = [&](const float (&z)[K][VEC]) {
#pragma unroll
    for (int a = 0; a < K; ++a) {
      const float vm = vmax<VEC>(z[a]);
      const bool mv = vm > mth[a];
      if (__any_sync(__activemask(), mv)) {
        if (mv) {
          const float f = ex2((mr[a] - vm) * c);
          s[a] *= f;
#pragma unroll
          for (int b = 0; b < K; ++b) kk[a][b] *= f;
          mr[a] = vm;
          mth[a] = vm + kLazy / c;
          nmc[a] = -vm * c;
        }
      }
    }
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
#pragma unroll
      for (int a = 0; a < K; ++a) {
        const float e = ex2(fmaf(z[a][j], c, nmc[a]));
        s[a] += e;
#pragma unroll
        for (int b = 0; b < K; ++b)
          if (b != a) kk[a][b] = fmaf(e, z[a][j] - z[b][j], kk[a][b]);
      }
    }
  };
  int v = e_begin / VEC + threadIdx.x;
  for (; v + kThreads < v1; v += 2 * kThreads) {
    raw_t r0[K], r1[K];
#pragma unroll
    for (int a = 0; a < K; ++a) {
      r0[a] = in_ext(rows[a] + (size_t)v * VEC, 16, p.x_draft, p.status) ? io::load(rows[a], v) : make_uint4(0, 0, 0, 0);
      r1[a] = in_ext(rows[a] + (size_t)(v + kThreads) * VEC, 16, p.x_draft, p.status) ? io::load(rows[a], v + kThreads)
                                                                                        : make_uint4(0, 0, 0, 0);
    }
    float z[K][VEC];
#pragma unroll
    for (int a = 0; a < K; ++a) io::unpack(r0[a], z[a]);
    fold(z);
#pragma unroll
    for (int a = 0; a < K; ++a) io::unpack(r1[a], z[a]);
    fold(z);
  }
  if (v < v1) {
    float z[K][VEC];
#pragma unroll
    for (int a = 0; a < K; ++a)
      io::unpack(in_ext(rows[a] + (size_t)v * VEC, 16, p.x_draft, p.status) ? io::load(rows[a], v) : make_uint4(0, 0, 0, 0),
                 z[a]);
    fold(z);
  }

  pair_partial_write<K>(p.part + tile, mr, s, kk, c, p);
  __syncthreads();  // every writer's partial entries precede thread 0's ticket
  if (threadIdx.x == 0) {
    // release: the tile's partial before its ticket; acquire: the other tiles' partials
    // before this block's reads
    const unsigned old = atom_add_acq_rel_gpu(p.cnt + gi, 1u);
    s_last = (old + 1u == (unsigned)p.nchunks) ? 1 : 0;
  }
  __syncthreads();
  if (!s_last) return;

  pair_merge<K>(p, gi);
}

// Rows off the 16-byte grid: the same pairwise sums through per-warp bulk-copy rings of the
// aligned blocks covering each run (the K rows may sit at K different offsets). Warp w
// takes the w-th contiguous run of every stage of the K rows, one slot per row (each with
// its own phase); lane l reads the elements l, l + 32, ... of a run and folds them in as
// strided groups.
template <int K>
__host__ __device__ constexpr int pair_staged_smem() {
  return kCS * kWarps * K * kWarpSlot;
}

// The lazy-reference update and the sums of one group of G elements of every row.
template <int K, int G>
__device__ __forceinline__ void pair_fold(float (&mr)[K], float (&mth)[K], float (&nmc)[K], float (&s)[K],
                                          float (&kk)[K][K], const float (&z)[K][G], float c) {
#pragma unroll
  for (int a = 0; a < K; ++a) {
    const float vm = vmax<G>(z[a]);
    const bool mv = vm > mth[a];
    if (__any_sync(__activemask(), mv)) {
      if (mv) {
        const float f = ex2((mr[a] - vm) * c);
        s[a] *= f;
#pragma unroll
        for (int b = 0; b < K; ++b) kk[a][b] *= f;
        mr[a] = vm;
        mth[a] = vm + kLazy / c;
        nmc[a] = -vm * c;
      }
    }
  }
#pragma unroll
  for (int j = 0; j < G; ++j) {
#pragma unroll
    for (int a = 0; a < K; ++a) {
      const float e = ex2(fmaf(z[a][j], c, nmc[a]));
      s[a] += e;
#pragma unroll
      for (int b = 0; b < K; ++b)
        if (b != a) kk[a][b] = fmaf(e, z[a][j] - z[b][j], kk[a][b]);
    }
  }
}

template <typename E, int K>
__global__ void __launch_bounds__(kThreads, 2) pair_staged_kernel(const __grid_constant__ PairParams p) {
  extern __shared__ __align__(128) unsigned char dsm[];
  griddep_wait();  // earlier work on the stream (the verification, the prologue) has completed
  griddep_launch();
  __shared__ int s_last;
  __shared__ __align__(8) uint64_t s_bars[kWarps][kCS];
  constexpr int SW = kWarpRowBytes / (int)sizeof(E);  // elements of a warp's run of a row
  constexpr int S = SW * kWarps;                      // elements of a stage
  constexpr int U = SW / 32;                          // per lane per run and row
  constexpr unsigned WSTAGE = K * kWarpSlot;          // a warp's part of one stage
  const int tile = blockIdx.x;
  const int gi = tile / p.nchunks, chunk = tile - gi * p.nchunks;
  const int g = gi / p.gamma, i = gi - g * p.gamma;
  const size_t V = (size_t)p.V;
  const E* rows[K];
#pragma unroll
  for (int a = 0; a < K; ++a)
    rows[a] = static_cast<const E*>(p.draft) + ((size_t)(g * K + a) * p.gamma + i) * V;
  const int e_begin = chunk * p.chunk_elems;
  const int e_end = min(e_begin + p.chunk_elems, p.V);
  const float c = p.c;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  float mr[K], mth[K], nmc[K], s[K], kk[K][K];
  int ph[K];  // S and SW elements are whole 16-byte blocks: every run of a row has its phase
#pragma unroll
  for (int a = 0; a < K; ++a) {
    mr[a] = -INFINITY;
    mth[a] = -INFINITY;
    nmc[a] = 0.f;
    s[a] = 0.f;
    ph[a] = phase16(rows[a] + e_begin);
#pragma unroll
    for (int b = 0; b < K; ++b) kk[a][b] = 0.f;
  }
  WarpRing ring;
  ring.init(s_bars[warp]);
  const uint32_t wbase = (uint32_t)__cvta_generic_to_shared(dsm) + (uint32_t)warp * WSTAGE;
  const int nst = (e_end - e_begin + S - 1) / S;
  auto issue = [&](int k) {
    if (lane == 0 && k < nst) {
      const uint32_t slot = wbase + (uint32_t)((k % kCS) * kWarps) * WSTAGE;
      const int e0 = e_begin + k * S + warp * SW, n = min(SW, e_end - e0);
      const void* src[K];
      uint32_t nb[K], total = 0u;
#pragma unroll
      for (int a = 0; a < K; ++a) {
        src[a] = nullptr;
        nb[a] = run_blocks<E>(rows[a], e0, n, &src[a]);
        if (nb[a] && !in_ext(src[a], nb[a], p.x_draft, p.status)) nb[a] = 0;
        total += nb[a];
      }
      const uint32_t bar = ring.bars + 8u * (uint32_t)(k % kCS);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the reads of the slot precede the copies
      mbar_expect_arrive(bar, total);
#pragma unroll
      for (int a = 0; a < K; ++a)
        if (nb[a]) bulk_copy(slot + (uint32_t)a * kWarpSlot, src[a], nb[a], bar);
    }
  };
#pragma unroll
  for (int k = 0; k < kCS - 1; ++k) issue(k);
  for (int k = 0; k < nst; ++k) {
    __syncwarp();        // every lane is done with stage k - 1
    issue(k + kCS - 1);  // into the slot of stage k - 1
    ring.wait(k, p.status);
    const unsigned char* slot = dsm + (size_t)(warp + (k % kCS) * kWarps) * WSTAGE;
    const int n = min(SW, e_end - (e_begin + k * S + warp * SW));
    if (lane + (U - 1) * 32 < n) {  // the whole strided group is inside the run
      float z[K][U];
#pragma unroll
      for (int a = 0; a < K; ++a) {
        const E* sr = reinterpret_cast<const E*>(slot + a * kWarpSlot) + ph[a];
#pragma unroll
        for (int j = 0; j < U; ++j) z[a][j] = sh_elem<E>(sr, lane + 32 * j);
      }
      pair_fold<K, U>(mr, mth, nmc, s, kk, z, c);
    } else {
      for (int x = lane; x < n; x += 32) {
        float z[K][1];
#pragma unroll
        for (int a = 0; a < K; ++a)
          z[a][0] = sh_elem<E>(reinterpret_cast<const E*>(slot + a * kWarpSlot) + ph[a], x);
        pair_fold<K, 1>(mr, mth, nmc, s, kk, z, c);
      }
    }
  }

  pair_partial_write<K>(p.part + tile, mr, s, kk, c, p);
  __syncthreads();  // every writer's partial entries precede thread 0's ticket
  if (threadIdx.x == 0) {
    // release: the tile's partial before its ticket; acquire: the other tiles' partials
    // before this block's reads
    const unsigned old = atom_add_acq_rel_gpu(p.cnt + gi, 1u);
    s_last = (old + 1u == (unsigned)p.nchunks) ? 1 : 0;
  }
  __syncthreads();
  if (!s_last) return;

  pair_merge<K>(p, gi);
}

// sum_j e[j] (x[j] - y[j]) with packed f32x2 subtractions and FMAs
template <int VEC>
__device__ __forceinline__ float dot_diff(const float (&e)[VEC], const float (&x)[VEC], const float (&y)[VEC]) {
  if constexpr (VEC == 1) {
    return e[0] * (x[0] - y[0]);
  } else {
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < VEC / 2; ++j)
      acc = fma2(make_float2(e[2 * j], e[2 * j + 1]),
                 sub2(make_float2(x[2 * j], x[2 * j + 1]), make_float2(y[2 * j], y[2 * j + 1])), acc);
    return acc.x + acc.y;
  }
}

// ---------------------------------------------------------------------------
// Fused multi-draft tiles (aligned rows): one block per (group, row r, vocabulary chunk)
// reads the K candidates' target rows r and, for r < gamma, their draft rows r, each
// logit once, through a per-thread 3- or 4-stage cp.async ring (one 16-byte vector per row
// per stage, lane-interleaved as in the tile kernel). Per candidate it keeps the tile
// kernel's statistics (target maximum, index and, stochastic, sum; draft sum and the KL
// sum against the candidate's own target row) and writes them as that candidate's
// partial, so the ordinary per-sequence tickets and finalisation decide the candidates;
// from the same draft exponentials it keeps the pairwise sums of the matrix.
template <int K>
__host__ __device__ constexpr int multi_stages() {
  // two blocks per SM: 4 x 24 KB (K = 3; G=64, gamma=8, V=128256: 175.0 against 177.1 us
  // with 3 stages, same box), 3 x 32 KB (K = 4)
  return K <= 3 ? 4 : 3;
}

template <int K>
__host__ __device__ constexpr int multi_smem() {
  return multi_stages<K>() * 2 * K * kThreads * 16;
}

// One stage of a fused tile on a draft position (K <= 3), thread-local. The lazy references
// of the K draft rows (and, stochastic, of the K target rows) are checked with one vote;
// one difference z_a - z_b feeds both K_ab and K_ba (each pair sum chained from its
// accumulator and folded once per vector). Per candidate -- stochastic: the target maximum
// (no index: nothing reads the argmax of a stochastic multi-draft row) and sum, and the
// verification's KL sum against the candidate's own target row; greedy: the argmax.
// bf16 keeps the 2K vectors packed and goes through them a pair of elements at a time
// (every exponential used as soon as it is computed); fp32 unpacks the K draft vectors
// together and computes all their exponentials before the pairwise sums.
template <typename E, int VEC, int K, bool STOCH>
__device__ __forceinline__ void multi_pair_stage(const uint4* sq, int e0, float c, float cq, TAcc (&ta)[K],
                                                 DAcc (&da)[K], float (&kk)[K][K]) {
  using io = IO<E, VEC>;
  static_assert(VEC % 2 == 0, "packed pairs of elements");
  if constexpr (VEC == 8) {
    // bf16: the 2K vectors stay packed until each pair of elements is used -- their maxima
    // taken on the packed values -- so that a thread holds 2K words of raw data rather than
    // 16K unpacked floats and the candidates' exponentials of a pair of elements are used
    // as soon as they are computed
    uint4 rd[K], rt[K];
    float vmd[K], vmt[K];
    bool mv = false;
#pragma unroll
    for (int a = 0; a < K; ++a) {
      rd[a] = sq[(K + a) * kThreads];
      vmd[a] = vmax_bf16x8(rd[a]);
      mv = mv || vmd[a] > da[a].mth;
      rt[a] = sq[a * kThreads];
      if constexpr (STOCH) {
        vmt[a] = vmax_bf16x8(rt[a]);
        ta[a].m = fmaxf(ta[a].m, vmt[a]);
        mv = mv || vmt[a] > ta[a].mth;
      }
    }
    if (__any_sync(__activemask(), mv)) {
#pragma unroll
      for (int a = 0; a < K; ++a) {
        if (vmd[a] > da[a].mth) {
          const float f = ex2((da[a].mr - vmd[a]) * cq);
          da[a].s = make_float2(da[a].s.x * f, da[a].s.y * f);
          da[a].k = make_float2(da[a].k.x * f, da[a].k.y * f);
#pragma unroll
          for (int b = 0; b < K; ++b) kk[a][b] *= f;
          da[a].mr = vmd[a];
          da[a].mth = vmd[a] + kLazy / cq;
          da[a].nmc = -vmd[a] * cq;
        }
        if constexpr (STOCH) {
          if (vmt[a] > ta[a].mth) {
            const float f = ex2((ta[a].mr - vmt[a]) * c);
            ta[a].s = make_float2(ta[a].s.x * f, ta[a].s.y * f);
            ta[a].mr = vmt[a];
            ta[a].mth = vmt[a] + kLazy / c;
            ta[a].nmc = -vmt[a] * c;
          }
        }
      }
    }
    // K_ab += sum e_a (z_a - z_b); K_ba += sum e_b (z_b - z_a), kept negated in its chain
    float2 pk[K][K];
#pragma unroll
    for (int a = 0; a < K; ++a)
#pragma unroll
      for (int b = a + 1; b < K; ++b) {
        pk[a][b] = make_float2(kk[a][b], 0.f);
        pk[b][a] = make_float2(-kk[b][a], 0.f);
      }
    const float2 cq2 = make_float2(cq, cq), c2 = make_float2(c, c);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float2 zd[K], ed[K];
#pragma unroll
      for (int a = 0; a < K; ++a) {
        zd[a] = bf16_pair(rd[a], j);
        const float2 x = fma2(zd[a], cq2, make_float2(da[a].nmc, da[a].nmc));
        ed[a] = make_float2(ex2(x.x), ex2(x.y));
        da[a].s = add2(da[a].s, ed[a]);
      }
#pragma unroll
      for (int a = 0; a < K; ++a)
#pragma unroll
        for (int b = a + 1; b < K; ++b) {
          const float2 d = sub2(zd[a], zd[b]);
          pk[a][b] = fma2(ed[a], d, pk[a][b]);
          pk[b][a] = fma2(ed[b], d, pk[b][a]);
        }
      if constexpr (STOCH) {
#pragma unroll
        for (int a = 0; a < K; ++a) {
          const float2 zt = bf16_pair(rt[a], j);
          const float2 x = fma2(zt, c2, make_float2(ta[a].nmc, ta[a].nmc));
          ta[a].s = add2(ta[a].s, make_float2(ex2(x.x), ex2(x.y)));
          da[a].k = fma2(ed[a], sub2(zd[a], zt), da[a].k);
        }
      }
    }
#pragma unroll
    for (int a = 0; a < K; ++a)
#pragma unroll
      for (int b = a + 1; b < K; ++b) {
        kk[a][b] = pk[a][b].x + pk[a][b].y;
        kk[b][a] = -(pk[b][a].x + pk[b][a].y);
      }
    if constexpr (!STOCH) {
#pragma unroll
      for (int a = 0; a < K; ++a) {
        float ft[VEC];
        io::unpack(rt[a], ft);
        argmax_update<VEC>(ta[a], ft, e0);
      }
    }
  } else {
    // fp32: the K draft vectors unpacked together
    float fd[K][VEC], vm[K];
    bool mv = false;
#pragma unroll
    for (int a = 0; a < K; ++a) {
      io::unpack(sq[(K + a) * kThreads], fd[a]);
      vm[a] = vmax<VEC>(fd[a]);
      mv = mv || vm[a] > da[a].mth;
    }
    if (__any_sync(__activemask(), mv)) {
#pragma unroll
      for (int a = 0; a < K; ++a) {
        if (vm[a] > da[a].mth) {
          const float f = ex2((da[a].mr - vm[a]) * cq);
          da[a].s = make_float2(da[a].s.x * f, da[a].s.y * f);
          da[a].k = make_float2(da[a].k.x * f, da[a].k.y * f);
#pragma unroll
          for (int b = 0; b < K; ++b) kk[a][b] *= f;
          da[a].mr = vm[a];
          da[a].mth = vm[a] + kLazy / cq;
          da[a].nmc = -vm[a] * cq;
        }
      }
    }
    float ed[K][VEC];
#pragma unroll
    for (int a = 0; a < K; ++a) da[a].s = add2(da[a].s, exp_sum2<VEC>(fd[a], cq, da[a].nmc, ed[a]));
#pragma unroll
    for (int a = 0; a < K; ++a) {
#pragma unroll
      for (int b = a + 1; b < K; ++b) {
        // K_ab += sum e_a (z_a - z_b); K_ba += sum e_b (z_b - z_a), kept negated in the chain
        float2 pab = make_float2(kk[a][b], 0.f), nba = make_float2(-kk[b][a], 0.f);
#pragma unroll
        for (int j = 0; j < VEC / 2; ++j) {
          const float2 d = sub2(make_float2(fd[a][2 * j], fd[a][2 * j + 1]), make_float2(fd[b][2 * j], fd[b][2 * j + 1]));
          pab = fma2(make_float2(ed[a][2 * j], ed[a][2 * j + 1]), d, pab);
          nba = fma2(make_float2(ed[b][2 * j], ed[b][2 * j + 1]), d, nba);
        }
        kk[a][b] = pab.x + pab.y;
        kk[b][a] = -(nba.x + nba.y);
      }
    }
#pragma unroll
    for (int a = 0; a < K; ++a) {
      float ft[VEC];
      io::unpack(sq[a * kThreads], ft);
      if constexpr (STOCH) {
        const float tm = vmax<VEC>(ft);
        ta[a].m = fmaxf(ta[a].m, tm);
        lazy_ref(ta[a].mr, ta[a].mth, ta[a].nmc, ta[a].s, nullptr, tm, c);
        float et[VEC];
        ta[a].s = add2(ta[a].s, exp_sum2<VEC>(ft, c, ta[a].nmc, et));
#pragma unroll
        for (int j = 0; j < VEC / 2; ++j)
          da[a].k = fma2(make_float2(ed[a][2 * j], ed[a][2 * j + 1]),
                         sub2(make_float2(fd[a][2 * j], fd[a][2 * j + 1]), make_float2(ft[2 * j], ft[2 * j + 1])),
                         da[a].k);
      } else {
        argmax_update<VEC>(ta[a], ft, e0);
      }
    }
  }
}

template <typename E, int VEC, int K, int MODE>
__global__ void __launch_bounds__(kThreads, 2) multi_rows_kernel(const __grid_constant__ RowsParams p,
                                                                 const __grid_constant__ PairParams q) {
  using io = IO<E, VEC>;
  constexpr bool STOCH = MODE == M_STOCH;
  constexpr int kMS = multi_stages<K>();
  extern __shared__ __align__(128) unsigned char dsm[];
  griddep_wait();  // the prologue, and everything earlier on the stream, has completed
  griddep_launch();
  __shared__ int s_last[K + 1];
  const int gamma = p.gamma, nchunks = p.nchunks;
  const int per = (gamma + 1) * nchunks;
  const int tile = blockIdx.x;
  const int g = tile / per, rem = tile - g * per;
  const int r = rem / nchunks, chunk = rem - r * nchunks;
  const bool pair = r < gamma;
  const size_t V = (size_t)p.V;
  const E* trow[K];
  const E* drow[K];
#pragma unroll
  for (int k = 0; k < K; ++k) {
    const size_t b = (size_t)g * K + k;
    trow[k] = static_cast<const E*>(p.target) + (b * (gamma + 1) + r) * V;
    drow[k] = pair ? static_cast<const E*>(p.draft) + (b * gamma + r) * V : trow[k];
  }
  const int e_begin = chunk * p.chunk_elems;
  const int e_end = min(e_begin + p.chunk_elems, p.V);
  const int v0 = e_begin / VEC, v1 = e_end / VEC;
  const float c = p.c;   // target scale (the greedy call's argmax needs none)
  const float cq = q.c;  // draft scale, log2(e) / T: the matrix's and, stochastic, the verification's

  TAcc ta[K];
  DAcc da[K];
  float kk[K][K];
#pragma unroll
  for (int k = 0; k < K; ++k) {
    init(ta[k]);
    init(da[k]);
#pragma unroll
    for (int b = 0; b < K; ++b) kk[k][b] = 0.f;
  }

  constexpr unsigned SLOT = 2 * K * kThreads * 16;
  const int t = threadIdx.x;
  const uint32_t base = (uint32_t)__cvta_generic_to_shared(dsm) + 16u * t;
  const int nst = (v1 - v0 + kThreads - 1) / kThreads;
  const int nr = pair ? 2 * K : K;
  auto issue = [&](int st) {
    if (st < nst) {
      const int v = v0 + t + st * kThreads;
      if (v < v1) {
        const uint32_t slot = base + (uint32_t)(st % kMS) * SLOT;
#pragma unroll
        for (int j = 0; j < 2 * K; ++j) {
          const E* src = (j < K ? trow[j] : drow[j - K]) + (size_t)v * VEC;
          if (j < nr && in_ext(src, 16, j < K ? p.x_target : p.x_draft, p.status))
            cp_async16(slot + (uint32_t)(j * kThreads * 16), src);
        }
      }
    }
    cp_commit();
  };
#pragma unroll
  for (int st = 0; st < kMS - 1; ++st) issue(st);
  for (int st = 0; st < nst; ++st) {
    issue(st + kMS - 1);
    cp_wait<kMS - 1>();
    const int v = v0 + t + st * kThreads;
    if (v >= v1) continue;
    const uint4* sq = reinterpret_cast<const uint4*>(dsm + (size_t)(st % kMS) * SLOT) + t;
    const int e0 = v * VEC;
    if constexpr (K <= 3) {
      if (pair) {
        multi_pair_stage<E, VEC, K, STOCH>(sq, e0, c, cq, ta, da, kk);
        continue;
      }
    }
    // K = 4 pairs (every candidate's draft vectors held at once would spill: they are
    // unpacked per use) and the bonus row of every K
    constexpr bool PRE = K <= 3;
    float fdk[PRE ? K : 1][VEC];
    if (PRE && pair) {
#pragma unroll
      for (int a = 0; a < (PRE ? K : 0); ++a) io::unpack(sq[(K + a) * kThreads], fdk[a]);
    }
#pragma unroll
    for (int a = 0; a < K; ++a) {
      float ft[VEC];
      io::unpack(sq[a * kThreads], ft);
      if (!pair || !STOCH) {
        if (STOCH)
          tsum_update<VEC, VEC, false>(ta[a], ft, e0, c);  // the stochastic bonus row (no index)
        else
          argmax_update<VEC>(ta[a], ft, e0);   // greedy rows
      } else {
        const float vm = vmax<VEC>(ft);
        track_max<VEC, VEC, false>(ta[a], vm, e0);
        lazy_ref(ta[a].mr, ta[a].mth, ta[a].nmc, ta[a].s, nullptr, vm, c);
        float et[VEC];
        ta[a].s = add2(ta[a].s, exp_sum2<VEC>(ft, c, ta[a].nmc, et));
      }
      if (pair) {
        float fdu[VEC];
        if constexpr (!PRE) io::unpack(sq[(K + a) * kThreads], fdu);
        const float (&fd)[VEC] = PRE ? fdk[PRE ? a : 0] : fdu;
        float ed[VEC];
        const float vm = vmax<VEC>(fd);
        const bool mv = vm > da[a].mth;
        if (__any_sync(__activemask(), mv)) {
          if (mv) {
            const float f = ex2((da[a].mr - vm) * cq);
            da[a].s = make_float2(da[a].s.x * f, da[a].s.y * f);
            da[a].k = make_float2(da[a].k.x * f, da[a].k.y * f);
#pragma unroll
            for (int b = 0; b < K; ++b) kk[a][b] *= f;
            da[a].mr = vm;
            da[a].mth = vm + kLazy / cq;
            da[a].nmc = -vm * cq;
          }
        }
        da[a].s = add2(da[a].s, exp_sum2<VEC>(fd, cq, da[a].nmc, ed));
        if (STOCH) da[a].k.x += dot_diff<VEC>(ed, fd, ft);
#pragma unroll
        for (int b = 0; b < K; ++b) {
          if (b == a) continue;
          if constexpr (PRE) {
            kk[a][b] += dot_diff<VEC>(ed, fd, fdk[b]);
          } else {
            float fb[VEC];
            io::unpack(sq[(K + b) * kThreads], fb);
            kk[a][b] += dot_diff<VEC>(ed, fd, fb);
          }
        }
      }
    }
  }
  cp_wait<0>();

  // partials: one per candidate in the tile kernel's layout, one pairwise partial
  const int kind = pair ? (STOCH ? K_PAIR : K_ARGMAX) : (STOCH ? K_TSUM : K_ARGMAX);
#pragma unroll
  for (int a = 0; a < K; ++a) {
    const Partial part = reduce_tile<BlockSync, E, VEC>(kind, ta[a], da[a], c, trow[a], cq, &p.x_target, p.status);
    const size_t row = ((size_t)g * K + a) * (gamma + 1) + r;
    float4* dst = reinterpret_cast<float4*>(p.part + row * nchunks + chunk);
    if (threadIdx.x == 0 && in_ext(dst, sizeof(Partial), p.x_ws, p.status)) {
      __stcg(dst, make_float4(part.tm, part.ts, __int_as_float(part.tidx), __int_as_float(part.bad)));
      __stcg(dst + 1, make_float4(part.dm, part.ds, part.dk, part.ds2));
    }
    __syncthreads();  // reduce_tile's shared arrays are reused by the next candidate
  }
  if (pair) {
    float mr[K], sm[K];
#pragma unroll
    for (int a = 0; a < K; ++a) {
      mr[a] = da[a].mr;
      sm[a] = da[a].s.x + da[a].s.y;
    }
    pair_partial_write<K>(q.part + ((size_t)g * gamma + r) * nchunks + chunk, mr, sm, kk, cq, q);
  }
  __syncthreads();  // every writer's partial entries precede thread 0's fence
  if (threadIdx.x == 0) {
    __threadfence();
    bool any = false;
    for (int a = 0; a < K; ++a) {
      const unsigned old = in_ext(p.cnt + (size_t)g * K + a, sizeof(unsigned), p.x_ws, p.status)
                               ? atomicAdd(p.cnt + (size_t)g * K + a, 1u) : 0u;
      s_last[a] = (old + 1u == (unsigned)per) ? 1 : 0;
      any = any || s_last[a];
    }
    s_last[K] = 0;
    if (pair) {
      const unsigned old = in_ext(q.cnt + (size_t)g * gamma + r, sizeof(unsigned), q.x_ws, q.status)
                               ? atomicAdd(q.cnt + (size_t)g * gamma + r, 1u) : 0u;
      s_last[K] = (old + 1u == (unsigned)nchunks) ? 1 : 0;
      any = any || s_last[K];
    }
    if (any) __threadfence();  // ... and the other tiles' partials before this block's reads
  }
  __syncthreads();
  for (int a = 0; a < K; ++a) {
    if (s_last[a]) {
      const int b = g * K + a;
      finalize<E, MODE, BlockSync>(p, b, gamma, b * (gamma + 1), b * gamma);
      __syncthreads();
    }
  }
  if (s_last[K]) pair_merge<K>(q, g * gamma + r);
  if constexpr (STOCH) {
    __syncthreads();  // the finalisers' writes precede the count
    if (threadIdx.x == 0) tile_done<MODE>(p);
  }
}

// Per group: the candidate with the most accepted drafts (the lowest index among equals;
// -1 when every candidate had a data error) and its tokens.
__global__ void select_kernel(const int32_t* n_acc, const int32_t* out_tok, int G, int K, int gamma,
                              int32_t* best_k, int32_t* best_n, int32_t* best_tok) {
  griddep_wait();  // the verification of every candidate has completed
  griddep_launch();
  const int g = blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= G) return;
  int best = -1, bn = -1;
  for (int k = 0; k < K; ++k) {
    const int n = n_acc[(size_t)g * K + k];
    if (n > bn) {
      bn = n;
      best = k;
    }
  }
  best_k[g] = best;
  best_n[g] = bn;
  for (int j = 0; j <= gamma; ++j)
    best_tok[(size_t)g * (gamma + 1) + j] = best >= 0 ? out_tok[((size_t)g * K + best) * (gamma + 1) + j] : -1;
}

}  // namespace sv
