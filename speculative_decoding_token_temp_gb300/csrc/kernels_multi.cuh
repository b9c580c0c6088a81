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

#include "kernels.cuh"

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
};

template <typename E, int VEC, int K>
__global__ void __launch_bounds__(kThreads, 2) pair_kernel(const __grid_constant__ PairParams p) {
  using io = IO<E, VEC>;
  using raw_t = typename io::raw_t;
  griddep_wait();  // earlier work on the stream (the verification, the prologue) has completed
  griddep_launch();
  __shared__ float s_red[kWarps][K + K * K];
  __shared__ float s_ref[kWarps][K];
  __shared__ int s_last;
  __shared__ float s_M[K], s_S[K], s_K[K * K], s_N[K * K];
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
      r0[a] = io::load(rows[a], v);
      r1[a] = io::load(rows[a], v + kThreads);
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
    for (int a = 0; a < K; ++a) io::unpack(io::load(rows[a], v), z[a]);
    fold(z);
  }

  // block reduction: per row the largest reference, the sums moved to it
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
  PairPartial* dst = p.part + tile;
  if (threadIdx.x < K + K * K) {
    float t = 0.f;
    for (int w = 0; w < kWarps; ++w) t += s_red[w][threadIdx.x];
    if (threadIdx.x < K)
      __stcg(&dst->s[threadIdx.x], t);
    else
      __stcg(&dst->k[threadIdx.x - K], t);
  }
  if (threadIdx.x < K) __stcg(&dst->ref[threadIdx.x], DM[threadIdx.x]);
  __syncthreads();  // every writer's partial entries precede thread 0's fence
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned old = atomicAdd(p.cnt + gi, 1u);
    s_last = (old + 1u == (unsigned)p.nchunks) ? 1 : 0;
    if (s_last) __threadfence();
  }
  __syncthreads();
  if (!s_last) return;

  // merge the chunks of this (group, position): thread (a, j) owns S_a (j == K) or K_aj
  const PairPartial* pp = p.part + (size_t)gi * p.nchunks;
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
