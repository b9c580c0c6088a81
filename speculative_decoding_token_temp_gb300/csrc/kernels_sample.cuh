// Inverse-CDF sampling of the correction (residual) or bonus token, [SpS] section
// "核心算法数学原理：无损拒绝采样": y = min{v : C(v) > u * Z}, C the running sum in token
// order of w_v = max(0, p_v - q_v) over the rejected row pair, or of w_v = p_v over the
// bonus row; Z the total.
#pragma once

#include "kernels.cuh"

namespace sv {

// Weights of one loaded vector.
template <int VEC>
__device__ __forceinline__ void weights(int mode, const float (&t)[VEC], const float (&d)[VEC], float lt2, float ld2,
                                        float c, float (&w)[VEC]) {
  if (mode == S_RESID) {
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
      const float pv = ex2(fmaf(t[k], c, -lt2));
      const float qv = ex2(fmaf(d[k], c, -ld2));
      w[k] = fmaxf(pv - qv, 0.f);
    }
  } else {
#pragma unroll
    for (int k = 0; k < VEC; ++k) w[k] = ex2(fmaf(t[k], c, -lt2));
  }
}

// One sampling segment [e_begin, e_end), split into kWarps contiguous warp ranges, each
// walked in steps of 32 vectors (one per lane). Returns this warp's sum (fp64, in step
// order; identical in every lane). If `steps` is given, the fp32 step totals are stored
// at steps[warp * kMaxSteps + s].
template <typename E, int VEC>
__device__ __forceinline__ double segment_pass(const E* trow, const E* drow, int mode, float lt2, float ld2, float c,
                                               int e_begin, int e_end, float* steps) {
  using io = IO<E, VEC>;
  using raw_t = typename io::raw_t;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int v0 = e_begin / VEC, v1 = e_end / VEC;
  const int W = (v1 - v0 + kWarps - 1) / kWarps;
  const int wb = v0 + warp * W;
  const int we = min(wb + W, v1);
  const int nsteps = (we > wb) ? (we - wb + 31) / 32 : 0;
  double acc = 0.0;
  constexpr int U = 4;
  int s = 0;
  for (; s + U <= nsteps; s += U) {
    raw_t rt[U], rd[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = wb + (s + u) * 32 + lane;
      if (v < we) {
        rt[u] = io::load(trow, v);
        if (mode == S_RESID) rd[u] = io::load(drow, v);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = wb + (s + u) * 32 + lane;
      float ls = 0.f;
      if (v < we) {
        float ft[VEC], fd[VEC], w[VEC];
        io::unpack(rt[u], ft);
        if (mode == S_RESID) io::unpack(rd[u], fd);
        weights<VEC>(mode, ft, fd, lt2, ld2, c, w);
        ls = tree_sum<VEC>(w);
      }
      const float st = warp_sum(ls);
      if (steps != nullptr && lane == 0) steps[warp * kMaxSteps + s + u] = st;
      acc += (double)st;
    }
  }
  for (; s < nsteps; ++s) {
    const int v = wb + s * 32 + lane;
    float ls = 0.f;
    if (v < we) {
      float ft[VEC], fd[VEC], w[VEC];
      io::unpack(io::load(trow, v), ft);
      if (mode == S_RESID) io::unpack(io::load(drow, v), fd);
      weights<VEC>(mode, ft, fd, lt2, ld2, c, w);
      ls = tree_sum<VEC>(w);
    }
    const float st = warp_sum(ls);
    if (steps != nullptr && lane == 0) steps[warp * kMaxSteps + s] = st;
    acc += (double)st;
  }
  return acc;
}

template <typename E, int VEC>
__global__ void __launch_bounds__(kThreads) sample_kernel(const __grid_constant__ SampleParams p) {
  griddep_wait();  // the row statistics of every sequence are final
  __shared__ SeqRec s_rec;
  __shared__ int s_last, s_mode, s_seg, s_wsel, s_ssel;
  __shared__ double s_w[kWarps];
  __shared__ double s_target, s_base;
  __shared__ float s_steps[kWarps * kMaxSteps];
  const int b = blockIdx.x / p.nseg, seg = blockIdx.x - (blockIdx.x / p.nseg) * p.nseg;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    const int4 a = __ldcg(reinterpret_cast<const int4*>(p.rec + b));
    const int4 z = __ldcg(reinterpret_cast<const int4*>(p.rec + b) + 1);
    s_rec.state = a.x;
    s_rec.n = a.y;
    s_rec.t_row = a.z;
    s_rec.d_row = a.w;
    s_rec.lt2 = __int_as_float(z.x);
    s_rec.ld2 = __int_as_float(z.y);
    s_rec.us = __int_as_float(z.z);
    s_rec.mode = z.w;
  }
  __syncthreads();
  const SeqRec q = s_rec;
  if (q.state != REC_READY) return;
  if (q.t_row < 0 || q.t_row >= p.total_rows || (q.mode == S_RESID && (q.d_row < 0 || q.d_row >= p.total_draft))) {
    if (tid == 0 && seg == 0) atomicOr(p.status, SPEC_DEV_OFFSETS);
    return;
  }
  const size_t V = (size_t)p.V;
  const E* trow = static_cast<const E*>(p.target) + (size_t)q.t_row * V;
  const E* drow = static_cast<const E*>(p.draft) + (q.mode == S_RESID ? (size_t)q.d_row * V : 0);
  const float c = p.c;
  double* tot = p.segtot + (size_t)b * p.nseg;

  {
    const int e0 = seg * p.seg_elems, e1 = min(e0 + p.seg_elems, p.V);
    const double ws = segment_pass<E, VEC>(trow, drow, q.mode, q.lt2, q.ld2, c, e0, e1, nullptr);
    if (lane == 0) s_w[warp] = ws;
    __syncthreads();
    if (tid == 0) {
      double t = 0.0;
      for (int w = 0; w < kWarps; ++w) t += s_w[w];
      __stcg(tot + seg, t);
      __threadfence();
      const unsigned old = atomicAdd(p.cnt + b, 1u);
      s_last = (old + 1u == (unsigned)p.nseg) ? 1 : 0;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
  }

  // ---- the last segment block of sequence b chooses the token
  int mode = q.mode;
  if (tid == 0) {
    double Z = 0.0;
    for (int s = 0; s < p.nseg; ++s) Z += __ldcg(tot + s);
    s_mode = (mode == S_RESID && !(Z > 1e-30)) ? S_P : mode;  // zero residual: draw from p
  }
  __syncthreads();
  if (s_mode != mode) {
    mode = s_mode;
    for (int s = 0; s < p.nseg; ++s) {
      const int e0 = s * p.seg_elems, e1 = min(e0 + p.seg_elems, p.V);
      const double ws = segment_pass<E, VEC>(trow, drow, mode, q.lt2, q.ld2, c, e0, e1, nullptr);
      if (lane == 0) s_w[warp] = ws;
      __syncthreads();
      if (tid == 0) {
        double t = 0.0;
        for (int w = 0; w < kWarps; ++w) t += s_w[w];
        tot[s] = t;
      }
      __syncthreads();
    }
  }
  if (tid == 0) {
    double Z = 0.0;
    for (int s = 0; s < p.nseg; ++s) Z += __ldcg(tot + s);
    const double target = (double)q.us * Z;
    double acc = 0.0;
    int sel = -1;
    for (int s = 0; s < p.nseg; ++s) {
      const double t = __ldcg(tot + s);
      if (acc + t > target) {
        sel = s;
        break;
      }
      acc += t;
    }
    if (sel < 0) {  // only rounding can get here: take the last segment with mass
      acc = 0.0;
      for (int s = 0; s < p.nseg; ++s) {
        const double t = __ldcg(tot + s);
        if (t > 0.0) {
          sel = s;
          s_base = acc;
        }
        acc += t;
      }
      if (sel < 0) sel = 0, s_base = 0.0;
    } else {
      s_base = acc;
    }
    s_seg = sel;
    s_target = target;
  }
  __syncthreads();
  const int sel = s_seg;
  const int e0 = sel * p.seg_elems, e1 = min(e0 + p.seg_elems, p.V);
  segment_pass<E, VEC>(trow, drow, mode, q.lt2, q.ld2, c, e0, e1, s_steps);
  __syncthreads();
  const int v0 = e0 / VEC, v1 = e1 / VEC;
  const int W = (v1 - v0 + kWarps - 1) / kWarps;
  if (tid == 0) {
    const double target = s_target;
    double acc = s_base;
    int ws = -1, ss = -1, lw = -1, lst = -1;
    double lbase = acc;
    for (int w = 0; w < kWarps && ws < 0; ++w) {
      const int wb = v0 + w * W, we = min(wb + W, v1);
      const int nsteps = (we > wb) ? (we - wb + 31) / 32 : 0;
      for (int s = 0; s < nsteps; ++s) {
        const double t = (double)s_steps[w * kMaxSteps + s];
        if (acc + t > target) {
          ws = w;
          ss = s;
          break;
        }
        if (t > 0.0) {
          lw = w;
          lst = s;
          lbase = acc;
        }
        acc += t;
      }
    }
    if (ws < 0) {  // rounding: fall back to the last step with mass
      ws = lw < 0 ? 0 : lw;
      ss = lst < 0 ? 0 : lst;
      acc = lbase;
    }
    s_wsel = ws;
    s_ssel = ss;
    s_base = acc;
  }
  __syncthreads();
  if (warp == 0) {
    using io = IO<E, VEC>;
    const int wb = v0 + s_wsel * W, we = min(wb + W, v1);
    const int v = wb + s_ssel * 32 + lane;
    float w[VEC];
#pragma unroll
    for (int k = 0; k < VEC; ++k) w[k] = 0.f;
    if (v < we) {
      float ft[VEC], fd[VEC];
      io::unpack(io::load(trow, v), ft);
      if (mode == S_RESID) io::unpack(io::load(drow, v), fd);
      weights<VEC>(mode, ft, fd, q.lt2, q.ld2, c, w);
    }
    const float ls = tree_sum<VEC>(w);
    float incl = ls;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += y;
    }
    float excl = __shfl_up_sync(kFull, incl, 1);
    if (lane == 0) excl = 0.f;
    const double rem = s_target - s_base;
    const unsigned hit = __ballot_sync(kFull, (double)incl > rem && ls > 0.f);
    const unsigned pos = __ballot_sync(kFull, ls > 0.f);
    int L;
    bool exact;
    if (hit) {
      L = __ffs(hit) - 1;
      exact = true;
    } else {
      L = pos ? 31 - __clz(pos) : 0;
      exact = false;
    }
    if (lane == L) {
      int y = -1, lastpos = -1;
      float run = excl;
      for (int k = 0; k < VEC; ++k) {
        run += w[k];
        if (w[k] > 0.f) lastpos = k;
        if (exact && y < 0 && w[k] > 0.f && (double)run > rem) y = k;
      }
      if (y < 0) y = (lastpos >= 0) ? lastpos : 0;
      p.out_tok[q.t_row] = (v < we) ? v * VEC + y : e0;
    }
  }
}

}  // namespace sv
