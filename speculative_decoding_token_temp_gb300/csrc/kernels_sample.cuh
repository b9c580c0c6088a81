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
                                        float c, float cd, float (&w)[VEC]) {
  if (mode == S_RESID) {
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
      const float pv = ex2(fmaf(t[k], c, -lt2));
      const float qv = ex2(fmaf(d[k], cd, -ld2));
      w[k] = fmaxf(pv - qv, 0.f);
    }
  } else {
#pragma unroll
    for (int k = 0; k < VEC; ++k) w[k] = ex2(fmaf(t[k], c, -lt2));
  }
}

// ---------------------------------------------------------------------------
// Sampling.
//
// The masses of 32-vector slices of the row pair (or bonus row) are stored in `table`
// (global scratch of the sequence) in token order; the block that completes a sequence
// scans the table in fp64 and locates the slice holding the crossing
// y = min{v : C(v) > u * Z}; the slice's warp re-reads it from global memory and finds y.
// Z == 0 on a residual falls back to p of the same row.

constexpr int kSlicesPerStage = 2 * kWarps;
// Polls of a sequence record before the sampler gives up (SPEC_DEV_TIMEOUT): each is a
// 256 ns sleep and two L2 reads, so the wait is bounded at well under a second.
constexpr int kPollLimit = 1 << 18;
// Largest table the crossing search stages in shared memory (entry e sits at e + e / 32,
// which keeps the lanes' contiguous ranges on distinct banks); longer tables are read
// from global memory.
constexpr int kTableSmem = 11264;
static_assert(kTableSmem + kTableSmem / 32 <= kRowsSmem / 4, "staged table exceeds the staging buffer");

__device__ __forceinline__ int staged(int e) { return e + (e >> 5); }

// Fixed-point image of a non-negative float mass: m * 2^(150 - eM + top), eM being the
// biased exponent of the table's largest mass (at least 1). Every image is below
// 2^(24 + top), so with top = 38 - ceil(log2 n) the sum of n images stays below 2^62 and
// every sum, scan and comparison over the table is exact integer arithmetic (GB300 runs
// fp64 at a small fraction of its fp32 rate; a dependent fp64 chain here cost microseconds).
// Bits below 2^-(24 + top) of the largest mass are dropped. The sign bit is ignored
// (a -0 mass is 0).
__device__ __forceinline__ unsigned long long fixed_mass(float m, int eM, int top) {
  const unsigned bits = __float_as_uint(m) & 0x7fffffffu;
  const int ex = (int)(bits >> 23);
  const unsigned long long mant = (bits & 0x7fffffu) | (ex ? 0x800000u : 0u);
  const int sh = max(ex, 1) - eM + top;
  return sh >= 0 ? mant << sh : (sh > -24 ? mant >> -sh : 0ull);
}

// floor(u * Z) for a float u in [0, 1) and an integer Z < 2^63, exactly: u = mu * 2^-s with
// an integer mu < 2^24 and s >= 24. u >= 1 (or NaN) gives Z, u <= 0 gives 0.
__device__ __forceinline__ unsigned long long scaled_floor(float u, unsigned long long Z) {
  if (!(u < 1.f)) return Z;
  if (!(u > 0.f)) return 0ull;
  const unsigned bits = __float_as_uint(u);
  const int eu = (int)(bits >> 23);
  const unsigned long long mu = (bits & 0x7fffffu) | (eu ? 0x800000u : 0u);
  const int s = 150 - max(eu, 1);
  const unsigned long long lo = Z * mu, hi = __umul64hi(Z, mu);
  if (s >= 128) return 0ull;
  if (s >= 64) return hi >> (s - 64);
  return (lo >> s) | (hi << (64 - s));
}

struct CrossResult {
  float Z;    // total mass
  float rem;  // u * Z minus the mass before the chosen entry
  int ent;    // chosen entry
};

// Per-thread sums of the two-level crossing search sit after the staged table.
constexpr int kSumsOffset = (kTableSmem + kTableSmem / 32) * 4;
static_assert(kSumsOffset % 8 == 0 && kSumsOffset + kThreads * 8 <= kRowsSmem, "crossing sums exceed the staging buffer");
constexpr unsigned long long kMassBit = 1ull << 63;  // a thread's entries include one with mass

// Inverse-CDF crossing over the n float masses of `table` (token order), called by every
// thread of the block, on the fixed-point images: the first entry with mass whose running
// total (inclusive) exceeds u * Z; when none does (u >= 1), the last entry with mass; when
// no entry has mass, entry 0. Level 1: thread t sums its contiguous entries
// [t * per, (t + 1) * per). Level 2: warp 0 scans the 256 thread sums (lane l holds those of
// threads 8l .. 8l + 7), then the chosen lane walks its threads and the chosen thread's
// entries. The table is staged in shared memory (padded layout) when it fits, and every
// thread finds the largest mass first. Results in r, valid after return.
__device__ __forceinline__ void block_crossing(const float* table, int n, float u, unsigned char* smem, CrossResult& r,
                                               unsigned* s_max) {
  float* stage = reinterpret_cast<float*>(smem);
  unsigned long long* sums = reinterpret_cast<unsigned long long*>(smem + kSumsOffset);
  const bool fits = n <= kTableSmem;
  auto at = [&](int e) -> float { return fits ? stage[staged(e)] : __ldcg(table + e); };
  unsigned mx = 0u;
  for (int e = threadIdx.x; e < n; e += kThreads) {
    const float m = __ldcg(table + e);
    if (fits) stage[staged(e)] = m;
    mx = max(mx, __float_as_uint(m) & 0x7fffffffu);
  }
  mx = __reduce_max_sync(kFull, mx);
  if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = mx;
  __syncthreads();
  unsigned m = 0u;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) m = max(m, s_max[w]);
  const int eM = max((int)(m >> 23), 1);
  const int lg = n > 1 ? 32 - __clz(n - 1) : 0;
  const int top = 38 - lg;
  const int per = (n + kThreads - 1) / kThreads;
  {
    const int lo = min(n, (int)threadIdx.x * per), hi = min(n, lo + per);
    unsigned long long sum = 0ull;
    bool mass = false;
    for (int e = lo; e < hi; ++e) {
      const float x = at(e);
      sum += fixed_mass(x, eM, top);
      mass = mass || x > 0.f;
    }
    sums[threadIdx.x] = sum | (mass ? kMassBit : 0ull);
  }
  __syncthreads();
  if ((threadIdx.x >> 5) == 0) {
    const int lane = threadIdx.x & 31;
    constexpr int TPL = kThreads / 32;  // threads per lane
    unsigned long long v[TPL];
    unsigned tmass = 0u;
    unsigned long long lsum = 0ull;
#pragma unroll
    for (int j = 0; j < TPL; ++j) {
      const unsigned long long x = sums[lane * TPL + j];
      v[j] = x & ~kMassBit;
      if (x & kMassBit) tmass |= 1u << j;
      lsum += v[j];
    }
    unsigned long long incl = lsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += y;
    }
    const unsigned long long Z = __shfl_sync(kFull, incl, 31);
    const unsigned long long excl = incl - lsum;
    const unsigned long long target = scaled_floor(u, Z);
    // integer totals: A + q > floor(u Z) exactly when A + q > u Z
    const unsigned hit = __ballot_sync(kFull, incl > target);
    const unsigned pos = __ballot_sync(kFull, tmass != 0u);
    const int L = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : 0);
    if (lane == L) {
      // the thread: the first whose sum passes the target, else the last with mass
      unsigned long long acc = excl, tb = excl;
      int T = -1;
#pragma unroll
      for (int j = 0; j < TPL; ++j) {
        if (hit) {
          if (T < 0 && acc + v[j] > target) {
            T = L * TPL + j;
            tb = acc;
          }
        } else if (tmass & (1u << j)) {
          T = L * TPL + j;
          tb = acc;
        }
        acc += v[j];
      }
      if (T < 0) T = L * TPL;
      // the entry of thread T
      const int lo = min(n, T * per), hi = min(n, lo + per);
      unsigned long long a = tb, b = tb, lastb = tb;
      int ent = -1, last = -1;
      for (int e = lo; e < hi; ++e) {
        const float x = at(e);
        const unsigned long long q = fixed_mass(x, eM, top);
        if (x > 0.f) {
          last = e;
          lastb = a;
          if (hit && a + q > target) {
            ent = e;
            b = a;
            break;
          }
        }
        a += q;
      }
      if (ent < 0) {
        ent = last >= 0 ? last : lo;
        b = last >= 0 ? lastb : tb;
      }
      const int sc = eM - 150 - top;  // image -> mass
      r.Z = ldexpf(__ull2float_rn(Z), sc);
      r.rem = ldexpf(__ull2float_rn(target >= b ? target - b : 0ull), sc);
      r.ent = min(ent, max(n - 1, 0));
    }
  }
  __syncthreads();  // the next pass's copies may rewrite this shared memory
}

// The 16-byte blocks covering row [row, row + V) lie in buffer x (bounds-checked build; the
// mass passes and the slice re-read read nothing else of the row).
template <typename E>
__device__ __forceinline__ bool row_ok(const E* row, int V, const Ext& x, uint32_t* status) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(row);
  const uintptr_t lo = a & ~(uintptr_t)15, hi = (a + (uintptr_t)V * sizeof(E) + 15) & ~(uintptr_t)15;
  return in_ext(reinterpret_cast<const void*>(lo), (size_t)(hi - lo), x, status);
}

// Elements e0 + j outside the row [0, V) weigh nothing.
template <int VEC>
__device__ __forceinline__ void edge_mask(float (&ft)[VEC], float (&fd)[VEC], int e0, int V) {
#pragma unroll
  for (int j = 0; j < VEC; ++j)
    if (e0 + j < 0 || e0 + j >= V) ft[j] = fd[j] = -INFINITY;
}

// Masses of stages [k0, k1) of the row pair (or row): in each 512-vector stage thread t
// takes vectors t and t + 256 (lane-contiguous, so every copy instruction moves 512
// consecutive bytes) through its private cp.async ring; entry (2k + h) * kWarps + w of
// `table` receives the mass of warp w's 32-vector slice of half h of stage k -- token
// order. PH: trow and drow are the rows' aligned bases (row element e is their element
// e + ph), and the elements of the first and last vectors outside the row weigh 0.
template <typename E, int VEC, bool PH>
__device__ __forceinline__ void mass_pass(const E* trow, const E* drow, int mode, float lt2, float ld2, float c, float cd,
                                          int NV, int k0, int k1, float* table, unsigned char* smem, int ph, int V) {
  constexpr unsigned SLOT = kCV * kThreads * 16;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(smem) + 16u * t;
  const int nst = k1 - k0;
  auto issue = [&](int k) {
    if (k < nst) {
      const uint32_t slot = sbase + (uint32_t)(k % kCS) * SLOT;
#pragma unroll
      for (int j = 0; j < kCV; ++j) {
        if (j >= 2 && mode != S_RESID) continue;
        const int v = (k0 + k) * 2 * kThreads + (j & 1) * kThreads + t;
        if (v < NV) cp_async16(slot + (uint32_t)(j * kThreads * 16), ((j >= 2) ? drow : trow) + (size_t)v * VEC);
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
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int v = (k0 + k) * 2 * kThreads + h * kThreads + t;
      float ls = 0.f;
      if (v < NV) {
        float ft[VEC], fd[VEC], w[VEC];
        IO<E, VEC>::unpack(q[h * kThreads], ft);
        if (mode == S_RESID) IO<E, VEC>::unpack(q[(2 + h) * kThreads], fd);
        if (PH && (v == 0 || v == NV - 1)) edge_mask<VEC>(ft, fd, v * VEC - ph, V);
        weights<VEC>(mode, ft, fd, lt2, ld2, c, cd, w);
        ls = tree_sum<VEC>(w);
      }
      const float ws = warp_sum(ls);
      if (lane == 0) __stcg(table + ((size_t)(k0 + k) * 2 + h) * kWarps + warp, ws);
    }
  }
  cp_wait<0>();
}

// The warp that owns table entry `ent` (stage k, half h, warp w) re-reads its 32-vector
// slice -- one vector per lane, in token order -- and returns the token where the
// running mass passes rem. PH: trow and drow are the rows' aligned bases (row element e is
// their element e + ph).
template <typename E, int VEC, bool PH>
__device__ __forceinline__ int slice_token(const E* trow, const E* drow, int mode, float lt2, float ld2, float c, float cd,
                                           int V, int NV, int ent, float rem, int ph = 0) {
  const int lane = threadIdx.x & 31;
  const int k = ent / kSlicesPerStage, h = (ent / kWarps) & 1, w = ent % kWarps;
  const int v = k * 2 * kThreads + h * kThreads + w * 32 + lane;
  float wt[VEC];
#pragma unroll
  for (int j = 0; j < VEC; ++j) wt[j] = 0.f;
  if (v < NV) {
    float ft[VEC], fd[VEC];
    IO<E, VEC>::unpack(ld_stream16(trow + (size_t)v * VEC), ft);
    if (mode == S_RESID) IO<E, VEC>::unpack(ld_stream16(drow + (size_t)v * VEC), fd);
    if (PH && (v == 0 || v == NV - 1)) edge_mask<VEC>(ft, fd, v * VEC - ph, V);
    weights<VEC>(mode, ft, fd, lt2, ld2, c, cd, wt);
  }
  const float ls = tree_sum<VEC>(wt);
  float incl = ls;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  float excl = __shfl_up_sync(kFull, incl, 1);
  if (lane == 0) excl = 0.f;
  const unsigned hit = __ballot_sync(kFull, incl > rem && ls > 0.f);
  const unsigned pos = __ballot_sync(kFull, ls > 0.f);
  const int L = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : 0);
  int tok = 0;
  if (lane == L) {
    int y = -1, lastpos = -1;
    float run = excl;
    for (int j = 0; j < VEC; ++j) {
      run += wt[j];
      if (wt[j] > 0.f) {
        lastpos = j;
        if (hit && y < 0 && run > rem) y = j;
      }
    }
    if (y < 0) y = lastpos >= 0 ? lastpos : 0;
    tok = v * VEC + y - ph;
    if (tok >= V) tok = V - 1;
    if (tok < 0) tok = 0;
  }
  return __shfl_sync(kFull, tok, L);
}

// ---------------------------------------------------------------------------
// Residual masses of a row pair whose two rows sit at different offsets within the 16-byte
// grid (pht for the target row, phd for the draft row; the rows' aligned bases trv, drv):
// the aligned sampler's stages over the target's vectors v < NVt, and for each the draft's
// elements at the same row indices, which lie in the draft's aligned vectors w = v + dw
// and w + 1 (dw * VEC + s = phd - pht, 0 < s < VEC), shifted in registers (one code path
// for every shift: a block samples sequences of different shifts one after another, and
// per-shift instances measured slower here through the instruction cache): each lane copies its own w
// (when it is one of the draft row's NVd blocks), takes w + 1 from the next lane's slot
// after a warp barrier, and lane 31 copies its own w + 1 into a ring beside the main one
// (kShiftXSlot bytes per stage). Only the first and last target vectors hold elements
// outside the row, and only their draft elements can come from blocks that were not
// copied; those elements are masked. Elements outside the row weigh 0.
template <typename E, int VEC>
__device__ __forceinline__ void mass_pass_shifted(int sft, const E* trv, const E* drv, int dw, float lt2, float ld2,
                                                  float c, float cd, int NVt, int NVd, int k0, int k1, float* table,
                                                  unsigned char* smem, int pht, int V) {
  constexpr unsigned SLOT = kCV * kThreads * 16;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(smem) + 16u * t;
  unsigned char* xring = smem + kCS * SLOT;
  const uint32_t xbase = (uint32_t)__cvta_generic_to_shared(xring) + (uint32_t)(warp * 32);
  const int nst = k1 - k0;
  auto issue = [&](int k) {
    if (k < nst) {
      const uint32_t slot = sbase + (uint32_t)(k % kCS) * SLOT;
      const uint32_t xs = xbase + (uint32_t)(k % kCS) * kShiftXSlot;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int v = (k0 + k) * 2 * kThreads + h * kThreads + t, w = v + dw;
        if (v < NVt) cp_async16(slot + (uint32_t)(h * kThreads * 16), trv + (size_t)v * VEC);
        if (w >= 0 && w < NVd) cp_async16(slot + (uint32_t)((2 + h) * kThreads * 16), drv + (ptrdiff_t)w * VEC);
        if (lane == 31 && w + 1 >= 0 && w + 1 < NVd) cp_async16(xs + 16u * h, drv + (ptrdiff_t)(w + 1) * VEC);
      }
    }
    cp_commit();
  };
  __syncwarp();  // the warp's lanes are done with every slot (the previous pass, the crossing search)
#pragma unroll
  for (int k = 0; k < kCS - 1; ++k) issue(k);
  for (int k = 0; k < nst; ++k) {
    __syncwarp();  // every lane has read the slot issue() refills
    issue(k + kCS - 1);
    cp_wait<kCS - 1>();
    __syncwarp();  // the lanes' copies of stage k are visible to the whole warp
    const uint4* q = reinterpret_cast<const uint4*>(smem + (size_t)(k % kCS) * SLOT) + t;
    const uint4* qx = reinterpret_cast<const uint4*>(xring + (size_t)(k % kCS) * kShiftXSlot) + warp * 2;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int v = (k0 + k) * 2 * kThreads + h * kThreads + t;
      float ls = 0.f;
      if (v < NVt) {
        float ft[VEC], fd[VEC], w[VEC];
        IO<E, VEC>::unpack(q[h * kThreads], ft);
        const uint4 n = lane < 31 ? q[(2 + h) * kThreads + 1] : qx[h];
        IO<E, VEC>::unpack(shift_vec_rt<E>(q[(2 + h) * kThreads], n, sft), fd);
        if (v == 0 || v == NVt - 1) edge_mask<VEC>(ft, fd, v * VEC - pht, V);
        weights<VEC>(S_RESID, ft, fd, lt2, ld2, c, cd, w);
        ls = tree_sum<VEC>(w);
      }
      const float ws = warp_sum(ls);
      if (lane == 0) __stcg(table + ((size_t)(k0 + k) * 2 + h) * kWarps + warp, ws);
    }
  }
  cp_wait<0>();
}

// The slice re-read of a row pair at two offsets: lane l takes target vector v and the
// draft's vectors w = v + dw and w + 1 straight from global memory (each when it is one of
// the row's blocks), shifted as in mass_pass_sh; then as slice_token.
template <typename E, int VEC>
__device__ __forceinline__ int slice_token_shifted(int s, const E* trv, const E* drv, int dw, float lt2, float ld2,
                                                   float c, float cd, int V, int NVt, int NVd, int ent, float rem,
                                                   int pht) {
  const int lane = threadIdx.x & 31;
  const int k = ent / kSlicesPerStage, h = (ent / kWarps) & 1, w = ent % kWarps;
  const int v = k * 2 * kThreads + h * kThreads + w * 32 + lane;
  float wt[VEC];
#pragma unroll
  for (int j = 0; j < VEC; ++j) wt[j] = 0.f;
  if (v < NVt) {
    float ft[VEC], fd[VEC];
    IO<E, VEC>::unpack(ld_stream16(trv + (size_t)v * VEC), ft);
    const int wv = v + dw;
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    const uint4 a = (wv >= 0 && wv < NVd) ? ld_stream16(drv + (ptrdiff_t)wv * VEC) : zero;
    const uint4 b = (wv + 1 >= 0 && wv + 1 < NVd) ? ld_stream16(drv + (ptrdiff_t)(wv + 1) * VEC) : zero;
    const uint4 sh = shift_vec_rt<E>(a, b, s);
    IO<E, VEC>::unpack(sh, fd);
    if (v == 0 || v == NVt - 1) edge_mask<VEC>(ft, fd, v * VEC - pht, V);
    weights<VEC>(S_RESID, ft, fd, lt2, ld2, c, cd, wt);
  }
  const float ls = tree_sum<VEC>(wt);
  float incl = ls;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  float excl = __shfl_up_sync(kFull, incl, 1);
  if (lane == 0) excl = 0.f;
  const unsigned hit = __ballot_sync(kFull, incl > rem && ls > 0.f);
  const unsigned pos = __ballot_sync(kFull, ls > 0.f);
  const int L = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : 0);
  int tok = 0;
  if (lane == L) {
    int y = -1, lastpos = -1;
    float run = excl;
    for (int j = 0; j < VEC; ++j) {
      run += wt[j];
      if (wt[j] > 0.f) {
        lastpos = j;
        if (hit && y < 0 && run > rem) y = j;
      }
    }
    if (y < 0) y = lastpos >= 0 ? lastpos : 0;
    tok = v * VEC + y - pht;
    if (tok >= V) tok = V - 1;
    if (tok < 0) tok = 0;
  }
  return __shfl_sync(kFull, tok, L);
}

// Aligned-row sampler. The B rows to sample are cut into 512-vector stages, B * nst of
// them in sequence order, and every block streams a contiguous range of them: long ranges
// for the sequences the tile kernel decides first, short ones for the last few, so that
// the work left once the last sequence is decided is spread over many blocks (the host
// sizes the grid to one wave of resident blocks). A range may cover the end of one sequence and
// the start of the next; for each part the block adds the part's stage count to the
// sequence's ticket, and the block whose part completes the nst stages scans the
// sequence's table and draws its token.
// PH (aligned sampler): rows at one offset within the 16-byte grid, p.ph. SH (with PH):
// every row at its own offset (p.ph = VEC - 1 sizes the stages for the largest); a row
// pair whose two rows differ in offset takes the shifted pass.
template <typename E, int VEC, bool PH = false, bool SH = false>
__global__ void __launch_bounds__(kThreads, 4) sample2_kernel(const __grid_constant__ SampleParams p) {
  static_assert(!SH || PH, "rows at their own offsets are phased rows");
  extern __shared__ __align__(128) unsigned char dsm[];
  // No griddepcontrol.wait: the grid starts while the tile kernel drains, and each part
  // waits only for its own sequence's record (published with release semantics by the
  // sequence's last tile; the prologue re-armed it before this grid could launch).
  __shared__ SeqRec s_rec;
  __shared__ int s_last;
  __shared__ CrossResult sc;
  __shared__ unsigned s_max[kWarps];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const size_t V = (size_t)p.V;
  const int ph = PH ? p.ph : 0;               // the rows' offset within the 16-byte grid
  const int NV = (p.V + ph + VEC - 1) / VEC;  // vectors of a row's aligned blocks
  const int nst = (NV + 2 * kThreads - 1) / (2 * kThreads);
  const long long total = (long long)p.B * nst;
  long long u0, u1;
  if ((int)blockIdx.x < p.nb_head) {
    u0 = (long long)blockIdx.x * p.seg_head;
    u1 = min(p.head_total, u0 + p.seg_head);
  } else {
    u0 = p.head_total + (long long)((int)blockIdx.x - p.nb_head) * p.seg_tail;
    u1 = min(total, u0 + p.seg_tail);
  }
  for (long long u = u0; u < u1;) {
    const int b = (int)(u / nst);
    const int k0 = (int)(u - (long long)b * nst);
    const int k1 = (int)min((long long)nst, k0 + (u1 - u));
    u += k1 - k0;
    if (!in_ext(p.rec + b, sizeof(SeqRec), p.x_ws, p.status) ||
        !in_ext(p.table + (size_t)b * p.table_stride, sizeof(float) * p.table_stride, p.x_ws, p.status) ||
        !in_ext(p.cnt + b, sizeof(unsigned), p.x_ws, p.status))
      continue;  // (uniform over the block)
    if (tid == 0) {
      int st = ld_acquire_gpu(&p.rec[b].state);
      for (int it = 0; st == REC_PENDING && it < kPollLimit; ++it) {
        if ((unsigned)ld_acquire_gpu(reinterpret_cast<const int*>(p.tiles_done)) == p.ntiles) {
          // every tile has finished: a record still pending now will never be published
          st = ld_acquire_gpu(&p.rec[b].state);
          if (st == REC_PENDING) st = REC_SKIP;
          break;
        }
        __nanosleep(256);
        st = ld_acquire_gpu(&p.rec[b].state);
      }
      if (st == REC_PENDING) atomicOr(p.status, SPEC_DEV_TIMEOUT);
      const int4 a = __ldcg(reinterpret_cast<const int4*>(p.rec + b));
      const int4 z = __ldcg(reinterpret_cast<const int4*>(p.rec + b) + 1);
      s_rec.state = st;
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
    __syncthreads();  // s_rec may be rewritten for the next part
    if (q.state != REC_READY) continue;
    if (q.t_row < 0 || q.t_row >= p.total_rows || (q.mode == S_RESID && (q.d_row < 0 || q.d_row >= p.total_draft))) {
      if (tid == 0) atomicOr(p.status, SPEC_DEV_OFFSETS);
      continue;
    }
    const E* trow = static_cast<const E*>(p.target) + (size_t)q.t_row * V;
    const E* drow = static_cast<const E*>(p.draft) + (q.mode == S_RESID ? (size_t)q.d_row * V : 0);
    if (!row_ok(trow, p.V, p.x_target, p.status) || (q.mode == S_RESID && !row_ok(drow, p.V, p.x_draft, p.status)))
      continue;
    float* table = p.table + (size_t)b * p.table_stride;
    // SH: the target row's own offset and vectors, and for a residual the draft row's shift
    // against it (sft = 0: one offset, the phased pass)
    int pht = ph, phd = ph, NVt = NV, NVd = NV, sft = 0, dwv = 0;
    if constexpr (SH) {
      pht = phase16(trow);
      phd = q.mode == S_RESID ? phase16(drow) : pht;
      NVt = (p.V + pht + VEC - 1) / VEC;
      NVd = (p.V + phd + VEC - 1) / VEC;
      sft = (phd - pht + VEC) % VEC;
      dwv = (phd - pht - sft) / VEC;
    }
    if (SH && sft != 0)
      mass_pass_shifted<E, VEC>(sft, trow - pht, drow - phd, dwv, q.lt2, q.ld2, p.c, p.cd, NVt, NVd, k0, k1, table, dsm,
                                pht, p.V);
    else
      mass_pass<E, VEC, PH>(trow - pht, drow - pht, q.mode, q.lt2, q.ld2, p.c, p.cd, NVt, k0, k1, table, dsm, pht, p.V);
    __syncthreads();  // orders every warp's table entries before thread 0's fence
    if (tid == 0) {
      // release: the block's table entries before its ticket; acquire: the other blocks'
      // entries before this block's reads
      const unsigned part = (unsigned)(k1 - k0);
      const unsigned old = atom_add_acq_rel_gpu(p.cnt + b, part);
      s_last = (old + part == (unsigned)nst) ? 1 : 0;
    }
    __syncthreads();
    if (!s_last) continue;
    int mode = q.mode;
    const int nent = nst * kSlicesPerStage;
    for (int attempt = 0; attempt < 2; ++attempt) {
      block_crossing(table, nent, q.us, dsm, sc, s_max);
      if (!(mode == S_RESID && !(sc.Z > 1e-30f))) break;
      mode = S_P;  // zero residual: the masses of p of the same row, whole row in this block
      mass_pass<E, VEC, PH>(trow - pht, drow - pht, mode, q.lt2, q.ld2, p.c, p.cd, NVt, 0, nst, table, dsm, pht, p.V);
      __syncthreads();
    }
    const int ent = sc.ent;
    if (warp == ent % kWarps) {
      const int y = (SH && mode == S_RESID && sft != 0)
                        ? slice_token_shifted<E, VEC>(sft, trow - pht, drow - phd, dwv, q.lt2, q.ld2, p.c, p.cd, p.V,
                                                      NVt, NVd, ent, sc.rem, pht)
                        : slice_token<E, VEC, PH>(trow - pht, drow - pht, mode, q.lt2, q.ld2, p.c, p.cd, p.V,
                                                          NVt, ent, sc.rem, pht);
      if (lane == 0 && in_idx(q.t_row, p.total_rows, p.status)) p.out_tok[q.t_row] = y;
    }
    __syncthreads();
  }
  // This grid does not complete before the tile kernel has: whatever follows on the
  // stream and waits for this grid sees every write of the call.
  griddep_wait();
}

}  // namespace sv
