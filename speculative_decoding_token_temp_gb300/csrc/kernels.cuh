// Device code of the draft-token verification library (sm_103a).
//
// Pipeline of one call (all on the caller's stream):
//   prologue_kernel  zeroes the per-sequence tickets and the finished-tile count, marks
//                    every sequence "pending", checks packed offsets.
//   rows_kernel      one block per (row, vocabulary chunk) tile. Streams the target row
//                    (and, for a pair, the draft row) once -- on aligned rows through a
//                    per-thread 3-stage cp.async ring in shared memory, otherwise through
//                    per-warp rings of bulk copies of whole aligned 16-byte blocks, read
//                    back at the row's phase -- and keeps per-thread online statistics: the
//                    raw maximum and its lowest index, sum_v exp((z_v - ref)/T), and for
//                    the draft row also sum_v exp((zd_v - ref_d)/T) (zd_v - zt_v).
//                    Block-reduces them into a 32-byte partial. The last tile of a
//                    sequence to finish (an atomic ticket, no waiting) merges the partials
//                    of all its rows and applies the acceptance rule, NKL, greedy or tree
//                    decision; a stochastic sequence's record for the sampler is published
//                    with release semantics.
//   sample2_kernel   (stochastic) one wave of blocks over the B sampled rows
//                    cut into 512-vector stages; starts while the tile kernel drains, each
//                    block waiting (bounded) only for its own sequences' records. Slice
//                    masses of the residual max(0, p - q) (or of p for the bonus row) go to
//                    a table; the block completing a sequence finds the inverse-CDF
//                    crossing in the table (exact fixed-point sums) and re-reads one slice.
//                    Rows off the 16-byte grid stream through per-warp bulk-copy rings as
//                    in the tile kernel.
// Every kernel is launched with programmatic dependent launch, so its blocks are resident
// before its predecessor drains, and executes griddepcontrol.wait before its first access
// to memory that earlier work on the stream reads or writes (the sampler instead polls
// the records, which it can only see after the prologue has re-armed them). The last
// kernel of a call executes griddepcontrol.wait before it exits, so it does not complete
// before the call's other kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "spec_verify.h"

#ifndef SPEC_BOUNDS_CHECK
#define SPEC_BOUNDS_CHECK 0
#endif

namespace sv {

// ---------------------------------------------------------------------------
// Bounds-checked build (SPEC_BOUNDS_CHECK=1, a debug variant of the library): every
// computed global access is first checked against its buffer -- a byte range widened to
// the 16-byte blocks that hold its first and last byte, since the vector paths read whole
// aligned blocks -- or its index against its array's length; a failed check ORs
// SPEC_DEV_BOUNDS into the status word and the access is skipped. In the ordinary build
// both checks are the constant true and generate no code.

// a buffer: its base and its length in bytes
struct Ext {
  const void* base;
  size_t bytes;
};

__device__ __forceinline__ bool in_ext(const void* p, size_t n, const Ext& e, uint32_t* status) {
#if SPEC_BOUNDS_CHECK
  const uintptr_t a = reinterpret_cast<uintptr_t>(p), b0 = reinterpret_cast<uintptr_t>(e.base);
  const uintptr_t lo = b0 & ~(uintptr_t)15, hi = (b0 + e.bytes + 15) & ~(uintptr_t)15;
  if (e.base != nullptr && a >= lo && a + n <= hi) return true;
  atomicOr(status, SPEC_DEV_BOUNDS);
  return false;
#else
  (void)p, (void)n, (void)e, (void)status;
  return true;
#endif
}

// index i of an array of n elements
__device__ __forceinline__ bool in_idx(long long i, long long n, uint32_t* status) {
#if SPEC_BOUNDS_CHECK
  if (i >= 0 && i < n) return true;
  atomicOr(status, SPEC_DEV_BOUNDS);
  return false;
#else
  (void)i, (void)n, (void)status;
  return true;
#endif
}

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr unsigned kFull = 0xffffffffu;
constexpr int kMaxRows = SPEC_MAX_GAMMA + 1;

// M_STOCH2: stochastic with a draft temperature of its own (the draft row is summed at
// both temperatures)
enum Mode : int { M_STOCH = 0, M_GREEDY = 1, M_NKL = 2, M_TREE = 3, M_STOCH2 = 4 };
__host__ __device__ constexpr bool is_stoch(int mode) { return mode == M_STOCH || mode == M_STOCH2; }
enum Kind : int { K_PAIR = 0, K_TSUM = 1, K_ARGMAX = 2 };
enum SampleMode : int { S_RESID = 0, S_P = 1 };
enum RecState : int { REC_READY = 0, REC_SKIP = 1, REC_PENDING = 2 };

// Per-tile partial statistics (32 bytes).
struct __align__(16) Partial {
  float tm, ts;   // target raw max, sum exp2((z - tm) * c)
  int tidx, bad;  // lowest index of the target max, non-finite seen
  float dm, ds;   // draft reference (<= raw max), sum exp2((zd - dm) * cd)
  float dk;       // sum exp2((zd - dm) * c) * (zd - zt)
  float ds2;      // separate draft temperature: sum exp2((zd - dm) * c); else 0
};

// What the sampler needs for one sequence (32 bytes).
struct __align__(16) SeqRec {
  int state, n, t_row, d_row;
  float lt2, ld2;  // log2 normalisers: p_v = exp2(zt_v * c - lt2), q_v = exp2(zd_v * c - ld2)
  float us;
  int mode;
};

struct RowsParams {
  const void* target;
  const void* draft;
  const int32_t* tokens;
  const float* u_accept;
  const float* u_sample;
  const int32_t* cu;
  const int32_t* row_seq;  // packed batches: the sequence of every row, written by the prologue
  const int32_t* node_tokens;
  int B, V, gamma, total_draft, total_rows, nchunks, chunk_elems, N;
  float c, invT, delta, inv_lnV;
  float cd;  // log2(e) / T_d, the draft scale (equal to c when the temperatures match)
  // policy epilogues (finalize)
  const int32_t* position;  // [B] 1-based position of the first draft, or null
  float dalpha, dmax;       // position-adaptive threshold
  int min_block;            // block-accept: shortest run, 0 = off
  int32_t* block_n;
  int32_t* block_tok;
  spec_stats_slot* stats;   // the slot of this call's bucket, or null
  int32_t* n_acc;
  int32_t* out_tok;
  float* p_x;
  float* q_x;
  float* alpha;
  float* nkl;
  uint8_t* mask;
  int32_t* g_n;
  int32_t* g_tok;
  int32_t* accept_len;
  int32_t* path_nodes;
  uint32_t* status;
  Partial* part;
  unsigned* cnt;
  SeqRec* rec;
  int depth;
  int8_t parent[SPEC_MAX_TREE_NODES];
  Ext x_target, x_draft, x_ws;  // the logit buffers and the workspace (bounds-checked build)
  int out_rows;                 // entries of out_tok and g_tok (tree: B * (depth + 1))
};

struct SampleParams {
  const void* target;
  const void* draft;
  int V, total_rows, total_draft, B;
  float c, cd;  // target and draft scales, log2(e) / T
  const SeqRec* rec;
  unsigned* cnt;
  int32_t* out_tok;
  uint32_t* status;
  float* table;       // aligned-row sampler: [B, table_stride] slice masses
  int table_stride;
  const unsigned* tiles_done;  // tiles of the tile kernel that have finished (stochastic)
  unsigned ntiles;
  // aligned-row sampler: the first nb_head blocks take seg_head stages each of the first
  // head_total stages, the remaining blocks seg_tail stages each of the rest
  long long head_total;
  int nb_head, seg_head, seg_tail;
  int ph;  // aligned-row sampler: the rows' common offset in elements within the 16-byte grid
  Ext x_target, x_draft, x_ws;  // the logit buffers and the workspace (bounds-checked build)
};

struct ProParams {
  const int32_t* cu;
  int B, gamma, total_draft;
  int32_t* row_seq;  // packed batches: [total_rows] the sequence of every row (written here), or null
  int hb;            // target rows per sequence beyond its drafts (1; the NKL call's pairs: 0)
  int total_rows;
  unsigned* cntA;  // B tickets, then the finished-tile count
  unsigned* cntB;
  SeqRec* rec;
  uint32_t* status;
  spec_stats_slot* stats;  // the slot of this call's bucket, or null
  long long bucket;
  unsigned* zero2;  // further tickets to zero (multi-draft matrix), or null
  int nzero2;
  Ext x_ws;  // the workspace (bounds-checked build)
};

// ---------------------------------------------------------------------------
// small helpers

__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ int ld_acquire_gpu(const int* a) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
  return v;
}
__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* a, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(a), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void red_add_release_gpu(unsigned* a, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void st_release_gpu(int* a, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed_gpu(int* a, int v) {
  asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float max_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

// Reductions over groups of W lanes (W = 32: the whole warp)
template <int W = 32>
__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = W / 2; o; o >>= 1) x = fmaxf(x, __shfl_xor_sync(kFull, x, o));
  return x;
}
__device__ __forceinline__ float warp_max_nan(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x = max_nan(x, __shfl_xor_sync(kFull, x, o));
  return x;
}
__device__ __forceinline__ float warp_min(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x = fminf(x, __shfl_xor_sync(kFull, x, o));
  return x;
}
template <int W = 32>
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = W / 2; o; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
  return x;
}
template <int W = 32>
__device__ __forceinline__ int warp_min_i(int x) {
#pragma unroll
  for (int o = W / 2; o; o >>= 1) x = min(x, __shfl_xor_sync(kFull, x, o));
  return x;
}
template <int W = 32>
__device__ __forceinline__ int warp_or(int x) {
#pragma unroll
  for (int o = W / 2; o; o >>= 1) x |= __shfl_xor_sync(kFull, x, o);
  return x;
}

// Barrier policies: the whole block, or only the NT consumer threads of a warp-specialised
// block (named barrier 1; the producer warp never joins it).
struct BlockSync {
  static constexpr int NT = kThreads;
  __device__ static void sync() { __syncthreads(); }
};
template <int N>
struct NamedSync {
  static constexpr int NT = N;
  __device__ static void sync() { asm volatile("bar.sync 1, %0;" ::"n"(N) : "memory"); }
};

// s was accumulated relative to max m; express it relative to M >= m.
__device__ __forceinline__ float rescale(float s, float m, float M, float c) {
  return (m == -INFINITY) ? s * 0.f : s * ex2((m - M) * c);
}

// per-thread cp.async staging of the tile kernel's aligned path
constexpr int kCS = 3;   // stages of each thread's cp.async ring (vector path)
constexpr int kCV = 4;   // 16-byte vectors per thread per stage
constexpr int kRowsSmem = kCS * kCV * kThreads * 16;  // dynamic shared memory of the vector path
// pairs at two phases: lane 31 of every warp also stages the draft vectors after its own
// (its neighbours read theirs from the next lane's slots), two per stage
constexpr int kShiftXSlot = kWarps * 2 * 16;
constexpr int kShiftSmem = kRowsSmem + kCS * kShiftXSlot;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------------------
// element access: E = uint16_t (bf16 bit patterns) or float; VEC elements per load

template <typename E, int VEC>
struct IO;

template <>
struct IO<uint16_t, 8> {
  using raw_t = uint4;
  __device__ static raw_t load(const uint16_t* row, int v) { return ld_stream16(row + (size_t)v * 8); }
  __device__ static void unpack(const raw_t& r, float (&f)[8]) {
    f[0] = __uint_as_float(r.x << 16);
    f[1] = __uint_as_float(r.x & 0xffff0000u);
    f[2] = __uint_as_float(r.y << 16);
    f[3] = __uint_as_float(r.y & 0xffff0000u);
    f[4] = __uint_as_float(r.z << 16);
    f[5] = __uint_as_float(r.z & 0xffff0000u);
    f[6] = __uint_as_float(r.w << 16);
    f[7] = __uint_as_float(r.w & 0xffff0000u);
  }
};

template <>
struct IO<float, 4> {
  using raw_t = uint4;
  __device__ static raw_t load(const float* row, int v) { return ld_stream16(row + (size_t)v * 4); }
  __device__ static void unpack(const raw_t& r, float (&f)[4]) {
    f[0] = __uint_as_float(r.x);
    f[1] = __uint_as_float(r.y);
    f[2] = __uint_as_float(r.z);
    f[3] = __uint_as_float(r.w);
  }
};

// Elements s .. s + VEC - 1 of the 2 VEC elements held by the aligned vector a and the one
// after it, b: a row's vector at another phase within the 16-byte grid. The shift is split
// into M whole 32-bit words (a template argument) and, for bf16, a half word applied by a
// byte permutation with the uniform selector sel (0x3210: none, 0x5432: the high element of
// one word, then the low element of the next).
template <typename E, int M>
__device__ __forceinline__ uint4 shift_vec(const uint4& a, const uint4& b, unsigned sel) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  if constexpr (sizeof(E) == 2) {
    static_assert(M >= 0 && M < 4, "a shift within one bf16 vector");
    return make_uint4(__byte_perm(w[M], w[M + 1], sel), __byte_perm(w[M + 1], w[M + 2], sel),
                      __byte_perm(w[M + 2], w[M + 3], sel), __byte_perm(w[M + 3], w[M + 4], sel));
  } else {
    static_assert(M > 0 && M < 4, "a shift within one fp32 vector");
    (void)sel;
    return make_uint4(w[M], w[M + 1], w[M + 2], w[M + 3]);
  }
}

// shift_vec with the whole shift s (0 < s < VEC) a runtime value: the whole words by two
// select stages (2 words, then 1), the half word (bf16) by the byte permutation. One code
// path for every shift, at a dozen more instructions per vector than the template.
template <typename E>
__device__ __forceinline__ uint4 shift_vec_rt(const uint4& a, const uint4& b, int s) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  const int m = sizeof(E) == 2 ? (s >> 1) : s;
  uint32_t u[6], v[5];
#pragma unroll
  for (int i = 0; i < 6; ++i) u[i] = (m & 2) ? w[i + 2] : w[i];
#pragma unroll
  for (int i = 0; i < 5; ++i) v[i] = (m & 1) ? u[i + 1] : u[i];
  if constexpr (sizeof(E) == 2) {
    const unsigned sel = (s & 1) ? 0x5432u : 0x3210u;
    return make_uint4(__byte_perm(v[0], v[1], sel), __byte_perm(v[1], v[2], sel), __byte_perm(v[2], v[3], sel),
                      __byte_perm(v[3], v[4], sel));
  } else {
    return make_uint4(v[0], v[1], v[2], v[3]);
  }
}

template <typename E>
__device__ __forceinline__ float elem_at(const E* row, int x);
template <>
__device__ __forceinline__ float elem_at<uint16_t>(const uint16_t* row, int x) {
  return __uint_as_float(((unsigned)__ldg(reinterpret_cast<const unsigned short*>(row) + x)) << 16);
}
template <>
__device__ __forceinline__ float elem_at<float>(const float* row, int x) {
  return __ldg(row + x);
}

// ---------------------------------------------------------------------------
// Staged rows (the multi-draft pair pass over rows that do not start on a 16-byte
// boundary: an offset base pointer, or a row length whose byte size is not a multiple of
// 16): each warp streams its own runs of a row through a private ring of shared-memory
// slots, filled by bulk copies (cp.async.bulk, completion counted in bytes on one mbarrier
// per slot) of the whole aligned 16-byte blocks that cover a run; its lanes then read
// single elements at the run's phase. The first and last block may reach up to 15 bytes before the run's first
// element or after its last; each block holds at least one element of the run, so it
// lies on the same mapped page, and the extra bytes are never used.

constexpr int kStageRowBytes = 8192;                      // one row of a pair in one block stage (twice that for a single row)
constexpr int kWarpRowBytes = kStageRowBytes / kWarps;    // a warp's run of a row of a pair in one stage
constexpr int kWarpSlot = kWarpRowBytes + 16;             // with room for the phase
constexpr int kRingPollLimit = 1 << 20;                   // bounded wait for a slot's bytes (SPEC_DEV_TIMEOUT)

// Elements of the 16-byte block holding p that precede p.
template <typename E>
__device__ __forceinline__ int phase16(const E* p) {
  return (int)((reinterpret_cast<uintptr_t>(p) & 15u) / sizeof(E));
}

// First aligned block and byte count of the blocks covering elements [e0, e0 + n) of row
// (0 bytes for n <= 0); element e0 + x then sits at element phase16(row + e0) + x of a copy.
template <typename E>
__device__ __forceinline__ uint32_t run_blocks(const E* row, int e0, int n, const void** src) {
  if (n <= 0) return 0u;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(row + e0);
  const uintptr_t b0 = a0 & ~(uintptr_t)15;
  *src = reinterpret_cast<const void*>(b0);
  return (uint32_t)((((a0 + (uintptr_t)n * sizeof(E) - 1) >> 4) - (b0 >> 4) + 1) << 4);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_arrive(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, unsigned parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// A warp's ring of kCS slots, initialised once per block. Its stages are numbered over
// the block's lifetime: stage q uses slot q % kCS, and its mbarrier completes phase
// q / kCS once the stage's bytes have landed. Every produced stage is waited for.
struct WarpRing {
  uint32_t bars;  // shared address of the warp's kCS mbarriers (8 bytes each)
  int next;       // stages produced before the current pass

  // lane 0 initialises the barriers (one arrival each: lane 0's, with the byte count)
  __device__ __forceinline__ void init(uint64_t* warp_bars) {
    bars = (uint32_t)__cvta_generic_to_shared(warp_bars);
    next = 0;
    if ((threadIdx.x & 31) == 0) {
#pragma unroll
      for (int j = 0; j < kCS; ++j) mbar_init(bars + 8u * j, 1u);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
  }
  // Called by lane 0 only: the copies of stage k (up to two runs) into slot addresses d0
  // and d1. The warp's lanes are done with the slot's previous stage (a __syncwarp before
  // this call).
  __device__ __forceinline__ void produce(int k, uint32_t d0, const void* s0, uint32_t n0, uint32_t d1,
                                          const void* s1, uint32_t n1) const {
    const uint32_t bar = bars + 8u * (uint32_t)(k % kCS);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the reads of the slot precede the copies
    mbar_expect_arrive(bar, n0 + n1);
    if (n0) bulk_copy(d0, s0, n0, bar);
    if (n1) bulk_copy(d1, s1, n1, bar);
  }
  // Every lane: waits (bounded) until stage k's bytes have landed.
  __device__ __forceinline__ void wait(int k, uint32_t* status) const {
    const uint32_t bar = bars + 8u * (uint32_t)(k % kCS);
    const unsigned parity = (unsigned)(k / kCS) & 1u;
    for (int it = 0; !mbar_try_wait(bar, parity); ++it) {
      if (it == kRingPollLimit) {
        if ((threadIdx.x & 31) == 0) atomicOr(status, SPEC_DEV_TIMEOUT);
        break;
      }
    }
  }
};

// one element of a staged copy, as float
template <typename E>
__device__ __forceinline__ float sh_elem(const E* s, int x);
template <>
__device__ __forceinline__ float sh_elem<uint16_t>(const uint16_t* s, int x) {
  return __uint_as_float(((unsigned)s[x]) << 16);
}
template <>
__device__ __forceinline__ float sh_elem<float>(const float* s, int x) {
  return s[x];
}

// ---------------------------------------------------------------------------
// packed arithmetic: two fp32 lanes per instruction (sm_100 family), 3-input min/max

// the compiler's float2 builtins (sm_100 family) pair the operands in registers itself
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
// a - b as one fused multiply-add: b * (-1) + a is exact before its single rounding
__device__ __forceinline__ float2 sub2(float2 a, float2 b) { return __ffma2_rn(b, make_float2(-1.f, -1.f), a); }
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float max3_nan(float a, float b, float c) {
  float d;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float min3(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// max of the 8 bf16 values of a 16-byte vector, taken on the packed pairs (the maximum of
// the exactly converted values; a NaN is ignored unless every value is NaN, as in vmax)
__device__ __forceinline__ float vmax_bf16x8(const uint4& r) {
  uint32_t a, b, m;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(a) : "r"(r.x), "r"(r.y));
  asm("max.bf16x2 %0, %1, %2;" : "=r"(b) : "r"(r.z), "r"(r.w));
  asm("max.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(a), "r"(b));
  return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
}
// elements 2j and 2j + 1 of a 16-byte vector of bf16, as floats
__device__ __forceinline__ float2 bf16_pair(const uint4& r, int j) {
  const uint32_t w = j == 0 ? r.x : j == 1 ? r.y : j == 2 ? r.z : r.w;
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// N-element max / min as a shallow tree of 3-input instructions (N in {1, 4, 8, 16})
template <int N>
__device__ __forceinline__ float vmax(const float (&t)[N]) {
  if constexpr (N == 16)
    return fmaxf(max3(max3(t[0], t[1], t[2]), max3(t[3], t[4], t[5]), max3(t[6], t[7], t[8])),
                 max3(max3(t[9], t[10], t[11]), max3(t[12], t[13], t[14]), t[15]));
  else if constexpr (N == 8) return max3(max3(t[0], t[1], t[2]), max3(t[3], t[4], t[5]), fmaxf(t[6], t[7]));
  else if constexpr (N == 4) return max3(t[0], t[1], fmaxf(t[2], t[3]));
  else return t[0];
}
template <int N>
__device__ __forceinline__ float vmax_nan(const float (&t)[N]) {
  if constexpr (N == 16)
    return max_nan(max3_nan(max3_nan(t[0], t[1], t[2]), max3_nan(t[3], t[4], t[5]), max3_nan(t[6], t[7], t[8])),
                   max3_nan(max3_nan(t[9], t[10], t[11]), max3_nan(t[12], t[13], t[14]), t[15]));
  else if constexpr (N == 8)
    return max3_nan(max3_nan(t[0], t[1], t[2]), max3_nan(t[3], t[4], t[5]), max_nan(t[6], t[7]));
  else if constexpr (N == 4) return max3_nan(t[0], t[1], max_nan(t[2], t[3]));
  else return t[0];
}
template <int N>
__device__ __forceinline__ float vmin(const float (&t)[N]) {
  if constexpr (N == 16)
    return fminf(min3(min3(t[0], t[1], t[2]), min3(t[3], t[4], t[5]), min3(t[6], t[7], t[8])),
                 min3(min3(t[9], t[10], t[11]), min3(t[12], t[13], t[14]), t[15]));
  else if constexpr (N == 8) return min3(min3(t[0], t[1], t[2]), min3(t[3], t[4], t[5]), fminf(t[6], t[7]));
  else if constexpr (N == 4) return min3(t[0], t[1], fminf(t[2], t[3]));
  else return t[0];
}

// ---------------------------------------------------------------------------
// per-thread online statistics.
//
// m is the exact running maximum of the raw logits (and idx the lowest index holding
// it). The sums are kept relative to a lazier reference mr <= m: mr moves (and the sums
// are rescaled) only when a new value exceeds it by more than kLazy in the exponent, so
// every term stays below 2^kLazy and the common case costs no rescale at all. Sums are
// kept as two fp32 lanes (even / odd elements) for the packed instructions.

constexpr float kLazy = 32.f;

// TAcc::g0, where the thread's maximum m lies: -1 none; >= 0 a group of whole vectors, the
// index of its first element (a multiple of the vector width) plus 1 when the group has a
// second vector, kThreads vectors further on (the streams fold vectors v and v + kThreads
// together); <= -2 the exact index i of m itself, stored as exact_idx(i) = -2 - i (an
// element folded in alone). The lowest index inside a group is found once, at the end of
// the tile, by the thread that holds the tile's maximum.
struct TAcc {
  float m, mr, mth, nmc, lo, hi;
  float2 s;
  int g0;
};
__host__ __device__ constexpr int exact_idx(int i) { return -2 - i; }
struct DAcc {
  float mr, mth, nmc;
  float2 s, k;
  float nmc2;  // separate draft temperature: the reference at the target scale
  float2 s2;   // and the draft sum at the target scale (k then uses it too)
};

__device__ __forceinline__ void init(TAcc& a) {
  a.m = -INFINITY; a.mr = -INFINITY; a.mth = -INFINITY; a.nmc = 0.f; a.lo = INFINITY; a.hi = -INFINITY;
  a.s = make_float2(0.f, 0.f); a.g0 = -1;
}
__device__ __forceinline__ void init(DAcc& a) {
  a.mr = -INFINITY; a.mth = -INFINITY; a.nmc = 0.f; a.s = make_float2(0.f, 0.f); a.k = make_float2(0.f, 0.f);
  a.nmc2 = 0.f; a.s2 = make_float2(0.f, 0.f);
}

template <int VEC>
__device__ __forceinline__ float tree_sum(const float (&e)[VEC]) {
  if constexpr (VEC == 1) {
    return e[0];
  } else if constexpr (VEC == 4) {
    return (e[0] + e[1]) + (e[2] + e[3]);
  } else {
    return ((e[0] + e[1]) + (e[2] + e[3])) + ((e[4] + e[5]) + (e[6] + e[7]));
  }
}

template <int VEC>
__device__ __forceinline__ int lowest_match(const float (&t)[VEC], float v) {
  int k = VEC - 1;
#pragma unroll
  for (int j = VEC - 2; j >= 0; --j)
    if (t[j] == v) k = j;
  return k;
}

// Element index of position k of a group whose first H elements start at e0 and whose
// remaining elements start at e1 (e1 = e0 + H for a contiguous group).
template <int H>
__device__ __forceinline__ int group_index(int k, int e0, int e1) {
  return k < H ? e0 + k : e1 + (k - H);
}

// exp2(t * c + nmc) for every element, summed into a pair of lanes (pairwise tree)
template <int VEC>
__device__ __forceinline__ float2 exp_sum2(const float (&t)[VEC], float c, float nmc, float (&e)[VEC]) {
  if constexpr (VEC == 1) {
    e[0] = ex2(fmaf(t[0], c, nmc));
    return make_float2(e[0], 0.f);
  } else {
    const float2 c2 = make_float2(c, c), n2 = make_float2(nmc, nmc);
    float2 acc[VEC / 2];
#pragma unroll
    for (int j = 0; j < VEC / 2; ++j) {
      const float2 x = fma2(make_float2(t[2 * j], t[2 * j + 1]), c2, n2);
      e[2 * j] = ex2(x.x);
      e[2 * j + 1] = ex2(x.y);
      acc[j] = make_float2(e[2 * j], e[2 * j + 1]);
    }
#pragma unroll
    for (int w = VEC / 4; w >= 1; w >>= 1)
#pragma unroll
      for (int j = 0; j < w; ++j) acc[j] = add2(acc[j], acc[j + w]);
    return acc[0];
  }
}

// Exact max. A group only records where it starts (TAcc::g0): the group's VEC elements are
// one vector from e0 (H == VEC) or two, H from e0 and H from e1 = e0 + kThreads * H (H ==
// VEC / 2); H == 0: no group is recorded (an element folded in alone, whose index the
// caller keeps).
template <int VEC, int H, bool IDX>
__device__ __forceinline__ void track_max(TAcc& a, float vm, int e0) {
  static_assert(H == 0 || H == VEC || 2 * H == VEC, "one or two vectors");
  if (IDX && H > 0) {
    if (vm > a.m) a.g0 = (H == VEC) ? e0 : (e0 | 1);
  }
  a.m = fmaxf(a.m, vm);
}

// move the sum reference when vm exceeds it by more than kLazy (rare; warp-uniform branch)
__device__ __forceinline__ void lazy_ref(float& mr, float& mth, float& nmc, float2& s, float2* k, float vm, float c) {
  const bool mv = vm > mth;
  if (__any_sync(__activemask(), mv)) {
    if (mv) {
      const float f = ex2((mr - vm) * c);
      s = make_float2(s.x * f, s.y * f);
      if (k) *k = make_float2(k->x * f, k->y * f);
      mr = vm;
      mth = vm + kLazy / c;
      nmc = -vm * c;
    }
  }
}

// The same for a draft row summed at two scales (its own cd for s, the target's c for s2
// and k): one reference, each sum rescaled at its own scale; the threshold keeps both
// exponents below kLazy.
__device__ __forceinline__ void lazy_ref2(float& mr, float& mth, float& nmc, float& nmc2, float2& s, float2& s2,
                                          float2& k, float vm, float cd, float c) {
  const bool mv = vm > mth;
  if (__any_sync(__activemask(), mv)) {
    if (mv) {
      const float fd = ex2((mr - vm) * cd), ft = ex2((mr - vm) * c);
      s = make_float2(s.x * fd, s.y * fd);
      s2 = make_float2(s2.x * ft, s2.y * ft);
      k = make_float2(k.x * ft, k.y * ft);
      mr = vm;
      mth = vm + kLazy / fmaxf(c, cd);
      nmc = -vm * cd;
      nmc2 = -vm * c;
    }
  }
}

// target row with sum (bonus row of the stochastic call); lo tracks the minimum so a
// -inf entry, which the sum alone cannot see, is still reported. IDX: record the group
// holding the maximum (for its index).
template <int VEC, int H = VEC, bool IDX = true>
__device__ __forceinline__ void tsum_update(TAcc& a, const float (&t)[VEC], int e0, float c) {
  const float vm = vmax<VEC>(t);
  a.lo = fminf(a.lo, vmin<VEC>(t));
  track_max<VEC, H, IDX>(a, vm, e0);
  lazy_ref(a.mr, a.mth, a.nmc, a.s, nullptr, vm, c);
  float e[VEC];
  a.s = add2(a.s, exp_sum2<VEC>(t, c, a.nmc, e));
}

// argmax only (greedy and tree rows): no exponentials; hi propagates NaN
template <int VEC, int H = VEC>
__device__ __forceinline__ void argmax_update(TAcc& a, const float (&t)[VEC], int e0) {
  const float vh = vmax_nan<VEC>(t);
  a.hi = max_nan(a.hi, vh);
  a.lo = fminf(a.lo, vmin<VEC>(t));
  track_max<VEC, H, true>(a, vh, e0);
}

// (target row, draft row) pair; a -inf or NaN in either makes the KL sum non-finite.
// SEPT: the draft row also has its own scale cd (q = softmax(zd / T_d)); its sum at the
// target scale c (for NKL at the target temperature) goes to s2, and k uses that scale.
template <int VEC, bool IDX, int H = VEC, bool SEPT = false>
__device__ __forceinline__ void pair_update(TAcc& a, DAcc& d, const float (&t)[VEC], const float (&z)[VEC], int e0,
                                            float c, float cd = 0.f) {
  const float tm = vmax<VEC>(t), dm = vmax<VEC>(z);
  track_max<VEC, H, IDX>(a, tm, e0);
  lazy_ref(a.mr, a.mth, a.nmc, a.s, nullptr, tm, c);
  float et[VEC], ed[VEC];
  a.s = add2(a.s, exp_sum2<VEC>(t, c, a.nmc, et));
  if constexpr (SEPT) {
    lazy_ref2(d.mr, d.mth, d.nmc, d.nmc2, d.s, d.s2, d.k, dm, cd, c);
    float eq[VEC];
    d.s = add2(d.s, exp_sum2<VEC>(z, cd, d.nmc, eq));
    d.s2 = add2(d.s2, exp_sum2<VEC>(z, c, d.nmc2, ed));
  } else {
    // the draft at its own scale cd (cd == c unless the draft's temperature differs and
    // the caller wants no NKL, which alone reads k at the target scale)
    lazy_ref(d.mr, d.mth, d.nmc, d.s, &d.k, dm, cd);
    d.s = add2(d.s, exp_sum2<VEC>(z, cd, d.nmc, ed));
  }
  if constexpr (VEC == 1) {
    d.k.x = fmaf(ed[0], z[0] - t[0], d.k.x);
  } else if constexpr (VEC <= 4) {
#pragma unroll
    for (int j = 0; j < VEC / 2; ++j) {
      const float2 dz = sub2(make_float2(z[2 * j], z[2 * j + 1]), make_float2(t[2 * j], t[2 * j + 1]));
      d.k = fma2(make_float2(ed[2 * j], ed[2 * j + 1]), dz, d.k);
    }
  } else {
    // two independent accumulation chains, folded at the end of the group
    float2 k1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < VEC / 2; j += 2) {
      const float2 dz0 = sub2(make_float2(z[2 * j], z[2 * j + 1]), make_float2(t[2 * j], t[2 * j + 1]));
      const float2 dz1 = sub2(make_float2(z[2 * j + 2], z[2 * j + 3]), make_float2(t[2 * j + 2], t[2 * j + 3]));
      d.k = fma2(make_float2(ed[2 * j], ed[2 * j + 1]), dz0, d.k);
      k1 = fma2(make_float2(ed[2 * j + 2], ed[2 * j + 3]), dz1, k1);
    }
    d.k = add2(d.k, k1);
  }
}

// ---------------------------------------------------------------------------
// block reduction of a tile into a Partial (valid in thread 0)

// Lowest index of the value m inside the group g (TAcc::g0 >= 0: its first vector, and
// the vector kThreads vectors on when bit 0 is set), re-read from the row (an L2 hit: the
// tile has just streamed it).
template <typename E, int VEC>
__device__ __forceinline__ int resolve_index(const E* row, int g, float m, const Ext* xr = nullptr,
                                             uint32_t* status = nullptr) {
  if (g < 0) return INT_MAX;
  const int g0 = g & ~1;
  float f[VEC];
  if (xr != nullptr && !in_ext(row + g0, 16, *xr, status)) return INT_MAX;
  IO<E, VEC>::unpack(ld_stream16(row + g0), f);
#pragma unroll
  for (int k = 0; k < VEC; ++k)
    if (f[k] == m) return g0 + k;
  if (!(g & 1)) return INT_MAX;
  const int g1 = g0 + kThreads * VEC;
  if (xr != nullptr && !in_ext(row + g1, 16, *xr, status)) return INT_MAX;
  IO<E, VEC>::unpack(ld_stream16(row + g1), f);
#pragma unroll
  for (int k = 0; k < VEC; ++k)
    if (f[k] == m) return g1 + k;
  return INT_MAX;
}

// row != nullptr: the target maximum's index is resolved from the recorded groups; PRE:
// the caller has already resolved it into ta.g0. SEPT: the draft sum s is at scale cd, s2
// and k at c.
// xr, status: the row's buffer for the bounds-checked build (null: unchecked).
template <class SY, typename E = float, int VEC = 1, bool SEPT = false, bool PRE = false>
__device__ __forceinline__ Partial reduce_tile(int kind, const TAcc& ta, const DAcc& da, float c,
                                               const E* row = nullptr, float cd = 0.f, const Ext* xr = nullptr,
                                               uint32_t* status = nullptr) {
  constexpr int NW = SY::NT / 32;
  __shared__ float s_m[2][NW];
  __shared__ float s_v[5][NW];
  __shared__ int s_i[NW];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float wtm = warp_max(ta.m);
  const float wdm = (kind == K_PAIR) ? warp_max(da.mr) : -INFINITY;
  if (lane == 0) {
    s_m[0][warp] = wtm;
    s_m[1][warp] = wdm;
  }
  SY::sync();
  float TM = s_m[0][0], DM = s_m[1][0];
#pragma unroll
  for (int w = 1; w < NW; ++w) {
    TM = fmaxf(TM, s_m[0][w]);
    DM = fmaxf(DM, s_m[1][w]);
  }
  static_assert(VEC > 1, "groups are whole vectors");
  int my_idx = INT_MAX;
  if (ta.m == TM) {
    if constexpr (PRE)
      my_idx = ta.g0 >= 0 ? ta.g0 : INT_MAX;
    else if (ta.g0 <= -2)
      my_idx = row ? exact_idx(ta.g0) : INT_MAX;  // exact_idx is its own inverse
    else
      my_idx = row ? resolve_index<E, VEC>(row, ta.g0, TM, xr, status) : INT_MAX;
  }
  const int wi = warp_min_i(my_idx);
  float v0 = 0.f, v1 = 0.f, v2 = 0.f, v3 = 0.f, v4 = 0.f;
  if (kind == K_ARGMAX) {
    v0 = warp_max_nan(ta.hi);
    v1 = warp_min(ta.lo);
  } else {
    // target sums are expressed relative to the exact tile maximum TM (mr <= m <= TM);
    // draft sums relative to DM, the largest draft reference
    v0 = warp_sum(rescale(ta.s.x + ta.s.y, ta.mr, TM, c));
    if (kind == K_TSUM) v1 = warp_min(ta.lo);
    if (kind == K_PAIR) {
      const float fd = (da.mr == -INFINITY) ? 0.f : ex2((da.mr - DM) * cd);
      v2 = warp_sum((da.s.x + da.s.y) * fd);
      if constexpr (SEPT) {
        const float ft = (da.mr == -INFINITY) ? 0.f : ex2((da.mr - DM) * c);
        v3 = warp_sum((da.k.x + da.k.y) * ft);
        v4 = warp_sum((da.s2.x + da.s2.y) * ft);
      } else {
        v3 = warp_sum((da.k.x + da.k.y) * fd);
      }
    }
  }
  if (lane == 0) {
    s_v[0][warp] = v0;
    s_v[1][warp] = v1;
    s_v[2][warp] = v2;
    s_v[3][warp] = v3;
    s_v[4][warp] = v4;
    s_i[warp] = wi;
  }
  SY::sync();
  Partial out;
  out.tm = TM;
  out.dm = DM;
  out.ds2 = 0.f;
  out.tidx = INT_MAX;
  out.ts = out.ds = out.dk = 0.f;
  out.bad = 0;
  if (threadIdx.x == 0) {
    int idx = INT_MAX;
    float a0 = s_v[0][0], a1 = s_v[1][0], a2 = 0.f, a3 = 0.f, a4 = 0.f;
    for (int w = 0; w < NW; ++w) idx = min(idx, s_i[w]);
    if (kind == K_ARGMAX) {
      for (int w = 1; w < NW; ++w) {
        a0 = max_nan(a0, s_v[0][w]);
        a1 = fminf(a1, s_v[1][w]);
      }
      out.bad = (isnan(a0) || a0 == INFINITY || a1 == -INFINITY) ? 1 : 0;
    } else {
      a0 = 0.f;
      for (int w = 0; w < NW; ++w) {
        a0 += s_v[0][w];
        a2 += s_v[2][w];
        a3 += s_v[3][w];
        a4 += s_v[4][w];
      }
      out.ts = a0;
      bool bad = !isfinite(a0) || !isfinite(TM);
      if (kind == K_TSUM) {
        for (int w = 1; w < NW; ++w) a1 = fminf(a1, s_v[1][w]);
        bad = bad || a1 == -INFINITY;
      } else {
        out.ds = a2;
        out.dk = a3;
        out.ds2 = a4;
        bad = bad || !isfinite(a2) || !isfinite(a3) || !isfinite(a4) || !isfinite(DM);
      }
      out.bad = bad ? 1 : 0;
    }
    out.tidx = idx;
  }
  return out;
}

// ---------------------------------------------------------------------------
// merging the partials of one row (one warp per row)

struct RowStat {
  float tm, ts, dm, ds, dk, ds2;
  int tidx, bad;
};

// NKL of a merged row pair: KL(q || p) / ln V with
// KL = (K_d / S_d - (m_d - m_t)) / T - ln(S_d / S_t), in fp32 (GB300's fp64 rate is a small
// fraction of its fp32 rate). The log of the ratio keeps the normaliser term exact to one
// rounding; the other terms are the fp32 accumulators' own size.
// SEPT: the draft sum at the target scale is ds2 (ds is at the draft's own scale).
template <bool SEPT = false>
__device__ __forceinline__ float row_nkl(const RowStat& r, float invT, float inv_lnV) {
  const float S = SEPT ? r.ds2 : r.ds;
  const float kl = (r.dk / S - (r.dm - r.tm)) * invT - logf(S / r.ts);
  return kl * inv_lnV;
}

// A row whose tiles streamed only the whole 16-byte blocks of each chunk (a row off the
// 16-byte grid, or of a length that is not a whole number of blocks): the elements of the
// partial blocks at every chunk's two ends, which no tile read, are folded into the row's
// merge, each element as a partial of its own (its value as the maximum and reference,
// sums of 1).
template <typename E>
struct RowEdges {
  const E* t = nullptr;  // the target row; null: the row has no partial blocks
  const E* d = nullptr;  // the draft row of a pair (draft statistics folded too), else null
  int ph = 0;            // the target row's offset in elements within the 16-byte grid
  int V = 0, ce = 0;     // vocabulary; chunk length (a multiple of the vector width)
  bool sums = false;     // the sums (pair and sum rows) besides the maximum and its index
  bool sept = false;     // separate draft temperature: ds2 (the draft at the target scale) too
  const Ext* xt = nullptr;  // bounds-checked build: the buffers of t and d
  const Ext* xd = nullptr;
  uint32_t* status = nullptr;
};

// ds is merged at the draft scale cd, dk and ds2 at the target scale c. A group of W
// lanes (aligned within the warp; every lane of the warp calls it) merges one row.
template <int W = 32, typename E = float>
__device__ __forceinline__ RowStat merge_row(const Partial* pp, int nchunks, float c, float cd,
                                             const RowEdges<E>& edges = RowEdges<E>()) {
  constexpr int VEC = 16 / (int)sizeof(E);
  const int lane = threadIdx.x & (W - 1);
  float tm = -INFINITY, ts = 0.f, dm = -INFINITY, ds = 0.f, dk = 0.f, ds2 = 0.f;
  int idx = INT_MAX, bad = 0;
  // one element of a partial block: index e, target value xt, draft value xd
  auto fold_elem = [&](int e, float xt, float xd) {
    bad |= (!isfinite(xt) || (edges.d != nullptr && !isfinite(xd))) ? 1 : 0;
    if (xt > tm || (xt == tm && e < idx)) idx = e;
    const float M = fmaxf(tm, xt);
    if (edges.sums) ts = rescale(ts, tm, M, c) + ex2((xt - M) * c);
    tm = M;
    if (edges.d != nullptr) {
      const float D = fmaxf(dm, xd);
      const float f0 = (dm == -INFINITY) ? 0.f : ex2((dm - D) * c);
      const float g0 = (dm == -INFINITY) ? 0.f : ex2((dm - D) * cd);
      const float f1 = ex2((xd - D) * c);
      ds = ds * g0 + ex2((xd - D) * cd);
      dk = dk * f0 + f1 * (xd - xt);
      if (edges.sept) ds2 = ds2 * f0 + f1;
      dm = D;
    }
  };
  auto elem = [&](const E* row, const Ext* x, int e) -> float {
    return (x == nullptr || in_ext(row + e, sizeof(E), *x, edges.status)) ? elem_at<E>(row, e) : 0.f;
  };
  for (int ch = lane; ch < nchunks; ch += W) {
    const float4 lo = __ldcg(reinterpret_cast<const float4*>(pp + ch));
    const float4 hi = __ldcg(reinterpret_cast<const float4*>(pp + ch) + 1);
    const float qtm = lo.x, qts = lo.y;
    const int qidx = __float_as_int(lo.z), qbad = __float_as_int(lo.w);
    const float qdm = hi.x, qds = hi.y, qdk = hi.z, qds2 = hi.w;
    bad |= qbad;
    if (qtm > tm || (qtm == tm && qidx < idx)) idx = qidx;
    const float M = fmaxf(tm, qtm);
    ts = rescale(ts, tm, M, c) + rescale(qts, qtm, M, c);
    tm = M;
    const float D = fmaxf(dm, qdm);
    const float f0 = (dm == -INFINITY) ? 0.f : ex2((dm - D) * c);
    const float f1 = (qdm == -INFINITY) ? 0.f : ex2((qdm - D) * c);
    const float g0 = (dm == -INFINITY) ? 0.f : ex2((dm - D) * cd);
    const float g1 = (qdm == -INFINITY) ? 0.f : ex2((qdm - D) * cd);
    ds = ds * g0 + qds * g1;
    dk = dk * f0 + qdk * f1;
    ds2 = ds2 * f0 + qds2 * f1;
    dm = D;
  }
  if (edges.t != nullptr) {
    // The partial blocks' elements, spread over the W lanes: chunk ch's head [e_begin, hend)
    // and tail [tbeg, e_end) -- as the tile kernel leaves them out of its stream, fewer than
    // VEC each -- take slots ch * NE ... ch * NE + NE - 1, and lane l folds slots l, l + W,
    // ... (a few loads per lane, issued together), each element as a partial of its own; the
    // lanes' states are then merged with the chunk partials' below.
    constexpr int NE = 2 * (VEC - 1);
    const int ph = edges.ph;
#pragma unroll 4
    for (int f = lane; f < nchunks * NE; f += W) {
      const int ch = f / NE, k = f - ch * NE;
      const int e_begin = ch * edges.ce, e_end = min(e_begin + edges.ce, edges.V);
      const int vf0 = (e_begin + ph + VEC - 1) / VEC, vf1 = (e_end + ph) / VEC;
      const int hend = min(e_end, vf0 * VEC - ph), tbeg = max(hend, vf1 * VEC - ph);
      const int nh = hend - e_begin, nt = e_end - tbeg;
      if (nh + nt > NE) {
        // a chunk without a whole block (a tiny vocabulary): its first slot's lane folds it all
        if (k == 0)
          for (int e = e_begin; e < e_end; ++e)
            fold_elem(e, elem(edges.t, edges.xt, e), edges.d ? elem(edges.d, edges.xd, e) : 0.f);
        continue;
      }
      const int e = k < nh ? e_begin + k : (k - nh < nt ? tbeg + (k - nh) : -1);
      if (e >= 0) fold_elem(e, elem(edges.t, edges.xt, e), edges.d ? elem(edges.d, edges.xd, e) : 0.f);
    }
  }
  RowStat r;
  r.tm = warp_max<W>(tm);
  r.tidx = warp_min_i<W>(tm == r.tm ? idx : INT_MAX);
  r.ts = warp_sum<W>(rescale(ts, tm, r.tm, c));
  r.dm = warp_max<W>(dm);
  const float fd = (dm == -INFINITY) ? 0.f : ex2((dm - r.dm) * c);
  const float gd = (dm == -INFINITY) ? 0.f : ex2((dm - r.dm) * cd);
  r.ds = warp_sum<W>(ds * gd);
  r.dk = warp_sum<W>(dk * fd);
  r.ds2 = warp_sum<W>(ds2 * fd);
  r.bad = warp_or<W>(bad) ? 1 : 0;
  return r;
}

}  // namespace sv
