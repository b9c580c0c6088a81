// Host entry points of the C ABI declared in include/spec_verify.h: argument checks,
// workspace layout, path selection (16-byte vectors or scalar) and launches.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "kernels.cuh"
#include "kernels_rows.cuh"
#include "kernels_multi.cuh"
#include "kernels_sample.cuh"
#include "plan.h"
#include "spec_verify.h"

#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <initializer_list>
#include <mutex>

namespace sv {
namespace {

inline long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }
inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// One wave of resident blocks of each kernel family on a device: the SM count times the
// blocks of that kernel one SM holds (cudaOccupancyMaxActiveBlocksPerMultiprocessor at its
// block size and shared memory), looked up once per device. bound() is the largest wave
// the workspace layout allows for (plan::kMaxWaveSlots), used where no device is involved
// (workspace sizes).
struct Geometry {
  long long tile_slots;      // rows_kernel tiles (one wave)
  long long fused_slots;     // multi_rows_kernel tiles
  long long sampler_blocks;  // sample2_kernel blocks
  static Geometry bound() {
    Geometry g;
    g.tile_slots = g.fused_slots = g.sampler_blocks = plan::kMaxWaveSlots;
    return g;
  }
};

struct Layout {
  size_t cntA, cntB, rec, part, table, seqmap, total;
  int nchunks, chunk_elems, table_stride;
  int cap_nchunks;  // chunks per row the partials are sized for (the largest wave's chunking)
  long long rows;
};

// The aligned-row sampler keeps one float per 32-vector (one warp, one half-stage) slice
// of a row's aligned blocks: 16 per 512-vector stage, with room for rows at any offset
// within the 16-byte grid.
int table_stride_for(int V, spec_dtype dt) {
  const int vec = dt == SPEC_BF16 ? 8 : 4;
  const long long nv = ceil_div((long long)V + vec - 1, vec);
  return (int)(ceil_div(nv, 2 * kThreads) * kSlicesPerStage);
}

// fused_k > 0: fused multi-draft tiles, each holding the rows of fused_k candidates.
// max_chunk: the longest vocabulary chunk of a tile. 0 = the measured best: 65536 tokens
// for single-row tiles and for the stochastic call's pairs (256 KB pair tiles: fewer
// tile epilogues; 185.6 against 191.7 us at the headline, same box), 49152 for the NKL
// call's pairs (150.3 us, against 152.0 with 32768 and 155.4 with 65536) unless a whole
// row fits in 65536 (B=256, gamma=8, V=50257: whole rows 74.4 against 79.1 us in two
// chunks, which also folds two sets of partial edge blocks per row).
// geo: the device's waves; the chunking follows them, while the offsets (and the total)
// are those of the largest wave allowed, so the workspace size does not depend on the
// device.
Layout layout(int B, int V, long long rows, bool sample, bool single_rows = false, spec_dtype dt = SPEC_F32,
              int max_chunk = 0, int fused_k = 0, const Geometry& geo = Geometry::bound()) {
  Layout L;
  L.rows = rows;
  const long long trows = fused_k > 0 ? rows / fused_k : rows;  // tiles per chunk
  const int mc = max_chunk > 0 ? max_chunk : ((single_rows || sample || V <= 65536) ? 65536 : 49152);
  const plan::Chunking run = plan::chunking(V, trows, mc, fused_k > 0 ? geo.fused_slots : geo.tile_slots);
  const plan::Chunking cap = plan::chunking(V, trows, mc, plan::kMaxWaveSlots);
  L.nchunks = run.nchunks;
  L.chunk_elems = run.chunk_elems;
  L.cap_nchunks = cap.nchunks;
  size_t off = 0;
  L.cntA = off;  // B tickets, then the count of finished tiles
  off = align256(off + sizeof(unsigned) * ((size_t)B + 1));
  L.cntB = off;
  off = align256(off + sizeof(unsigned) * (size_t)B);
  L.rec = off;
  off = align256(off + sizeof(SeqRec) * (size_t)B);
  L.part = off;
  off = align256(off + sizeof(Partial) * (size_t)(rows * cap.nchunks));
  L.table_stride = sample ? table_stride_for(V, dt) : 0;
  L.table = off;
  off = align256(off + sizeof(float) * (size_t)B * (size_t)L.table_stride);
  L.seqmap = off;  // packed batches: the sequence of every row
  off = align256(off + sizeof(int32_t) * (size_t)rows);
  L.total = off;
  return L;
}

long long rows_for(spec_mode mode, const spec_batch& g) {
  if (mode == SPEC_MODE_NKL) return g.total_draft;
  return (long long)g.total_draft + g.B;
}

bool aligned16(const void* p) { return p == nullptr || ((uintptr_t)p & 15u) == 0; }

// A workspace pointer that is set, 256-byte aligned and of at least `need` bytes.
bool workspace_ok(const void* ws, size_t bytes, size_t need) {
  return ws != nullptr && bytes >= need && ((uintptr_t)ws & 255u) == 0;
}

// every non-null pointer of the list on an n-byte boundary (its element size)
bool aligned_to(size_t n, std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (p != nullptr && ((uintptr_t)p % n) != 0) return false;
  return true;
}

size_t elem_bytes(spec_dtype dt) { return dt == SPEC_BF16 ? 2 : 4; }

spec_status check_batch(const spec_batch& g) {
  if (g.B < 0 || g.V < 1 || g.gamma < 0 || g.gamma > SPEC_MAX_GAMMA || g.total_draft < 0) return SPEC_ERR_INVALID_ARG;
  if (g.cu_draft == nullptr && (long long)g.B * g.gamma != g.total_draft) return SPEC_ERR_INVALID_ARG;
  if ((long long)g.total_draft > (long long)g.B * g.gamma) return SPEC_ERR_INVALID_ARG;
  // row indices and element offsets stay inside int / size_t arithmetic
  if ((long long)g.total_draft + g.B > (1LL << 30)) return SPEC_ERR_INVALID_ARG;
  if (g.V > (1 << 26)) return SPEC_ERR_INVALID_ARG;
  return SPEC_OK;
}

// Launch with programmatic stream serialisation (pdl = true): the kernel may start while
// its predecessor in the stream drains; it touches memory that earlier stream work reads
// or writes only after griddepcontrol.wait (or, in the sampler, after acquiring a record
// that can only be published after the wait).
template <typename K, typename P>
cudaError_t launch(K kernel, dim3 grid, dim3 block, cudaStream_t stream, const P& params, bool pdl) {
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, params);
}

template <typename K, typename P>
cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, cudaStream_t stream, const P& params) {
  return launch(kernel, grid, block, stream, params, true);
}

// slot of a statistics bucket (labels may be negative)
int stats_slot(int64_t bucket) {
  const int64_t m = bucket % SPEC_STATS_SLOTS;
  return (int)(m < 0 ? m + SPEC_STATS_SLOTS : m);
}

// Extra tickets the prologue of a call zeroes (the multi-draft matrix's).
struct ZeroRegion {
  unsigned* ptr = nullptr;
  int n = 0;
};

// hb: target rows per sequence beyond its drafts (1: the bonus row; 0 for the NKL call,
// whose rows are the draft pairs).
cudaError_t launch_prologue(const spec_batch& g, const Layout& L, char* ws, uint32_t* status, cudaStream_t stream,
                            const spec_options* opt = nullptr, ZeroRegion z = ZeroRegion(), int hb = 1) {
  ProParams pp;
  pp.cu = g.cu_draft;
  pp.B = g.B;
  pp.gamma = g.gamma;
  pp.total_draft = g.total_draft;
  pp.cntA = reinterpret_cast<unsigned*>(ws + L.cntA);
  pp.cntB = reinterpret_cast<unsigned*>(ws + L.cntB);
  pp.rec = reinterpret_cast<SeqRec*>(ws + L.rec);
  pp.status = status;
  pp.x_ws = Ext{ws, L.total};
  pp.stats = (opt && opt->stats) ? &opt->stats->slot[stats_slot(opt->stats_bucket)] : nullptr;
  pp.bucket = opt ? (long long)opt->stats_bucket : 0;
  pp.zero2 = z.ptr;
  pp.nzero2 = z.n;
  pp.row_seq = g.cu_draft != nullptr ? reinterpret_cast<int32_t*>(ws + L.seqmap) : nullptr;
  pp.total_rows = (int)L.rows;
  pp.hb = hb;
  const int threads = g.B > z.n ? g.B : z.n;
  return launch(prologue_kernel, dim3((unsigned)ceil_div(threads, kThreads)), dim3(kThreads), stream, pp, true);
}

// The vector path of rows_kernel stages its loads in kRowsSmem bytes of dynamic shared
// memory, above the default 48 KB limit: the limit is raised once per (kernel, device).
constexpr int kAttrDevices = 64;
constexpr int kTailSeqs = 16;   // sequences the sampler splits finely (the last decided)
constexpr int kTailStages = 1;  // their shortest range, in 512-vector stages (small batches split the last sequences finely)

template <typename K>
cudaError_t ensure_smem_attr(K kernel, std::atomic<unsigned long long>& done, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kAttrDevices) return cudaErrorInvalidDevice;
  const unsigned long long bit = 1ull << dev;
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

template <typename E, int VEC, int MODE, bool PH = false, bool SH = false>
cudaError_t launch_rows_t(const RowsParams& rp, long long tiles, cudaStream_t stream) {
  auto kern = rows_kernel<E, VEC, MODE, PH, SH>;
  const int smem = SH ? kShiftSmem : kRowsSmem;
  static std::atomic<unsigned long long> done{0};
  const cudaError_t e = ensure_smem_attr(kern, done, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3((unsigned)tiles);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, rp);
}

// One NVTX range per entry point, over the host side of the call (argument checks and the
// launches it enqueues), so that a timeline shows which calls issued which kernels. With no
// tool attached a push or pop costs a function-pointer test.
struct ApiRange {
  explicit ApiRange(const char* name) { nvtxRangePushA(name); }
  ~ApiRange() { nvtxRangePop(); }
  ApiRange(const ApiRange&) = delete;
  ApiRange& operator=(const ApiRange&) = delete;
};

// The tile kernel's layout of the rows: every row on the 16-byte grid (vector tiles); rows
// off the grid with one offset within it for both rows of every pair (phased vector tiles:
// each tile applies its row's offset; single rows always qualify); pairs whose two rows sit
// at different offsets within the grid (phased tiles whose draft vectors are shifted to the
// target's offset).
enum RowPath { P_VEC, P_PHASED, P_SHIFT };

template <int MODE>
cudaError_t launch_rows(bool bf16, RowPath path, const RowsParams& rp, long long tiles, cudaStream_t stream) {
  if constexpr (MODE == M_GREEDY || MODE == M_TREE) {
    if (bf16) return path == P_VEC ? launch_rows_t<uint16_t, 8, MODE>(rp, tiles, stream) : launch_rows_t<uint16_t, 8, MODE, true>(rp, tiles, stream);
    return path == P_VEC ? launch_rows_t<float, 4, MODE>(rp, tiles, stream) : launch_rows_t<float, 4, MODE, true>(rp, tiles, stream);
  } else {
    if (bf16) {
      if (path == P_VEC) return launch_rows_t<uint16_t, 8, MODE>(rp, tiles, stream);
      if (path == P_PHASED) return launch_rows_t<uint16_t, 8, MODE, true>(rp, tiles, stream);
      return launch_rows_t<uint16_t, 8, MODE, true, true>(rp, tiles, stream);
    }
    if (path == P_VEC) return launch_rows_t<float, 4, MODE>(rp, tiles, stream);
    if (path == P_PHASED) return launch_rows_t<float, 4, MODE, true>(rp, tiles, stream);
    return launch_rows_t<float, 4, MODE, true, true>(rp, tiles, stream);
  }
}

template <typename E, int VEC, bool PH = false, bool SH = false>
cudaError_t launch_sample2_t(const SampleParams& sp, long long blocks, cudaStream_t stream) {
  auto kern = sample2_kernel<E, VEC, PH, SH>;
  const int smem = SH ? kShiftSmem : kRowsSmem;
  static std::atomic<unsigned long long> done{0};
  const cudaError_t e = ensure_smem_attr(kern, done, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, sp);
}

// The sampler for the tile kernel's row layout: rows on the 16-byte grid, or all at the
// offset sp.ph within it (P_VEC, P_PHASED with rows of whole blocks); every row at its own
// offset (shifted: single rows, and pairs shifted to the target's offset).
enum SamplePath { S_VEC, S_SHIFT };

cudaError_t launch_sample2(bool bf16, SamplePath path, const SampleParams& sp, long long blocks, cudaStream_t stream) {
  if (bf16) {
    if (path == S_SHIFT) return launch_sample2_t<uint16_t, 8, true, true>(sp, blocks, stream);
    return sp.ph ? launch_sample2_t<uint16_t, 8, true>(sp, blocks, stream) : launch_sample2_t<uint16_t, 8>(sp, blocks, stream);
  }
  if (path == S_SHIFT) return launch_sample2_t<float, 4, true, true>(sp, blocks, stream);
  return sp.ph ? launch_sample2_t<float, 4, true>(sp, blocks, stream) : launch_sample2_t<float, 4>(sp, blocks, stream);
}

// Fused multi-draft tiles: when given, the verification launches multi_rows_kernel over
// (group, row, chunk) tiles instead of rows_kernel over (row, chunk) tiles. A fused tile
// reads 2K rows of a chunk of up to 65536 tokens (G=64, K=3, V=128256, same box: 176.4 us
// against 177.8 with whole rows and 177.3 with three chunks per row: the shorter tiles even
// out the last wave; with the pair stage on packed data the per-tile fixed work weighs less
// than it did at 229.5 against 222.5 us).
constexpr int kMultiChunk = 65536;
struct MultiTiles {
  int K = 0;
  PairParams pp;
};

template <typename E, int VEC, int K, int MODE>
cudaError_t launch_multi_t(const RowsParams& rp, const PairParams& pp, long long tiles, cudaStream_t stream) {
  auto kern = multi_rows_kernel<E, VEC, K, MODE>;
  static std::atomic<unsigned long long> done{0};
  const cudaError_t e = ensure_smem_attr(kern, done, multi_smem<K>());
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3((unsigned)tiles);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)multi_smem<K>();
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, rp, pp);
}

template <int MODE>
cudaError_t launch_multi(bool bf16, const MultiTiles& mt, const RowsParams& rp, long long tiles, cudaStream_t stream) {
  if (bf16) {
    if (mt.K == 2) return launch_multi_t<uint16_t, 8, 2, MODE>(rp, mt.pp, tiles, stream);
    if (mt.K == 3) return launch_multi_t<uint16_t, 8, 3, MODE>(rp, mt.pp, tiles, stream);
    return launch_multi_t<uint16_t, 8, 4, MODE>(rp, mt.pp, tiles, stream);
  }
  if (mt.K == 2) return launch_multi_t<float, 4, 2, MODE>(rp, mt.pp, tiles, stream);
  if (mt.K == 3) return launch_multi_t<float, 4, 3, MODE>(rp, mt.pp, tiles, stream);
  return launch_multi_t<float, 4, 4, MODE>(rp, mt.pp, tiles, stream);
}

// Resident blocks of one kernel per SM at kThreads threads and `smem` bytes of dynamic
// shared memory (the attribute that allows more than 48 KB is set first).
template <typename K>
cudaError_t blocks_per_sm(K kernel, int smem, int* out) {
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, kernel, kThreads, (size_t)smem);
}

// The current device's waves, looked up once per device: the SM count times the resident
// blocks per SM of the tile kernel, of the fused multi-draft kernel (the fewest over K) and
// of the sampler. Every instance of a family shares its launch bounds and staging size.
cudaError_t device_geometry(Geometry* out) {
  static std::mutex mu;
  static Geometry cache[kAttrDevices];
  static std::atomic<unsigned long long> have{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kAttrDevices) return cudaErrorInvalidDevice;
  const unsigned long long bit = 1ull << dev;
  if (!(have.load(std::memory_order_acquire) & bit)) {
    std::lock_guard<std::mutex> lock(mu);
    if (!(have.load(std::memory_order_acquire) & bit)) {
      int sms = 0, ot = 0, os = 0, o2 = 0, o3 = 0, o4 = 0;
      if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
      if ((e = blocks_per_sm(rows_kernel<uint16_t, 8, M_STOCH, false>, kRowsSmem, &ot)) != cudaSuccess) return e;
      if ((e = blocks_per_sm(sample2_kernel<uint16_t, 8>, kRowsSmem, &os)) != cudaSuccess) return e;
      if ((e = blocks_per_sm(multi_rows_kernel<uint16_t, 8, 2, M_STOCH>, multi_smem<2>(), &o2)) != cudaSuccess) return e;
      if ((e = blocks_per_sm(multi_rows_kernel<uint16_t, 8, 3, M_STOCH>, multi_smem<3>(), &o3)) != cudaSuccess) return e;
      if ((e = blocks_per_sm(multi_rows_kernel<uint16_t, 8, 4, M_STOCH>, multi_smem<4>(), &o4)) != cudaSuccess) return e;
      const int om = o2 < o3 ? (o2 < o4 ? o2 : o4) : (o3 < o4 ? o3 : o4);
      Geometry g;
      g.tile_slots = (long long)sms * (ot > 0 ? ot : 1);
      g.fused_slots = (long long)sms * (om > 0 ? om : 1);
      g.sampler_blocks = (long long)sms * (os > 0 ? os : 1);
      cache[dev] = g;
      have.fetch_or(bit, std::memory_order_acq_rel);
    }
  }
  *out = cache[dev];
  return cudaSuccess;
}

// The buffers a call's kernels may touch, for the bounds-checked build: target rows
// [total_draft + B, V], draft rows [total_draft, V] (absent: null), the workspace.
struct Extents {
  Ext target, draft, ws;
};

Extents call_extents(const spec_batch& g, spec_dtype dt, const void* target, const void* draft, const void* ws,
                     size_t ws_bytes) {
  const size_t es = dt == SPEC_BF16 ? 2 : 4, V = (size_t)g.V;
  Extents x;
  x.target = Ext{target, target ? ((size_t)g.total_draft + (size_t)g.B) * V * es : 0};
  x.draft = Ext{draft, draft ? (size_t)g.total_draft * V * es : 0};
  x.ws = Ext{ws, ws_bytes};
  return x;
}

RowsParams base_params(const spec_batch& g, const Layout& L, char* ws, uint32_t* status) {
  RowsParams rp;
  memset(&rp, 0, sizeof(rp));
  rp.cu = g.cu_draft;
  rp.row_seq = g.cu_draft != nullptr ? reinterpret_cast<const int32_t*>(ws + L.seqmap) : nullptr;
  rp.B = g.B;
  rp.V = g.V;
  rp.gamma = g.gamma;
  rp.total_draft = g.total_draft;
  rp.total_rows = (int)L.rows;
  rp.nchunks = L.nchunks;
  rp.chunk_elems = L.chunk_elems;
  rp.status = status;
  rp.part = reinterpret_cast<Partial*>(ws + L.part);
  rp.cnt = reinterpret_cast<unsigned*>(ws + L.cntA);
  rp.rec = reinterpret_cast<SeqRec*>(ws + L.rec);
  rp.inv_lnV = g.V > 1 ? (float)(1.0 / log((double)g.V)) : 0.f;
  rp.x_ws = Ext{ws, L.total};
  rp.out_rows = (int)L.rows;
  return rp;
}

bool vec_path(spec_dtype dt, int V, const void* a, const void* b) {
  const int es = dt == SPEC_BF16 ? 2 : 4;
  return ((long long)V * es) % 16 == 0 && aligned16(a) && aligned16(b);
}

// b == nullptr: single rows. Rows of a whole number of 16-byte blocks keep their base's
// offset within the grid, so the rows of every pair share it when the bases do.
RowPath row_path(spec_dtype dt, int V, const void* a, const void* b) {
  if (vec_path(dt, V, a, b)) return P_VEC;
  if (b == nullptr) return P_PHASED;
  const int es = dt == SPEC_BF16 ? 2 : 4;
  if (((long long)V * es) % 16 == 0 && (((uintptr_t)a ^ (uintptr_t)b) & 15u) == 0) return P_PHASED;
  return P_SHIFT;
}

bool temperature_ok(float T) { return isfinite(T) && T > 0.f; }

// Host checks of an options block for a call of the given kind (stochastic, greedy or
// NKL) on batch g; fields the call does not use are not looked at. An output array of
// no elements (block_n when B = 0, block_tokens when no sequence has a draft) may be NULL.
spec_status check_options(const spec_options* o, spec_mode mode, const spec_batch& g) {
  if (o == nullptr) return SPEC_OK;
  if (mode == SPEC_MODE_STOCHASTIC && !(o->temperature_draft == 0.f || temperature_ok(o->temperature_draft)))
    return SPEC_ERR_INVALID_ARG;
  if (mode != SPEC_MODE_GREEDY && o->position != nullptr &&
      !(isfinite(o->delta_alpha) && isfinite(o->delta_max)))
    return SPEC_ERR_INVALID_ARG;
  if (mode != SPEC_MODE_NKL) {
    if (o->min_block_len < 0) return SPEC_ERR_INVALID_ARG;
    if (o->min_block_len > 0 && ((g.B > 0 && !o->block_n) || (g.total_draft > 0 && !o->block_tokens)))
      return SPEC_ERR_INVALID_ARG;
  }
  if (!aligned_to(4, {o->position, o->block_n, o->block_tokens}) || !aligned_to(8, {o->stats}))
    return SPEC_ERR_INVALID_ARG;
  return SPEC_OK;
}

// Copies the options a tile kernel uses into its parameters.
void apply_options(RowsParams& rp, const spec_options* o, spec_mode mode) {
  if (o == nullptr) return;
  if (mode != SPEC_MODE_GREEDY && o->position != nullptr) {
    rp.position = o->position;
    rp.dalpha = o->delta_alpha;
    rp.dmax = o->delta_max;
  }
  if (mode != SPEC_MODE_NKL) {
    if (o->min_block_len > 0) {
      rp.min_block = o->min_block_len;
      rp.block_n = o->block_n;
      rp.block_tok = o->block_tokens;
    }
    if (o->stats) rp.stats = &o->stats->slot[stats_slot(o->stats_bucket)];
  }
}

spec_status stochastic_impl(spec_batch g, spec_dtype dtype, const void* target_logits, const void* draft_logits,
                            const int32_t* draft_tokens, float temperature, const float* u_accept,
                            const float* u_sample, int32_t* n_accepted, int32_t* out_tokens, float* p_x, float* q_x,
                            float* alpha, float* nkl, uint8_t* nkl_mask, float nkl_delta, int32_t* greedy_n,
                            int32_t* greedy_tokens, const spec_options* options, uint32_t* device_status,
                            void* workspace, size_t workspace_bytes, spec_stream_t stream_, ZeroRegion zr,
                            const MultiTiles* mt = nullptr) {
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_DTYPE;
  spec_status st = check_batch(g);
  if (st != SPEC_OK) return st;
  if (!temperature_ok(temperature)) return SPEC_ERR_INVALID_ARG;
  st = check_options(options, SPEC_MODE_STOCHASTIC, g);
  if (st != SPEC_OK) return st;
  if (g.B == 0) return SPEC_OK;
  if (!target_logits || !n_accepted || !out_tokens || !u_sample || !device_status) return SPEC_ERR_INVALID_ARG;
  if (g.total_draft > 0 && (!draft_logits || !draft_tokens || !u_accept)) return SPEC_ERR_INVALID_ARG;
  if ((greedy_n == nullptr) != (greedy_tokens == nullptr)) return SPEC_ERR_INVALID_ARG;
  if (!aligned_to(elem_bytes(dtype), {target_logits, draft_logits}) ||
      !aligned_to(4, {draft_tokens, u_accept, u_sample, n_accepted, out_tokens, p_x, q_x, alpha, nkl, greedy_n,
                      greedy_tokens, device_status, g.cu_draft}))
    return SPEC_ERR_INVALID_ARG;
  // the workspace is checked first (its size does not depend on the device), then the
  // device's waves plan the chunks
  if (!workspace_ok(workspace, workspace_bytes,
                    layout(g.B, g.V, rows_for(SPEC_MODE_STOCHASTIC, g), true, false, dtype, mt ? kMultiChunk : 0,
                           mt ? mt->K : 0).total))
    return SPEC_ERR_WORKSPACE;
  Geometry geo;
  if (device_geometry(&geo) != cudaSuccess) return SPEC_ERR_CUDA;
  const Layout L = layout(g.B, g.V, rows_for(SPEC_MODE_STOCHASTIC, g), true, false, dtype, mt ? kMultiChunk : 0,
                          mt ? mt->K : 0, geo);
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  char* ws = static_cast<char*>(workspace);
  const bool bf16 = dtype == SPEC_BF16;
  const RowPath path = row_path(dtype, g.V, target_logits, draft_logits);

  if (launch_prologue(g, L, ws, device_status, stream, options, zr) != cudaSuccess) return SPEC_ERR_CUDA;
  RowsParams rp = base_params(g, L, ws, device_status);
  rp.target = target_logits;
  rp.draft = draft_logits;
  const Extents xs = call_extents(g, dtype, target_logits, draft_logits, workspace, L.total);
  rp.x_target = xs.target;
  rp.x_draft = xs.draft;
  rp.tokens = draft_tokens;
  rp.u_accept = u_accept;
  rp.u_sample = u_sample;
  rp.c = (float)(1.4426950408889634 / (double)temperature);
  rp.invT = (float)(1.0 / (double)temperature);
  const float Td = (options && options->temperature_draft > 0.f) ? options->temperature_draft : temperature;
  const bool sept = Td != temperature;
  rp.cd = sept ? (float)(1.4426950408889634 / (double)Td) : rp.c;
  rp.delta = nkl_delta;
  apply_options(rp, options, SPEC_MODE_STOCHASTIC);
  rp.n_acc = n_accepted;
  rp.out_tok = out_tokens;
  rp.p_x = p_x;
  rp.q_x = q_x;
  rp.alpha = alpha;
  rp.nkl = nkl;
  rp.mask = nkl_mask;
  rp.g_n = greedy_n;
  rp.g_tok = greedy_tokens;
  // fused multi-draft tiles: (group, row, chunk), one per group row instead of per sequence row
  const long long tiles = mt ? (long long)(g.B / mt->K) * (g.gamma + 1) * L.nchunks : L.rows * L.nchunks;
  // a draft temperature of its own needs the draft row at both scales only for the NKL
  // outputs (both rows at the target's temperature); without them the single-scale tiles
  // serve, the draft at its own scale cd
  const bool two_scales = sept && (nkl != nullptr || nkl_mask != nullptr);
  const cudaError_t le = mt           ? launch_multi<M_STOCH>(bf16, *mt, rp, tiles, stream)
                         : two_scales ? launch_rows<M_STOCH2>(bf16, path, rp, tiles, stream)
                                      : launch_rows<M_STOCH>(bf16, path, rp, tiles, stream);
  if (le != cudaSuccess) return SPEC_ERR_CUDA;

  SampleParams sp;
  memset(&sp, 0, sizeof(sp));
  sp.target = target_logits;
  sp.draft = draft_logits;
  sp.x_target = xs.target;
  sp.x_draft = xs.draft;
  sp.x_ws = xs.ws;
  sp.V = g.V;
  sp.total_rows = (int)L.rows;
  sp.total_draft = g.total_draft;
  sp.B = g.B;
  sp.c = rp.c;
  sp.cd = rp.cd;
  sp.rec = rp.rec;
  sp.cnt = reinterpret_cast<unsigned*>(ws + L.cntB);
  sp.out_tok = out_tokens;
  sp.status = device_status;
  sp.table = reinterpret_cast<float*>(ws + L.table);
  sp.table_stride = L.table_stride;
  sp.tiles_done = reinterpret_cast<const unsigned*>(ws + L.cntA) + g.B;
  sp.ntiles = (unsigned)tiles;
  // rows of a whole number of 16-byte blocks keep their base's offset: the aligned sampler
  // with that offset; any other layout: every row at its own offset (stages sized for the
  // largest, VEC - 1)
  const bool uniform = ((long long)g.V * (long long)elem_bytes(dtype)) % 16 == 0;
  const bool one_offset = path == P_VEC || (path == P_PHASED && uniform);
  const int vec = bf16 ? 8 : 4;
  sp.ph = one_offset ? (path == P_VEC ? 0 : (int)(((uintptr_t)target_logits & 15u) / elem_bytes(dtype))) : vec - 1;
  // One wave of blocks over the B * nst stages. The last kTailSeqs sequences (decided last
  // by the tile kernel) take short ranges of at least kTailStages stages on at most a
  // quarter of the wave, the others equal long ranges.
  const long long nv = ceil_div((long long)g.V + sp.ph, bf16 ? 8 : 4);  // the rows' aligned blocks
  const long long nst = ceil_div(nv, 2 * kThreads);
  const plan::SamplerPlan sg = plan::sampler_plan(g.B, nst, geo.sampler_blocks, kTailSeqs, kTailStages);
  sp.head_total = sg.head_total;
  sp.nb_head = (int)sg.nb_head;
  sp.seg_head = (int)sg.seg_head;
  sp.seg_tail = (int)sg.seg_tail;
  if (launch_sample2(bf16, one_offset ? S_VEC : S_SHIFT, sp, sg.nb_head + sg.nb_tail, stream) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return SPEC_OK;
}

spec_status greedy_impl(spec_batch g, spec_dtype dtype, const void* target_logits, const int32_t* draft_tokens,
                        int32_t* n_accepted, int32_t* out_tokens, const spec_options* options,
                        uint32_t* device_status, void* workspace, size_t workspace_bytes, spec_stream_t stream_,
                        ZeroRegion zr, const MultiTiles* mt = nullptr) {
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_DTYPE;
  spec_status st = check_batch(g);
  if (st != SPEC_OK) return st;
  st = check_options(options, SPEC_MODE_GREEDY, g);
  if (st != SPEC_OK) return st;
  if (g.B == 0) return SPEC_OK;
  if (!target_logits || !n_accepted || !out_tokens || !device_status) return SPEC_ERR_INVALID_ARG;
  if (g.total_draft > 0 && !draft_tokens) return SPEC_ERR_INVALID_ARG;
  if (!aligned_to(elem_bytes(dtype), {target_logits}) ||
      !aligned_to(4, {draft_tokens, n_accepted, out_tokens, device_status, g.cu_draft}))
    return SPEC_ERR_INVALID_ARG;
  if (!workspace_ok(workspace, workspace_bytes,
                    layout(g.B, g.V, rows_for(SPEC_MODE_GREEDY, g), false, true, SPEC_F32, mt ? kMultiChunk : 0,
                           mt ? mt->K : 0).total))
    return SPEC_ERR_WORKSPACE;
  Geometry geo;
  if (device_geometry(&geo) != cudaSuccess) return SPEC_ERR_CUDA;
  const Layout L = layout(g.B, g.V, rows_for(SPEC_MODE_GREEDY, g), false, true, SPEC_F32, mt ? kMultiChunk : 0,
                          mt ? mt->K : 0, geo);
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  char* ws = static_cast<char*>(workspace);
  if (launch_prologue(g, L, ws, device_status, stream, options, zr) != cudaSuccess) return SPEC_ERR_CUDA;
  RowsParams rp = base_params(g, L, ws, device_status);
  rp.target = target_logits;
  rp.x_target = call_extents(g, dtype, target_logits, nullptr, workspace, L.total).target;
  rp.tokens = draft_tokens;
  rp.n_acc = n_accepted;
  rp.out_tok = out_tokens;
  rp.c = rp.cd = 1.f;
  apply_options(rp, options, SPEC_MODE_GREEDY);
  if (mt) {
    rp.draft = mt->pp.draft;  // the fused tiles also read the draft rows (for the matrix)
    rp.x_draft = mt->pp.x_draft;
    if (launch_multi<M_GREEDY>(dtype == SPEC_BF16, *mt, rp, (long long)(g.B / mt->K) * (g.gamma + 1) * L.nchunks,
                               stream) != cudaSuccess)
      return SPEC_ERR_CUDA;
    return SPEC_OK;
  }
  if (launch_rows<M_GREEDY>(dtype == SPEC_BF16, row_path(dtype, g.V, target_logits, nullptr), rp,
                            L.rows * L.nchunks, stream) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return SPEC_OK;
}

// ---------------------------------------------------------------------------
// multi-draft verification: the candidates' verification workspace, then the matrix's
// tickets and partials

struct MultiLayout {
  size_t verify, tickets, part, total;
  int nchunks, chunk_elems;    // two-pass matrix (pair_kernel) chunking
  int vchunks, vchunk_elems;   // the verification's chunking, used by the fused tiles
};

spec_batch multi_as_batch(const spec_multi_batch& m) {
  spec_batch g;
  g.B = m.G * m.K;
  g.gamma = m.gamma;
  g.V = m.V;
  g.total_draft = m.G * m.K * m.gamma;
  g.cu_draft = nullptr;
  return g;
}

spec_status check_multi(const spec_multi_batch& m) {
  if (m.G < 0 || m.K < 2 || m.K > SPEC_MAX_CANDIDATES || m.gamma < 0 || m.gamma > SPEC_MAX_GAMMA || m.V < 1)
    return SPEC_ERR_INVALID_ARG;
  if ((long long)m.G * m.K * (m.gamma + 1) > (1LL << 30)) return SPEC_ERR_INVALID_ARG;
  return check_batch(multi_as_batch(m));
}

// geo: the device's waves (the chunkings follow them; sizes and offsets are those of the
// largest wave allowed, as in layout()).
MultiLayout multi_layout(const spec_multi_batch& m, spec_dtype dt, bool stochastic,
                         const Geometry& geo = Geometry::bound()) {
  const spec_batch g = multi_as_batch(m);
  const spec_mode mode = stochastic ? SPEC_MODE_STOCHASTIC : SPEC_MODE_GREEDY;
  MultiLayout M;
  const Layout Lv = layout(g.B, g.V, rows_for(mode, g), stochastic, !stochastic, dt, kMultiChunk, m.K, geo);
  const Layout Lp = layout(g.B, g.V, rows_for(mode, g), stochastic, !stochastic, dt);  // two-pass: plain tiles
  M.verify = align256(Lv.total > Lp.total ? Lv.total : Lp.total);
  M.vchunks = Lv.nchunks;
  M.vchunk_elems = Lv.chunk_elems;
  const long long rows = (long long)m.G * m.gamma;
  // a two-pass tile reads K rows of one chunk: about 64 K elements in all
  const int pmax = 65536 / (m.K > 0 ? m.K : 1);
  const plan::Chunking run = plan::chunking(m.V, rows, pmax, geo.tile_slots);
  const plan::Chunking cap = plan::chunking(m.V, rows, pmax, plan::kMaxWaveSlots);
  M.nchunks = run.nchunks;
  M.chunk_elems = run.chunk_elems;
  const int pchunks = cap.nchunks > Lv.cap_nchunks ? cap.nchunks : Lv.cap_nchunks;
  M.tickets = M.verify;
  M.part = align256(M.tickets + sizeof(unsigned) * (size_t)rows);
  M.total = align256(M.part + sizeof(PairPartial) * (size_t)rows * pchunks);
  return M;
}

template <typename E, int VEC>
cudaError_t launch_pair_t(int K, const PairParams& pp, long long tiles, cudaStream_t stream) {
  const dim3 grid((unsigned)tiles), block(kThreads);
  if (K == 2) return launch(pair_kernel<E, VEC, 2>, grid, block, stream, pp, true);
  if (K == 3) return launch(pair_kernel<E, VEC, 3>, grid, block, stream, pp, true);
  return launch(pair_kernel<E, VEC, 4>, grid, block, stream, pp, true);
}

template <typename E, int K>
cudaError_t launch_pair_staged_k(const PairParams& pp, long long tiles, cudaStream_t stream) {
  auto kern = pair_staged_kernel<E, K>;
  constexpr int smem = pair_staged_smem<K>();
  static std::atomic<unsigned long long> done{0};
  const cudaError_t e = ensure_smem_attr(kern, done, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3((unsigned)tiles);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, pp);
}

template <typename E>
cudaError_t launch_pair_staged(int K, const PairParams& pp, long long tiles, cudaStream_t stream) {
  if (K == 2) return launch_pair_staged_k<E, 2>(pp, tiles, stream);
  if (K == 3) return launch_pair_staged_k<E, 3>(pp, tiles, stream);
  return launch_pair_staged_k<E, 4>(pp, tiles, stream);
}

// aligned rows: 16-byte vector loads; any other layout: the staged kernel
cudaError_t launch_pair(bool bf16, bool vec, int K, const PairParams& pp, long long tiles, cudaStream_t stream) {
  if (bf16) return vec ? launch_pair_t<uint16_t, 8>(K, pp, tiles, stream) : launch_pair_staged<uint16_t>(K, pp, tiles, stream);
  return vec ? launch_pair_t<float, 4>(K, pp, tiles, stream) : launch_pair_staged<float>(K, pp, tiles, stream);
}

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" {

size_t spec_workspace_bytes(spec_batch g, spec_dtype dtype, spec_mode mode) {
  if (check_batch(g) != SPEC_OK || (dtype != SPEC_F32 && dtype != SPEC_BF16)) return 0;
  return layout(g.B, g.V, rows_for(mode, g), mode == SPEC_MODE_STOCHASTIC, mode == SPEC_MODE_GREEDY, dtype).total;
}

size_t spec_tree_workspace_bytes(int32_t B, int32_t N, int32_t V) {
  if (B < 0 || N < 1 || N > SPEC_MAX_TREE_NODES || V < 1) return 0;
  return layout(B, V, (long long)B * (N + 1), false, true).total;
}

int32_t spec_tree_depth(const int32_t* parent, int32_t N) {
  if (parent == nullptr || N < 1 || N > SPEC_MAX_TREE_NODES) return -1;
  int depth[SPEC_MAX_TREE_NODES];
  int D = 0;
  for (int j = 0; j < N; ++j) {
    const int pj = parent[j];
    if (pj < -1 || pj >= j) return -1;
    depth[j] = pj < 0 ? 1 : depth[pj] + 1;
    if (depth[j] > D) D = depth[j];
  }
  return D;
}

spec_status spec_verify_stochastic(spec_batch g, spec_dtype dtype, const void* target_logits,
                                   const void* draft_logits, const int32_t* draft_tokens, float temperature,
                                   const float* u_accept, const float* u_sample, int32_t* n_accepted,
                                   int32_t* out_tokens, float* p_x, float* q_x, float* alpha, float* nkl,
                                   uint8_t* nkl_mask, float nkl_delta, int32_t* greedy_n, int32_t* greedy_tokens,
                                   uint32_t* device_status, void* workspace, size_t workspace_bytes,
                                   spec_stream_t stream) {
  return spec_verify_stochastic_ex(g, dtype, target_logits, draft_logits, draft_tokens, temperature, u_accept,
                                   u_sample, n_accepted, out_tokens, p_x, q_x, alpha, nkl, nkl_mask, nkl_delta,
                                   greedy_n, greedy_tokens, nullptr, device_status, workspace, workspace_bytes,
                                   stream);
}

spec_status spec_verify_stochastic_ex(spec_batch g, spec_dtype dtype, const void* target_logits,
                                      const void* draft_logits, const int32_t* draft_tokens, float temperature,
                                      const float* u_accept, const float* u_sample, int32_t* n_accepted,
                                      int32_t* out_tokens, float* p_x, float* q_x, float* alpha, float* nkl,
                                      uint8_t* nkl_mask, float nkl_delta, int32_t* greedy_n,
                                      int32_t* greedy_tokens, const spec_options* options, uint32_t* device_status,
                                      void* workspace, size_t workspace_bytes, spec_stream_t stream) {
  const ApiRange range("spec_verify_stochastic");
  return stochastic_impl(g, dtype, target_logits, draft_logits, draft_tokens, temperature, u_accept, u_sample,
                         n_accepted, out_tokens, p_x, q_x, alpha, nkl, nkl_mask, nkl_delta, greedy_n, greedy_tokens,
                         options, device_status, workspace, workspace_bytes, stream, ZeroRegion());
}

spec_status spec_verify_greedy(spec_batch g, spec_dtype dtype, const void* target_logits,
                               const int32_t* draft_tokens, int32_t* n_accepted, int32_t* out_tokens,
                               uint32_t* device_status, void* workspace, size_t workspace_bytes,
                               spec_stream_t stream) {
  return spec_verify_greedy_ex(g, dtype, target_logits, draft_tokens, n_accepted, out_tokens, nullptr,
                               device_status, workspace, workspace_bytes, stream);
}

spec_status spec_verify_greedy_ex(spec_batch g, spec_dtype dtype, const void* target_logits,
                                  const int32_t* draft_tokens, int32_t* n_accepted, int32_t* out_tokens,
                                  const spec_options* options, uint32_t* device_status, void* workspace,
                                  size_t workspace_bytes, spec_stream_t stream) {
  const ApiRange range("spec_verify_greedy");
  return greedy_impl(g, dtype, target_logits, draft_tokens, n_accepted, out_tokens, options, device_status,
                     workspace, workspace_bytes, stream, ZeroRegion());
}

spec_status spec_verify_tree(int32_t B, int32_t N, int32_t V, spec_dtype dtype, const void* target_logits,
                             const int32_t* node_tokens, const int32_t* parent, int32_t* accept_len,
                             int32_t* path_nodes, int32_t* out_tokens, uint32_t* device_status, void* workspace,
                             size_t workspace_bytes, spec_stream_t stream_) {
  const ApiRange range("spec_verify_tree");
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_DTYPE;
  if (B < 0 || V < 1 || V > (1 << 26)) return SPEC_ERR_INVALID_ARG;
  const int D = spec_tree_depth(parent, N);
  if (D < 1) return SPEC_ERR_INVALID_ARG;
  if ((long long)B * (N + 1) > (1LL << 30)) return SPEC_ERR_INVALID_ARG;
  if (B == 0) return SPEC_OK;
  if (!target_logits || !node_tokens || !accept_len || !path_nodes || !out_tokens || !device_status)
    return SPEC_ERR_INVALID_ARG;
  if (!aligned_to(elem_bytes(dtype), {target_logits}) ||
      !aligned_to(4, {node_tokens, accept_len, path_nodes, out_tokens, device_status}))
    return SPEC_ERR_INVALID_ARG;
  spec_batch g;
  g.B = B;
  g.gamma = N;
  g.V = V;
  g.total_draft = B * N;
  g.cu_draft = nullptr;
  if (!workspace_ok(workspace, workspace_bytes, layout(B, V, (long long)B * (N + 1), false, true).total))
    return SPEC_ERR_WORKSPACE;
  Geometry geo;
  if (device_geometry(&geo) != cudaSuccess) return SPEC_ERR_CUDA;
  const Layout L = layout(B, V, (long long)B * (N + 1), false, true, SPEC_F32, 0, 0, geo);
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  char* ws = static_cast<char*>(workspace);
  if (launch_prologue(g, L, ws, device_status, stream) != cudaSuccess) return SPEC_ERR_CUDA;
  RowsParams rp = base_params(g, L, ws, device_status);
  rp.target = target_logits;
  rp.x_target = call_extents(g, dtype, target_logits, nullptr, workspace, L.total).target;
  rp.node_tokens = node_tokens;
  rp.N = N;
  rp.depth = D;
  for (int j = 0; j < N; ++j) rp.parent[j] = (int8_t)parent[j];
  rp.accept_len = accept_len;
  rp.path_nodes = path_nodes;
  rp.out_tok = out_tokens;
  rp.c = rp.cd = 1.f;
  if (launch_rows<M_TREE>(dtype == SPEC_BF16, row_path(dtype, V, target_logits, nullptr), rp, L.rows * L.nchunks,
                          stream) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return SPEC_OK;
}

spec_status spec_nkl(spec_batch g, spec_dtype dtype, const void* target_logits, const void* draft_logits,
                     float temperature, float delta, float* nkl, uint8_t* nkl_mask, uint32_t* device_status,
                     void* workspace, size_t workspace_bytes, spec_stream_t stream) {
  return spec_nkl_ex(g, dtype, target_logits, draft_logits, temperature, delta, nkl, nkl_mask, nullptr,
                     device_status, workspace, workspace_bytes, stream);
}

spec_status spec_nkl_ex(spec_batch g, spec_dtype dtype, const void* target_logits, const void* draft_logits,
                        float temperature, float delta, float* nkl, uint8_t* nkl_mask, const spec_options* options,
                        uint32_t* device_status, void* workspace, size_t workspace_bytes, spec_stream_t stream_) {
  const ApiRange range("spec_nkl");
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_DTYPE;
  spec_status st = check_batch(g);
  if (st != SPEC_OK) return st;
  if (!temperature_ok(temperature)) return SPEC_ERR_INVALID_ARG;
  st = check_options(options, SPEC_MODE_NKL, g);
  if (st != SPEC_OK) return st;
  if (g.B == 0 || g.total_draft == 0) return SPEC_OK;
  if (!target_logits || !draft_logits || !nkl || !device_status) return SPEC_ERR_INVALID_ARG;
  if (!aligned_to(elem_bytes(dtype), {target_logits, draft_logits}) || !aligned_to(4, {nkl, device_status, g.cu_draft}))
    return SPEC_ERR_INVALID_ARG;
  if (!workspace_ok(workspace, workspace_bytes, layout(g.B, g.V, rows_for(SPEC_MODE_NKL, g), false).total))
    return SPEC_ERR_WORKSPACE;
  Geometry geo;
  if (device_geometry(&geo) != cudaSuccess) return SPEC_ERR_CUDA;
  const Layout L = layout(g.B, g.V, rows_for(SPEC_MODE_NKL, g), false, false, SPEC_F32, 0, 0, geo);
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  char* ws = static_cast<char*>(workspace);
  if (launch_prologue(g, L, ws, device_status, stream, nullptr, ZeroRegion(), 0) != cudaSuccess) return SPEC_ERR_CUDA;
  RowsParams rp = base_params(g, L, ws, device_status);
  rp.target = target_logits;
  rp.draft = draft_logits;
  const Extents xs = call_extents(g, dtype, target_logits, draft_logits, workspace, L.total);
  rp.x_target = xs.target;
  rp.x_draft = xs.draft;
  rp.c = rp.cd = (float)(1.4426950408889634 / (double)temperature);
  rp.invT = (float)(1.0 / (double)temperature);
  rp.delta = delta;
  rp.nkl = nkl;
  rp.mask = nkl_mask;
  apply_options(rp, options, SPEC_MODE_NKL);
  if (launch_rows<M_NKL>(dtype == SPEC_BF16, row_path(dtype, g.V, target_logits, draft_logits), rp,
                         L.rows * L.nchunks, stream) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return SPEC_OK;
}

size_t spec_multi_workspace_bytes(spec_multi_batch m, spec_dtype dtype, int32_t stochastic) {
  if (check_multi(m) != SPEC_OK || (dtype != SPEC_F32 && dtype != SPEC_BF16)) return 0;
  return multi_layout(m, dtype, stochastic != 0).total;
}

spec_status spec_verify_multi(spec_multi_batch m, spec_dtype dtype, int32_t stochastic, const void* target_logits,
                              const void* draft_logits, const int32_t* draft_tokens, float temperature,
                              const float* u_accept, const float* u_sample, float consensus_nkl,
                              float divergence_nkl, int32_t* n_accepted, int32_t* out_tokens, int32_t* best_k,
                              int32_t* best_n, int32_t* best_tokens, float* pair_nkl, uint8_t* consensus,
                              uint8_t* divergence, uint32_t* device_status, void* workspace,
                              size_t workspace_bytes, spec_stream_t stream_) {
  const ApiRange range("spec_verify_multi");
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_DTYPE;
  spec_status st = check_multi(m);
  if (st != SPEC_OK) return st;
  if (!temperature_ok(temperature) || !isfinite(consensus_nkl) || !isfinite(divergence_nkl))
    return SPEC_ERR_INVALID_ARG;
  if (m.G == 0) return SPEC_OK;
  if (!target_logits || !n_accepted || !out_tokens || !best_k || !best_n || !best_tokens || !device_status)
    return SPEC_ERR_INVALID_ARG;
  if (m.gamma > 0 && (!draft_logits || !draft_tokens)) return SPEC_ERR_INVALID_ARG;
  if (stochastic && (!u_sample || (m.gamma > 0 && !u_accept))) return SPEC_ERR_INVALID_ARG;
  if (!aligned_to(elem_bytes(dtype), {target_logits, draft_logits}) ||
      !aligned_to(4, {draft_tokens, u_accept, u_sample, n_accepted, out_tokens, best_k, best_n, best_tokens, pair_nkl,
                      device_status}))
    return SPEC_ERR_INVALID_ARG;
  if (!workspace_ok(workspace, workspace_bytes, multi_layout(m, dtype, stochastic != 0).total))
    return SPEC_ERR_WORKSPACE;
  Geometry geo;
  if (device_geometry(&geo) != cudaSuccess) return SPEC_ERR_CUDA;
  const MultiLayout ML = multi_layout(m, dtype, stochastic != 0, geo);
  char* ws = static_cast<char*>(workspace);
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const spec_batch g = multi_as_batch(m);
  ZeroRegion zr;
  zr.ptr = reinterpret_cast<unsigned*>(ws + ML.tickets);
  zr.n = m.G * m.gamma;
  PairParams pp;
  memset(&pp, 0, sizeof(pp));
  pp.draft = draft_logits;
  pp.V = m.V;
  pp.gamma = m.gamma;
  pp.K = m.K;
  pp.G = m.G;
  pp.c = (float)(1.4426950408889634 / (double)temperature);
  pp.invT = (float)(1.0 / (double)temperature);
  pp.inv_lnV = m.V > 1 ? (float)(1.0 / log((double)m.V)) : 0.f;
  pp.c_thr = consensus_nkl;
  pp.d_thr = divergence_nkl;
  pp.part = reinterpret_cast<PairPartial*>(ws + ML.part);
  pp.cnt = zr.ptr;
  pp.pair_nkl = pair_nkl;
  pp.cons = consensus;
  pp.div = divergence;
  pp.status = device_status;
  pp.x_draft = call_extents(multi_as_batch(m), dtype, nullptr, draft_logits, workspace, ML.total).draft;
  pp.x_ws = Ext{workspace, ML.total};
  // aligned rows: fused (group, row, chunk) tiles read every logit once and fill the
  // matrix on the way; otherwise the batch kernels, then a second pass over the drafts
  const bool fused = m.gamma > 0 && vec_path(dtype, m.V, target_logits, draft_logits);
  MultiTiles mt;
  mt.K = m.K;
  mt.pp = pp;
  mt.pp.nchunks = ML.vchunks;
  mt.pp.chunk_elems = ML.vchunk_elems;
  st = stochastic ? stochastic_impl(g, dtype, target_logits, draft_logits, draft_tokens, temperature, u_accept,
                                    u_sample, n_accepted, out_tokens, nullptr, nullptr, nullptr, nullptr, nullptr,
                                    0.15f, nullptr, nullptr, nullptr, device_status, workspace, ML.verify, stream_,
                                    zr, fused ? &mt : nullptr)
                  : greedy_impl(g, dtype, target_logits, draft_tokens, n_accepted, out_tokens, nullptr,
                                device_status, workspace, ML.verify, stream_, zr, fused ? &mt : nullptr);
  if (st != SPEC_OK) return st;
  if (m.gamma > 0 && !fused) {
    pp.nchunks = ML.nchunks;
    pp.chunk_elems = ML.chunk_elems;
    const long long tiles = (long long)m.G * m.gamma * ML.nchunks;
    if (launch_pair(dtype == SPEC_BF16, vec_path(dtype, m.V, draft_logits, nullptr), m.K, pp, tiles, stream) !=
        cudaSuccess)
      return SPEC_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3((unsigned)ceil_div(m.G, kThreads));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int G = m.G, K = m.K, gm = m.gamma;
  if (cudaLaunchKernelEx(&cfg, select_kernel, (const int32_t*)n_accepted, (const int32_t*)out_tokens, G, K, gm,
                         best_k, best_n, best_tokens) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return SPEC_OK;
}

spec_status spec_accept_summary(const spec_accept_stats* stats, int64_t bucket_now, int32_t window, double* out,
                                spec_stream_t stream_) {
  const ApiRange range("spec_accept_summary");
  if (!stats || !out || window < 1 || window > SPEC_STATS_SLOTS || !aligned_to(8, {stats, out}))
    return SPEC_ERR_INVALID_ARG;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(SPEC_STATS_SLOTS);
  cfg.stream = reinterpret_cast<cudaStream_t>(stream_);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const long long now = (long long)bucket_now;
  const int w = (int)window;
  if (cudaLaunchKernelEx(&cfg, summary_kernel, stats, now, w, out) != cudaSuccess) return SPEC_ERR_CUDA;
  return SPEC_OK;
}

spec_status spec_selftest_wait_timeout(uint32_t* device_status, void* workspace, size_t workspace_bytes,
                                       spec_stream_t stream_) {
  // one dense sequence, one draft, an 8-token bf16 vocabulary: the prologue re-arms its
  // record, and the sampler waits for a decision and a tile count that no tile kernel
  // ever provides (nothing is read from the logits: the record never becomes ready)
  spec_batch g;
  g.B = 1;
  g.gamma = 1;
  g.V = 8;
  g.total_draft = 1;
  g.cu_draft = nullptr;
  if (!device_status || !aligned_to(4, {device_status})) return SPEC_ERR_INVALID_ARG;
  const Layout L = layout(g.B, g.V, rows_for(SPEC_MODE_STOCHASTIC, g), true, false, SPEC_BF16);
  if (!workspace || workspace_bytes < L.total || ((uintptr_t)workspace & 255u)) return SPEC_ERR_WORKSPACE;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  char* ws = static_cast<char*>(workspace);
  if (launch_prologue(g, L, ws, device_status, stream) != cudaSuccess) return SPEC_ERR_CUDA;
  SampleParams sp;
  memset(&sp, 0, sizeof(sp));
  sp.V = g.V;
  sp.total_rows = (int)L.rows;
  sp.total_draft = g.total_draft;
  sp.B = g.B;
  sp.c = sp.cd = 1.f;
  sp.rec = reinterpret_cast<SeqRec*>(ws + L.rec);
  sp.cnt = reinterpret_cast<unsigned*>(ws + L.cntB);
  sp.status = device_status;
  sp.table = reinterpret_cast<float*>(ws + L.table);
  sp.table_stride = L.table_stride;
  sp.tiles_done = reinterpret_cast<const unsigned*>(ws + L.cntA) + g.B;  // zeroed by the prologue, never counted
  sp.x_ws = Ext{workspace, L.total};
  sp.ntiles = 1u;
  sp.head_total = 0;
  sp.nb_head = 0;
  sp.seg_head = 1;
  sp.seg_tail = kTailStages;
  // an ordinary stream-ordered launch (no programmatic dependent launch): the sampler
  // starts only after the prologue has completed, so the record it polls is re-armed
  auto kern = sample2_kernel<uint16_t, 8>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kRowsSmem) != cudaSuccess)
    return SPEC_ERR_CUDA;
  kern<<<1, kThreads, kRowsSmem, stream>>>(sp);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  return SPEC_OK;
}

const char* spec_status_str(spec_status s) {
  switch (s) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_INVALID_ARG: return "invalid argument";
    case SPEC_ERR_DTYPE: return "unknown dtype";
    case SPEC_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case SPEC_ERR_CUDA: return "CUDA launch failed";
    case SPEC_ERR_TOO_LARGE: return "problem needs more scratch than SPEC_STATIC_SCRATCH_BYTES";
  }
  return "unknown status";
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Stochastic verification for callers that cannot allocate device memory.
//
// Some callers are handed their input and output buffers by a host framework and have
// no device allocator of their own: a plugin inside an inference server whose memory
// pool is owned by the server, or a decode loop that must not call cudaMalloc/cudaFree
// because those may synchronise the device or fragment a pool managed elsewhere. For
// them the scratch memory lives in the library itself: a fixed array in device memory,
// created when the library is loaded on a GPU and kept until the process exits.

#include <mutex>

static __device__ __align__(256) unsigned char spec_static_scratch[SPEC_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void* g_static_addr[kMaxDevices];  // device address of spec_static_scratch, per device

// Device address of the static scratch on the current device. Host code cannot use the
// symbol itself (on the host it names a stand-in, not device memory), so the address is
// looked up once per device with that device current and cached.
cudaError_t static_scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (g_static_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, spec_static_scratch);
    if (e != cudaSuccess) return e;
    g_static_addr[dev] = p;
  }
  *out = g_static_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" spec_status spec_verify_stochastic_static(
    spec_batch g, spec_dtype dtype, const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
    float temperature, const float* u_accept, const float* u_sample, int32_t* n_accepted, int32_t* out_tokens,
    float* p_x, float* q_x, float* alpha, float* nkl, uint8_t* nkl_mask, float nkl_delta, int32_t* greedy_n,
    int32_t* greedy_tokens, uint32_t* device_status, spec_stream_t stream) {
  const ApiRange range("spec_verify_stochastic_static");
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_DTYPE;
  if (check_batch(g) != SPEC_OK) return SPEC_ERR_INVALID_ARG;
  // Everything in the scratch that must start at zero (the per-sequence tickets) or in a
  // known state (the per-sequence records) is reset by the first kernel of every call;
  // the rest is written before it is read. Nothing carries over between calls.
  if (spec_workspace_bytes(g, dtype, SPEC_MODE_STOCHASTIC) > (size_t)SPEC_STATIC_SCRATCH_BYTES)
    return SPEC_ERR_TOO_LARGE;
  void* ws = nullptr;
  if (static_scratch_address(&ws) != cudaSuccess) return SPEC_ERR_CUDA;
  return spec_verify_stochastic(g, dtype, target_logits, draft_logits, draft_tokens, temperature, u_accept, u_sample,
                                n_accepted, out_tokens, p_x, q_x, alpha, nkl, nkl_mask, nkl_delta, greedy_n,
                                greedy_tokens, device_status, ws, (size_t)SPEC_STATIC_SCRATCH_BYTES, stream);
}
