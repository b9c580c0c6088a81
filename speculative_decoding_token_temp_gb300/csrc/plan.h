// Host-side launch planning of the verification kernels: how a row is cut into vocabulary
// chunks and how the sampler's stages are spread over its blocks, both as functions of the
// number of blocks one wave of the GPU holds (SMs x resident blocks per SM). Plain C++: no
// CUDA types, so it is compiled into the library and, on its own, into a CPU test.
#pragma once

namespace sv {
namespace plan {

inline long long cdiv(long long a, long long b) { return (a + b - 1) / b; }

// Largest wave the workspace layout allows for: the workspace size must not depend on the
// device, so its per-tile partials are sized for the chunking at this many slots, and a
// device with a larger wave is planned as if it had this one.
constexpr long long kMaxWaveSlots = 4096;
// Chunks are split no finer than this many tokens.
constexpr int kMinChunk = 8192;

struct Chunking {
  int nchunks;      // chunks per row
  int chunk_elems;  // tokens per chunk (the last may be shorter), a multiple of 8
};

// Vocabulary chunking of the tile kernels: chunks of at most max_chunk tokens, split
// further (down to kMinChunk) only while the grid of rows x chunks tiles still fits in one
// wave of `slots` resident blocks -- a partial second wave of tiles ends after the first.
// Chunk sizes are multiples of 8, so every chunk starts on a 16-byte vector boundary.
// rows: tiles per chunk (>= 1). The result is non-decreasing in slots.
inline Chunking chunking(int V, long long rows, int max_chunk, long long slots) {
  if (rows < 1) rows = 1;
  if (slots > kMaxWaveSlots) slots = kMaxWaveSlots;
  long long nc = cdiv(V, max_chunk);
  while (rows * (nc + 1) <= slots && V / (nc + 1) >= kMinChunk) ++nc;
  const long long ce = cdiv(cdiv(V, nc), 8) * 8;
  Chunking c;
  c.chunk_elems = (int)ce;
  c.nchunks = (int)cdiv(V, ce);
  return c;
}

// The sampler's grid: the B sampled rows are nst stages each, B * nst stages in sequence
// order. The last tail_seqs sequences (the tile kernel decides them last) are cut into
// short ranges of at least min_tail stages spread over at most a quarter of the wave; the
// other sequences take equal long ranges on the rest of the wave. Blocks [0, nb_head) take
// seg_head stages each of [0, head_total), the next nb_tail blocks seg_tail stages each of
// the rest; the grid never exceeds the wave.
struct SamplerPlan {
  long long head_total;
  long long nb_head, seg_head, nb_tail, seg_tail;
};

inline SamplerPlan sampler_plan(long long B, long long nst, long long wave, long long tail_seqs, long long min_tail) {
  if (wave < 1) wave = 1;
  SamplerPlan p;
  const long long ts = B < tail_seqs ? B : tail_seqs;
  const long long tail_total = ts * nst;
  p.head_total = (B - ts) * nst;
  const long long quarter = wave / 4 > 0 ? wave / 4 : 1;
  p.seg_tail = cdiv(tail_total, quarter);
  if (p.seg_tail < min_tail) p.seg_tail = min_tail;
  if (p.seg_tail < 1) p.seg_tail = 1;
  p.nb_tail = cdiv(tail_total, p.seg_tail);
  p.nb_head = 0;
  p.seg_head = 1;
  if (p.head_total > 0) {
    const long long room = wave - p.nb_tail;
    p.seg_head = cdiv(p.head_total, room < 1 ? 1 : room);
    p.nb_head = cdiv(p.head_total, p.seg_head);
  }
  return p;
}

}  // namespace plan
}  // namespace sv
