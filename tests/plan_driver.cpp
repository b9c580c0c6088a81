// Test driver for csrc/plan.h (host-side launch planning): reads queries from stdin and
// prints the plans, one line each.
//   chunk V rows max_chunk slots        -> nchunks chunk_elems
//   sampler B nst wave tail_seqs min    -> head_total nb_head seg_head nb_tail seg_tail
#include <cstdio>
#include <cstring>

#include "plan.h"

int main() {
  char kind[16];
  while (std::scanf("%15s", kind) == 1) {
    if (std::strcmp(kind, "chunk") == 0) {
      long long V, rows, mc, slots;
      if (std::scanf("%lld %lld %lld %lld", &V, &rows, &mc, &slots) != 4) return 2;
      const sv::plan::Chunking c = sv::plan::chunking((int)V, rows, (int)mc, slots);
      std::printf("%d %d\n", c.nchunks, c.chunk_elems);
    } else if (std::strcmp(kind, "sampler") == 0) {
      long long B, nst, wave, ts, mt;
      if (std::scanf("%lld %lld %lld %lld %lld", &B, &nst, &wave, &ts, &mt) != 5) return 2;
      const sv::plan::SamplerPlan p = sv::plan::sampler_plan(B, nst, wave, ts, mt);
      std::printf("%lld %lld %lld %lld %lld\n", p.head_total, p.nb_head, p.seg_head, p.nb_tail, p.seg_tail);
    } else {
      return 2;
    }
  }
  return 0;
}
