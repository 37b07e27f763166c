// Launch parameters of the split-KV decode kernels.
#pragma once

#include <stdint.h>

namespace gqa {

// The split kernels run a persistent grid; CTA c walks its stream-K range of
// tiles (see gqa_schedule.cuh) unit by unit.  A unit is (batch b, KV head g,
// head chunk hc): the query heads [g*n_rep + hc*heads_per_cta, ...) of
// group g against K/V head g.
struct SplitParams {
  const void *q;            // [B, H, D]
  const int32_t *seq_lens;  // [B]
  void *out;                // [B, H, D]       whole units are written here directly
  float *o_part;            // [2P, heads_per_cta, D] unnormalised partial outputs
  float *ml_part;           // [2P, heads_per_cta, 2] (running max in log2 units, sum)
  // Per-unit merge bookkeeping, one of the two (the other null):
  unsigned long long *unit_cnt;  // [B*G*HC] in-kernel merge: (call epoch << 32) | CTAs of the unit done
  int2 *unit_info;          // [B*G*HC] merge kernel: (first slot, last CTA) of a split unit, or -1
  unsigned epoch;           // nonzero, different for every call
  // Fused decode step (append != 0): the new token's K/V rows k_new/v_new
  // [B*G, D] go to cache row L_b of every (b, g) before attention over
  // L_b + 1 positions; the last CTA to finish then sets seq_lens[b] = L_b + 1.
  int append;
  const void *k_new, *v_new;
  void *k_cache, *v_cache;  // [B*G, Nmax, D]
  int32_t *seq_lens_w;      // the same array as seq_lens
  int row_chunks;           // 16-byte chunks per cache row (D * element size / 16)
  unsigned *done_cnt;       // CTAs finished, zero between calls; null with one CTA
  float scale_log2;         // scale * log2(e): softmax is evaluated with exp2
  int B, H, G, Nmax;
  int n_rep;                // H / G
  int heads_per_cta;
  int head_chunks;          // HC = ceil(n_rep / heads_per_cta)
};

}  // namespace gqa
