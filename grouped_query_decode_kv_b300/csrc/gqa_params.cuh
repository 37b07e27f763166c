// Launch parameters shared by the split-KV decode kernels and the combine.
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
  int2 *unit_info;          // [B*G*HC]        (first slot, last CTA) of split units
  float scale_log2;         // scale * log2(e): softmax is evaluated with exp2
  int B, H, G, Nmax;
  int n_rep;                // H / G
  int heads_per_cta;
  int head_chunks;          // HC = ceil(n_rep / heads_per_cta)
};

struct CombineParams {
  const int32_t *seq_lens;
  const float *o_part;
  const float *ml_part;
  const int2 *unit_info;
  void *out;
  int B, H, G, Nmax;
  int n_rep, heads_per_cta, head_chunks;
};

}  // namespace gqa
