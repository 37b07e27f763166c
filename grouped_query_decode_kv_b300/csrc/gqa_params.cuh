// Launch parameters shared by the split-KV decode kernels and the combine.
#pragma once

#include <stdint.h>

namespace gqa {

// One CTA of a split kernel owns (batch b, KV head g, head chunk hc,
// sequence split s): the positions [s*chunk, min((s+1)*chunk, L_b)) of K/V
// head g and the query heads [g*n_rep + hc*heads_per_cta, ...) of its group.
struct SplitParams {
  const void *q;            // [B, H, D]
  const int32_t *seq_lens;  // [B]
  void *out;                // [B, H, D]      written when a batch needs one split
  float *o_part;            // [B, H, S_max, D] unnormalised partial outputs
  float *ml_part;           // [B, H, S_max, 2] (running max in log2 units, sum)
  float scale_log2;         // scale * log2(e): softmax is evaluated with exp2
  int B, H, G, Nmax;
  int n_rep;                // H / G
  int chunk;                // positions per split, a multiple of the tile
  int S_max;                // ceil(Nmax / chunk)
  int heads_per_cta;
  int head_chunks;          // ceil(n_rep / heads_per_cta)
};

struct CombineParams {
  const int32_t *seq_lens;
  const float *o_part;
  const float *ml_part;
  void *out;
  int B, H, Nmax, chunk, S_max;
};

}  // namespace gqa
