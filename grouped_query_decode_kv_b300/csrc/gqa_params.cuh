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
  // tcgen05 kernel launched in thread-block clusters of cluster_k CTAs (0 or
  // 1: no clusters); see the cluster-aligned plan in gqa_schedule.cuh
  int cluster_k;
  int P;                    // CTAs of the split kernel (partial slots: 2P)
  // Fused decode step (append != 0): the new token's K/V rows k_new/v_new
  // [B*G, D] go to cache row L_b of every (b, g) before attention over
  // L_b + 1 positions; the last CTA to stop reading the lengths then sets
  // seq_lens[b] = L_b + 1.
  int append;
  const void *k_new, *v_new;
  void *k_cache, *v_cache;  // [B*G, Nmax, D]
  int32_t *seq_lens_w;      // the same array as seq_lens
  int row_chunks;           // 16-byte chunks per cache row (D * element size / 16)
  unsigned long long *done_cnt;  // (call epoch << 32) | CTAs finished; null with one CTA
  float scale_log2;         // scale * log2(e): softmax is evaluated with exp2
  int B, H, G, Nmax;
  int n_rep;                // H / G
  int heads_per_cta;
  int head_chunks;          // HC = ceil(n_rep / heads_per_cta)
  // Several query tokens per sequence (tokens > 1): q and out are
  // [B, tokens, heads_q, D] and token t sits at cached position
  // L_b - tokens + t, seeing positions n < L_b - (tokens - 1 - t).  The
  // kernels then treat the tokens * heads_q query rows of a sequence as its
  // "heads": H = tokens * heads_q and n_rep = tokens * rep_kv rows per KV
  // head, row v of group g being token (v - g*n_rep) / rep_kv, head
  // g*rep_kv + (v - g*n_rep) % rep_kv.  With tokens = 1 this is the plain
  // [B, H, D] layout.
  int tokens;
  int heads_q;              // query heads of one token
  int rep_kv;               // query heads of one token per KV head
  // FP8 (E4M3) cache: per-KV-head scales [G] of K and V (null otherwise)
  const float *k_scale, *v_scale;
};

// Checking build: a partial slot and head of the workspace, a row of q /
// out, a cache row of K/V head bg.
#define GQA_SLOT_OK(p, slot, h) \
  GQA_IN_BOUNDS((slot) >= 0 && (slot) < 2 * (p).P && (h) >= 0 && (h) < (p).heads_per_cta)
#define GQA_ROW_OK(p, row) GQA_IN_BOUNDS((size_t)(row) < (size_t)(p).B * (p).H)
#define GQA_CACHE_OK(p, bg, n) \
  GQA_IN_BOUNDS((bg) >= 0 && (bg) < (p).B * (p).G && (n) >= 0 && (n) < (p).Nmax)

// Row (of D elements) of q and out that holds query row v of batch row b.
// MULTI = false: the kernel was compiled for one token per sequence.
template <bool MULTI>
__device__ __forceinline__ size_t query_row(const SplitParams &p, int b, int v) {
  if (!MULTI || p.tokens == 1) return (size_t)b * p.H + v;
  const int g = v / p.n_rep, r = v - g * p.n_rep;
  const int t = r / p.rep_kv;
  return ((size_t)b * p.tokens + t) * p.heads_q + g * p.rep_kv + (r - t * p.rep_kv);
}

// Cached positions at the end of the sequence that query row v may not see
// (the later tokens of its own run): tokens - 1 - t.  0 with one token.
template <bool MULTI>
__device__ __forceinline__ int query_lag(const SplitParams &p, int v) {
  if (!MULTI || p.tokens == 1) return 0;
  return p.tokens - 1 - (v % p.n_rep) / p.rep_kv;
}

}  // namespace gqa
