// Log-sum-exp merge of the partial softmax states of a unit that the
// stream-K split cut between CTAs:
//   out = sum_k 2^(m_k - M) o_k / sum_k 2^(m_k - M) l_k,   M = max_k m_k
// over the unit's partials, always read in the same slot order, so the
// result does not depend on timing.  Two ways, chosen per kernel by the host:
//
//  * In the split kernel, by whichever of the unit's CTAs finishes last (no
//    second launch; for units of one or two heads, whose partials are
//    small).  Each unit has a 64-bit counter word in the workspace holding
//    (call epoch << 32) | finished CTAs.  A word left by another call (another
//    epoch) counts as zero, so the workspace needs no clearing; the merging
//    CTA puts the count back to zero, so a call captured in a graph can be
//    replayed.
//  * In a second kernel, one warp per (batch row, query head), launched as a
//    programmatic dependent of the split kernel (for units of many heads,
//    whose merge is spread over the whole GPU this way).  The unit's first
//    CTA records (its slot, the unit's last CTA) in unit_info.
#pragma once

#include "gqa_params.cuh"
#include "gqa_schedule.cuh"

namespace gqa {

struct UnitMerge {
  int last;        // this CTA merges the unit
  int slot0;       // partial slot of the unit's first CTA
  int c_lo;        // the unit's first CTA
  int n;           // number of CTAs (partials) of the unit
  int reads_done;  // fused step: warps that have read the lengths for the last time
};

// Counts one more finished CTA of the unit and returns the new count.  The
// compare-and-swap loop retries only while another CTA of the same unit
// updates the word, at most once per such CTA.
__device__ __forceinline__ unsigned arrive_unit(unsigned long long *cnt, unsigned epoch) {
  unsigned long long old = *reinterpret_cast<volatile unsigned long long *>(cnt), assumed, nv;
  do {
    assumed = old;
    const unsigned c = (unsigned)(assumed >> 32) == epoch ? (unsigned)assumed : 0u;
    nv = ((unsigned long long)epoch << 32) | (unsigned long long)(c + 1);
    old = atomicCAS(cnt, assumed, nv);
  } while (old != assumed);
  return (unsigned)nv;
}

// The same count split in two halves, so that the arrival at the end of a
// kernel is one atomic add.  tag_unit_counter runs early (before this CTA's
// work on the unit): a word tagged by another call, or never written, is
// replaced by (epoch << 32) | 0 with one compare-and-swap.  If the swap
// fails another CTA of this call changed the word first, and while a call
// runs only its own CTAs write the word (with this call's tag), so either
// way the word carries the tag before any of this CTA's adds.
__device__ __forceinline__ void tag_unit_counter(unsigned long long *cnt, unsigned epoch) {
  const unsigned long long old = *reinterpret_cast<volatile unsigned long long *>(cnt);
  if ((unsigned)(old >> 32) != epoch) atomicCAS(cnt, old, (unsigned long long)epoch << 32);
}

// This CTA's arrival on a word tagged by tag_unit_counter; returns the count
// including it.
__device__ __forceinline__ unsigned add_unit_arrival(unsigned long long *cnt) {
  return (unsigned)atomicAdd(cnt, 1ull) + 1u;
}

// Called by the `nthr` threads (tid 0..nthr-1) of the group that wrote this
// CTA's partial of a split unit (heads [h_first, h_first + nh) of batch row
// b), after those writes; `bar` synchronises the group.  When this CTA is the
// unit's last, the group merges all its partials into out.
template <typename T, int D, bool MULTI, class Bar>
__device__ __forceinline__ void finish_split_unit(const SplitParams &p, const Segment &seg, const CtaRange &range,
                                                  int b, int h_first, int nh, int tid, int nthr, UnitMerge *um,
                                                  Bar bar) {
  const long long T_total = range.T;
  __threadfence();
  bar();
  if (tid == 0) {
    const int P = range.P;
    const int c_lo = cta_of_tile(seg.unit_first, T_total, P);
    const int c_hi = cta_of_tile(seg.unit_first + seg.tiles - 1, T_total, P);
    const size_t u = (size_t)b * p.G * p.head_chunks + seg.uib;
    const int n = c_hi - c_lo + 1;
    const bool last = arrive_unit(p.unit_cnt + u, p.epoch) == (unsigned)n;
    if (last) {
      __threadfence();
      atomicExch(p.unit_cnt + u, (unsigned long long)p.epoch << 32);
    }
    um->last = last;
    um->c_lo = c_lo;
    um->n = n;
    // the unit is c_lo's first segment when c_lo's range starts inside the
    // unit's span (its charge, then its tiles)
    um->slot0 = cta_start(c_lo, T_total, P) >= seg.unit_first - range.cost ? 2 * c_lo : 2 * c_lo + 1;
  }
  bar();
  if (!um->last) return;
  const int c_lo = um->c_lo, n = um->n, slot0 = um->slot0, hpc = p.heads_per_cta;
  const float2 *ml = reinterpret_cast<const float2 *>(p.ml_part);
  for (int e = tid; e < nh * (D / 4); e += nthr) {
    const int h = e / (D / 4), d0 = (e % (D / 4)) * 4;
    float M = -INFINITY;
    for (int k = 0; k < n; ++k) {
      const int slot = k == 0 ? slot0 : 2 * (c_lo + k);
      M = fmaxf(M, __ldcg(ml + (size_t)slot * hpc + h).x);
    }
    float L = 0.f, a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    for (int k = 0; k < n; ++k) {
      const size_t ps = (size_t)(k == 0 ? slot0 : 2 * (c_lo + k)) * hpc + h;
      const float2 mk = __ldcg(ml + ps);
      const float w = merge_weight(mk.x, M);
      const float4 o = __ldcg(reinterpret_cast<const float4 *>(p.o_part + ps * D + d0));
      L += w * mk.y;
      a0 += w * o.x;
      a1 += w * o.y;
      a2 += w * o.z;
      a3 += w * o.w;
    }
    const float inv = (!MULTI || L > 0.f) ? 1.f / L : 0.f;  // 0: a query row that sees no position
    if (!GQA_ROW_OK(p, query_row<MULTI>(p, b, h_first + h))) continue;
    T *dst = reinterpret_cast<T *>(p.out) + query_row<MULTI>(p, b, h_first + h) * D + d0;
    dst[0] = from_float<T>(a0 * inv);
    dst[1] = from_float<T>(a1 * inv);
    dst[2] = from_float<T>(a2 * inv);
    dst[3] = from_float<T>(a3 * inv);
  }
}

// Atomics of the fused step's counter word at GPU scope with acquire and
// release semantics: the add (or the swap) that counts a CTA releases what the
// CTA did before it (its threads' reads of the lengths, ordered by the
// barrier ahead of the arrival) and acquires what the CTAs counted earlier
// did, so the CTA that counts last may then write the lengths.
__device__ __forceinline__ unsigned long long atom_add_acq_rel(unsigned long long *a, unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], %2;" : "=l"(old) : "l"(a), "l"(v) : "memory");
  return old;
}
__device__ __forceinline__ unsigned long long atom_cas_acq_rel(unsigned long long *a, unsigned long long cmp,
                                                               unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.acq_rel.gpu.global.cas.b64 %0, [%1], %2, %3;" : "=l"(old) : "l"(a), "l"(cmp), "l"(v) : "memory");
  return old;
}

// Counts one more finished CTA of a fused decode step on the 64-bit word
// (call epoch << 32) | count and returns the new count, 1..P for the grid's
// P CTAs.  Most CTAs count with one atomic add: the add returns the word as
// it was, and if that carried this call's tag the add was the count.  An add
// that found another tag (the previous call's, or memory never cleared) went
// into a stale word; that CTA then installs (epoch << 32) | 1, counting
// itself, with a compare-and-swap, or adds again once it sees that another
// CTA installed the tag.  A stale word never takes part in the count: the
// swap replaces it whole, and after it the word keeps this call's tag to the
// end of the call.  Each failed swap follows a change of the word by another
// CTA (at most one stale add each, then the tag), so a CTA retries at most P
// times; past that bound it flags GQA_DEVERR_TIMEOUT and returns 0, never a
// valid count.  The CTA counted last is the one that returns P.
__device__ __forceinline__ unsigned arrive_step(unsigned long long *cnt, unsigned epoch) {
  const unsigned long long tagged = (unsigned long long)epoch << 32;
  unsigned long long old = atom_add_acq_rel(cnt, 1ull);
  if ((unsigned)(old >> 32) == epoch) return (unsigned)old + 1u;
  unsigned long long cur = old + 1ull;  // the word as this add left it
  for (unsigned tries = 0;; ++tries) {
    if ((unsigned)(cur >> 32) == epoch) return (unsigned)atom_add_acq_rel(cnt, 1ull) + 1u;
    if (tries > gridDim.x) {
      flag_error(GQA_DEVERR_TIMEOUT);
      return 0u;
    }
    const unsigned long long seen = atom_cas_acq_rel(cnt, cur, tagged | 1ull);
    if (seen == cur) return 1u;
    cur = seen;
  }
}

// End of a fused decode step where a kernel counts after all of its work
// (an attention instantiation, should one be asked to append: the host
// launches the step instantiations, which count early), called by all `nthr`
// threads of a CTA after that work and a barrier of the whole CTA (every CTA
// comes, busy or idle, also after a timed-out wait).  The last CTA of the grid to count
// advances seq_lens[b] to L_b + 1 for every row that took the append, and
// puts the count back to zero under the same tag (so that a graph replay of
// the call, which keeps its epoch, starts from zero too; a plain store, since
// every CTA of the call has counted).  No CTA reads the lengths after its own
// arrival, so the update cannot be seen half way through the call, and the
// lengths the last CTA reads are those the whole call read.  `flag` is a
// shared word that broadcasts thread 0's finding.
__device__ __forceinline__ void finish_step(const SplitParams &p, int tid, int nthr, volatile int *flag) {
  if (tid == 0) {
    bool last = true;
    if (p.done_cnt) {
      last = arrive_step(p.done_cnt, p.epoch) == gridDim.x;
      if (last) *reinterpret_cast<volatile unsigned long long *>(p.done_cnt) = (unsigned long long)p.epoch << 32;
    }
    *flag = last;
  }
  __syncthreads();
  if (!*flag) return;
  for (int b = tid; b < p.B; b += nthr) {
    const int L = __ldg(p.seq_lens + b);
    if (append_ok(L, p.Nmax)) p.seq_lens_w[b] = L + 1;
  }
}

// Fused step, early arrival (the step instantiations of the split kernels):
// the CTA counts on the step word as soon as none of its threads will read the
// lengths again, which is long before its work ends, so the count and the
// last CTA's update of the lengths overlap the CTAs' remaining work instead
// of following it.  Each warp (or lone thread) that walks the segments
// signals once, after its last read (the start of its last segment, or the
// end of its loop); the producer warp, whose reads end with its last copy,
// waits for those signals and counts the CTA.

// One thread that walks the segments alone: it has done its last read.
__device__ __forceinline__ void signal_lengths_read_thread(UnitMerge *um) {
  asm volatile("red.release.cta.shared::cta.add.u32 [%0], 1;" ::"r"(smem_u32(&um->reads_done)) : "memory");
}

// One warp: every lane has done its last read of the lengths.
__device__ __forceinline__ void signal_lengths_read(UnitMerge *um, int lane) {
  __syncwarp();
  if (lane == 0) signal_lengths_read_thread(um);
}

// The producer warp, after its own last read: waits (bounded) for `n`
// consumer warps' signals, then counts the CTA; the warp of the CTA counted
// last advances the lengths.  After a timed-out wait it still counts, as
// every CTA must, with GQA_DEVERR_TIMEOUT set.
__device__ __forceinline__ void arrive_step_early(const SplitParams &p, UnitMerge *um, int n, int lane) {
  int last = 0;
  if (lane == 0) {
    const uint32_t a = smem_u32(&um->reads_done);
    auto seen = [&] {
      uint32_t v;
      asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
      return (int)v;
    };
    if (seen() < n) {
      const unsigned long long t0 = global_timer_ns();
      while (seen() < n) {
        if (global_timer_ns() - t0 > kWaitLimitNs) {
          flag_error(GQA_DEVERR_TIMEOUT);
          break;
        }
        __nanosleep(100);
      }
    }
    last = p.done_cnt ? arrive_step(p.done_cnt, p.epoch) == gridDim.x : 1;
    if (last && p.done_cnt)
      *reinterpret_cast<volatile unsigned long long *>(p.done_cnt) = (unsigned long long)p.epoch << 32;
  }
  __syncwarp();
  if (!__shfl_sync(0xffffffffu, last, 0)) return;
  for (int b = lane; b < p.B; b += 32) {
    const int L = __ldg(p.seq_lens + b);
    if (append_ok(L, p.Nmax)) p.seq_lens_w[b] = L + 1;
  }
}

// Combine-mode bookkeeping of a finished segment (one thread): the unit's
// first CTA records where its partials are, or that it was finished whole.
__device__ __forceinline__ void record_unit(const SplitParams &p, const Segment &seg, bool whole, int slot,
                                            const CtaRange &range, int b) {
  if (!p.unit_info || seg.t0 != 0) return;
  const size_t u = (size_t)b * p.G * p.head_chunks + seg.uib;
  p.unit_info[u] = whole ? make_int2(-1, -1)
                         : make_int2(slot, cta_of_tile(seg.unit_first + seg.tiles - 1, range.T, range.P));
}

// One warp per (b, h): the merge of the unit that holds head h when the
// split cut it (info.y >= 0).  Whole units and empty sequences were written
// by the split kernel.  It waits for the split grid to finish before it
// reads the workspace.  The loads are batched so that a merge costs a few
// L2 round trips whatever the number of partials: the length and the unit's
// record together, then the (m, l) of up to 32 partials (one per lane), then
// the partial rows four at a time; the sums still run over k = 0, 1, ... in
// order.
template <typename T, int D>
__global__ void __launch_bounds__(128) gqa_combine_kernel(const SplitParams p) {
  constexpr int PER_LANE = D / 32;
  constexpr unsigned FULL = 0xffffffffu;
  griddep_wait();
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long bh = (long long)blockIdx.x * 4 + warp;
  if (bh >= (long long)p.B * p.H) return;
  const int b = (int)(bh / p.H), h = (int)(bh % p.H);
  const int g = h / p.n_rep, rr = h % p.n_rep;
  const int hc = rr / p.heads_per_cta, hl = rr % p.heads_per_cta;
  // (an empty sequence has no record: it is read, not used)
  const int Lraw = p.seq_lens[b];
  const int2 info = p.unit_info[((size_t)b * p.G + g) * p.head_chunks + hc];
  if (max(0, min(Lraw, p.Nmax)) == 0 || info.y < 0) return;
  const int c_lo = info.x >> 1;
  const int n = info.y - c_lo + 1;  // number of partials
  if (!GQA_IN_BOUNDS(info.x >= 0 && info.y < p.P && n >= 1) || !GQA_ROW_OK(p, query_row<true>(p, b, h))) return;
  const float2 *ml = reinterpret_cast<const float2 *>(p.ml_part);
  auto slot_of = [&](int k) { return k == 0 ? info.x : 2 * (c_lo + k); };
  float2 mine = make_float2(-INFINITY, 0.f);  // (m, l) of partial `lane`
  float M = -INFINITY;
  for (int k = lane; k < n; k += 32) {
    const float2 v = ml[(size_t)slot_of(k) * p.heads_per_cta + hl];
    if (k == lane) mine = v;
    M = fmaxf(M, v.x);
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(FULL, M, off));
  float acc[PER_LANE];
#pragma unroll
  for (int e = 0; e < PER_LANE; ++e) acc[e] = 0.f;
  float l = 0.f;
  for (int k0 = 0; k0 < n; k0 += 32) {
    // weight and weighted sum of partial k0 + lane
    const int kl = k0 + lane;
    float2 v = mine;
    if (k0 > 0) v = kl < n ? ml[(size_t)slot_of(kl) * p.heads_per_cta + hl] : make_float2(-INFINITY, 0.f);
    const float w = kl < n ? merge_weight(v.x, M) : 0.f;
    const float wl = w * v.y;
    const int cnt = min(32, n - k0);
    for (int j = 0; j < cnt; j += 4) {
      float o[4][PER_LANE];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (j + u < cnt) {
          const float *op = p.o_part + ((size_t)slot_of(k0 + j + u) * p.heads_per_cta + hl) * D + lane * PER_LANE;
          if constexpr (PER_LANE == 4) {
            const float4 t = *reinterpret_cast<const float4 *>(op);
            o[u][0] = t.x;
            o[u][1] = t.y;
            o[u][2] = t.z;
            o[u][3] = t.w;
          } else {
            const float2 t = *reinterpret_cast<const float2 *>(op);
            o[u][0] = t.x;
            o[u][1] = t.y;
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float wu = __shfl_sync(FULL, w, (j + u) & 31);
        const float lu = __shfl_sync(FULL, wl, (j + u) & 31);
        if (j + u < cnt) {
          l += lu;
#pragma unroll
          for (int e = 0; e < PER_LANE; ++e) acc[e] += wu * o[u][e];
        }
      }
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  T *o = reinterpret_cast<T *>(p.out) + query_row<true>(p, b, h) * D + lane * PER_LANE;
#pragma unroll
  for (int e = 0; e < PER_LANE; ++e) o[e] = from_float<T>(acc[e] * inv);
}

}  // namespace gqa
