// Stream-K work split of one decode-attention call over a persistent grid.
//
// Work units are u = (b*G + g)*HC + hc (batch row b, KV head g, head chunk
// hc), in this order.  Every unit of batch row b holds tiles_b =
// ceil(L_b / BLOCK_N) tiles of BLOCK_N cached positions, so the call has
// T = sum_b G*HC*tiles_b tiles in one flat index space.  CTA c of a grid of
// P CTAs takes the contiguous range [start(c), start(c+1)):
//   start(c) = floor(c*T/P)   when T >= P (every range non-empty),
//   start(c) = min(c, T)      when T <  P (one tile each, the rest idle).
// So every CTA streams the same number of K/V bytes (to within one tile),
// whatever the lengths, and a range cuts a unit only at its two ends.
//
// A range is walked as segments: the part of one unit that lies in the
// range.  A segment that is a whole unit is finished in place (out written
// directly).  Otherwise it leaves a partial softmax state in a workspace
// slot: slot 2c for CTA c's first segment, 2c+1 for its last; the unit's CTAs
// are c_lo..c_hi (cta_of_tile of its first and last tile), its partials slot
// 2*c_lo or 2*c_lo+1 (the latter when the unit is not c_lo's first segment)
// and 2c for every later c, and the last of them to finish merges them
// (gqa_merge.cuh).
//
// When every non-empty sequence has the same length and there are no more
// units than CTAs, fewer than all CTAs may take part, so that range
// boundaries fall on unit boundaries (see aligned_cta_count): a CTA that ends
// one unit and starts another pays two epilogues and leaves two partials,
// which costs more than a few idle CTAs.
//
// Every unit also costs a fixed amount of work however few tiles it has (Q
// load, first-tile max, epilogue, partial), so for unequal lengths each
// non-empty unit is charged `unit_cost` extra virtual tiles ahead of its
// first real one: the flat space holds span = tiles_b + unit_cost virtual
// tiles per unit, and a CTA whose range crosses many short units gets fewer
// real tiles.  A range piece that holds only a unit's charge is no segment.
// With equal lengths (the aligned plan) the charge is 0.
//
// The lengths live in device memory, so each CTA derives T and its own
// starting row from seq_lens with a warp scan (O(B/32) steps per CTA; the
// first 64 rows are read once).
#pragma once

#include "gqa_device.cuh"

namespace gqa {

struct SchedParams {
  const int32_t *seq_lens;
  int B;
  int Nmax;
  int units_per_b;  // G * HC
  int block_n;      // positions per tile
  int append;       // fused decode step: the call appends one token first
  int unit_cost;    // extra virtual tiles charged per unit (see below)
  int cluster_k = 0;  // CTAs per thread-block cluster of the launch (0: no clusters)
  // speculative plan (before griddepcontrol.wait): lengths are read with
  // L1-bypassing loads, so that no stale copy stays in the non-coherent cache
  // for the real plan to hit
  int spec = 0;
};

__device__ __forceinline__ int clamp_len(int L, int Nmax) { return max(0, min(L, Nmax)); }

// A stored length L_b takes the step's append when 0 <= L_b < Nmax.
__device__ __forceinline__ bool append_ok(int L, int Nmax) { return L >= 0 && L < Nmax; }

// The number of cached positions attention covers for row b: the stored
// length, plus the appended token in a fused step, clamped to [0, Nmax].
__device__ __forceinline__ int attn_len(const int32_t *seq_lens, int b, int Nmax, int append) {
  const int L = __ldg(seq_lens + b);
  return clamp_len(append && append_ok(L, Nmax) ? L + 1 : L, Nmax);
}

__device__ __forceinline__ int row_tiles(const SchedParams &s, int b) {
  if (s.spec) {
    const int L = *(volatile const int32_t *)(s.seq_lens + b);
    return (clamp_len(s.append && append_ok(L, s.Nmax) ? L + 1 : L, s.Nmax) + s.block_n - 1) / s.block_n;
  }
  return (attn_len(s.seq_lens, b, s.Nmax, s.append) + s.block_n - 1) / s.block_n;
}

__device__ __forceinline__ long long cta_start(long long c, long long T, long long P) {
  if (T < P) return c < T ? c : T;
  const long long ct = c * T;
  // 32-bit division whenever the product allows (the common case)
  return ct < 0x7fffffffLL ? (long long)((int)ct / (int)P) : ct / P;
}

// The CTA whose range holds global tile t (0 <= t < T).
__device__ __forceinline__ int cta_of_tile(long long t, long long T, long long P) {
  if (T < P) return (int)t;
  return (int)(((t + 1) * P + T - 1) / T - 1);
}

__device__ __forceinline__ long long warp_incl_scan(long long v, int lane) {
  if (__all_sync(0xffffffffu, v < (1LL << 26))) {  // the 32-bit scan suffices
    int x = (int)v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += o;
    }
    return x;
  }
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const long long o = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += o;
  }
  return v;
}

// Sum of v >= 0 over the warp: one reduction instruction while every lane's
// value is small enough for its 32-bit form, else a 64-bit butterfly.
__device__ __forceinline__ long long warp_sum(long long v) {
  if (__all_sync(0xffffffffu, v < (1LL << 26))) return (long long)__reduce_add_sync(0xffffffffu, (unsigned)v);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// This CTA's place in the flat tile space, computed by one warp.
struct CtaRange {
  long long T;      // total (virtual) tiles of the call
  long long begin;  // first tile of this CTA
  long long end;    // one past its last tile
  long long pre_b;  // global index of the first tile of row b
  int b;            // row holding `begin` (valid when begin < end)
  int P;            // CTAs that take part (<= gridDim.x); the rest have empty ranges
  int cost;         // virtual tiles charged per non-empty unit
  int tiles_b;      // tiles of each unit of row b
  int cl;           // cluster plan, and this CTA's cluster has a unit: every CTA of
                    // the cluster works on a piece of that unit only (see below)
};

// First tile of piece q of a unit of `tiles` tiles cut into k pieces
// (cluster plan): floor(q * tiles / k), in 32 bits (q, k <= 8, tiles < 2^27).
__device__ __forceinline__ int piece_start(int q, int tiles, int k) { return q * tiles / k; }

// Virtual tiles of one unit of a row with `tiles` real tiles.
__device__ __forceinline__ long long unit_span(int tiles, int cost) { return tiles > 0 ? tiles + cost : 0; }

// CTAs used for T tiles when every non-empty unit holds the same number of
// tiles and there are no more units than CTAs: k = floor(P / units) CTAs per
// unit, each taking an equal piece of one unit, so that no CTA works on two
// units (two epilogues, two partials).  Measured on B300 against the plain
// split over all P CTAs: clearly faster with two CTAs per SM, where the idle
// CTAs leave no SM empty (MHA, 256 units on 296 CTAs: 78.8 against 81.4
// us), and for fused steps; with one CTA per SM, where it leaves SMs idle,
// attention alone is faster on the plain split (sweep G=4 44.6 against
// 46.0 us), which is not used yet.  With more units than CTAs, or units of
// unequal length, the plain tile-level split over all P CTAs is kept.
__device__ __forceinline__ int aligned_cta_count(long long units, int P) {
  return (units > 0 && units <= P) ? (int)(units * (P / units)) : P;
}

// All 32 lanes of one warp call this.  Also flags out-of-range lengths and
// zero-fills the output rows of empty sequences (L_b = 0) that this CTA owns
// (row b is owned by CTA b % P), writing `row_bytes` bytes per row of `out`.
// SPECULATIVE: a plan from lengths that an earlier kernel may still be
// changing, used only to pick tiles to prefetch into L2: no flags, no writes.
// `seen` (or null): the stored lengths of rows lane and 32 + lane as read
// (-1 past B), for spec_plan_holds.
template <bool SPECULATIVE = false>
__device__ __forceinline__ CtaRange warp_plan_range(const SchedParams &s, int lane, void *out, size_t row_bytes,
                                                    int2 *seen = nullptr) {
  if (seen) *seen = make_int2(-1, -1);
  const int c = blockIdx.x;
  int P = gridDim.x;
  long long T = 0;                 // real tiles
  int keep0 = 0, keep1 = 0;        // this lane's per-unit tile counts of rows lane and 32 + lane
  int tmin = 0x7fffffff, tmax = 0, rows = 0;  // per-unit tile counts of the non-empty rows
  for (int base = 0; base < s.B; base += 32) {
    const int b = base + lane;
    long long t = 0;
    int tu = 0;
    bool zero_mine = false;
    if (b < s.B) {
      const int Lstored = (SPECULATIVE || s.spec) ? *(volatile const int32_t *)(s.seq_lens + b) : __ldg(s.seq_lens + b);
      if (seen && base == 0) seen->x = Lstored;
      if (seen && base == 32) seen->y = Lstored;
      const bool appends = s.append && append_ok(Lstored, s.Nmax);
      const int Lraw = appends ? Lstored + 1 : Lstored;
      const int L = clamp_len(Lraw, s.Nmax);
      tu = (L + s.block_n - 1) / s.block_n;
      t = (long long)tu * s.units_per_b;
      const bool mine = (b % gridDim.x) == c;
      if (tu > 0) {
        tmin = min(tmin, tu);
        tmax = max(tmax, tu);
        ++rows;
      }
      if (!SPECULATIVE && mine && (Lraw <= 0 || Lraw > s.Nmax)) flag_error(GQA_DEVERR_ATTN_LEN);
      if (!SPECULATIVE && mine && s.append && !appends) flag_error(GQA_DEVERR_APPEND_LEN);
      zero_mine = !SPECULATIVE && mine && L == 0;
    }
    unsigned zero_rows = __ballot_sync(0xffffffffu, zero_mine);
    while (zero_rows) {  // warp-uniform loop over this chunk's empty rows
      const int src = __ffs(zero_rows) - 1;
      zero_rows &= zero_rows - 1;
      uint4 *o = reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(out) + (size_t)(base + src) * row_bytes);
      for (size_t i = lane; i < row_bytes / 16; i += 32) o[i] = make_uint4(0, 0, 0, 0);
    }
    if (base == 0) keep0 = tu;
    if (base == 32) keep1 = tu;
    T += warp_sum(t);
  }
  // warp-wide reductions, one instruction each (all values are >= 0)
  tmin = (int)__reduce_min_sync(0xffffffffu, (unsigned)tmin);
  tmax = (int)__reduce_max_sync(0xffffffffu, (unsigned)tmax);
  rows = (int)__reduce_add_sync(0xffffffffu, (unsigned)rows);
  const bool uniform = rows > 0 && tmin == tmax;
  CtaRange r;
  r.b = 0;
  r.pre_b = 0;
  r.tiles_b = 0;
  r.cl = 0;
  if (s.cluster_k > 1) {
    // Launched in clusters of k CTAs (the host made the grid hold k CTAs per
    // unit of a full batch): cluster j takes the j-th non-empty unit whole,
    // its CTA of rank q the tiles [floor(q*tiles/k), floor((q+1)*tiles/k)) of
    // it (possibly none), so that a unit's partials meet in one cluster.  No
    // charge.  A CTA with an empty piece still takes part in its cluster's
    // merge; r.b, r.pre_b and r.tiles_b then still name the unit.
    const int k = s.cluster_k;
    const int u = c / k;
    const int q = c - u * k;
    r.T = T;
    r.P = rows * s.units_per_b * k;
    r.cost = 0;
    r.begin = r.end = T;
    if ((long long)u >= (long long)rows * s.units_per_b) return r;  // a cluster with no unit: idle
    r.cl = 1;
    const int nr = u / s.units_per_b, uib = u - nr * s.units_per_b;
    long long acc = 0;
    int seen = 0;  // non-empty rows before this chunk
    for (int base = 0; base < s.B; base += 32) {
      const int b = base + lane;
      const int tu = base == 0 ? keep0 : base == 32 ? keep1 : (b < s.B ? row_tiles(s, b) : 0);
      const long long t = (long long)tu * s.units_per_b;
      const long long incl = warp_incl_scan(t, lane);
      const int ne = (b < s.B && tu > 0) ? 1 : 0;
      const unsigned nem = __ballot_sync(0xffffffffu, ne);
      const int rank = seen + __popc(nem & ((1u << lane) - 1u));  // non-empty rows before row b
      const unsigned hit = __ballot_sync(0xffffffffu, ne && rank == nr);
      if (hit) {
        const int src = __ffs(hit) - 1;
        r.b = base + src;
        r.pre_b = acc + __shfl_sync(0xffffffffu, incl - t, src);
        r.tiles_b = __shfl_sync(0xffffffffu, tu, src);
        const long long u0 = r.pre_b + (long long)uib * r.tiles_b;
        r.begin = u0 + piece_start(q, r.tiles_b, k);
        r.end = u0 + piece_start(q + 1, r.tiles_b, k);
        return r;
      }
      seen += __popc(nem);
      acc += __shfl_sync(0xffffffffu, incl, 31);
    }
    return r;
  }
  if (uniform) P = aligned_cta_count((long long)rows * s.units_per_b, P);
  const int cost = uniform ? 0 : s.unit_cost;
  T += (long long)cost * rows * s.units_per_b;
  r.T = T;
  r.P = P;
  r.cost = cost;
  r.begin = c < P ? cta_start(c, T, P) : T;
  r.end = c < P ? cta_start(c + 1, T, P) : T;
  if (r.begin >= r.end) return r;
  long long acc = 0;
  for (int base = 0; base < s.B; base += 32) {
    const int b = base + lane;
    const int tu = base == 0 ? keep0 : base == 32 ? keep1 : (b < s.B ? row_tiles(s, b) : 0);
    const long long t = unit_span(tu, cost) * s.units_per_b;
    const long long incl = warp_incl_scan(t, lane);
    const long long lo = acc + incl - t, hi = acc + incl;
    const unsigned hit = __ballot_sync(0xffffffffu, b < s.B && lo <= r.begin && r.begin < hi);
    if (hit) {
      const int src = __ffs(hit) - 1;
      r.b = base + src;
      r.pre_b = __shfl_sync(0xffffffffu, lo, src);
      r.tiles_b = __shfl_sync(0xffffffffu, tu, src);
      break;
    }
    acc += __shfl_sync(0xffffffffu, incl, 31);
  }
  return r;
}

// After the wait for earlier kernels: whether the plan a speculative pass
// made from the lengths `seen` (warp_plan_range<true>, before the wait) is
// this call's plan.  It is when B <= 64 (the pass read every length once,
// two rows per lane), every stored length still equals the one it read, and
// no row needs what the speculative pass leaves out (a length flag, the zero
// fill of an empty row).  The plan depends on nothing else, so the real
// pass would return the same range.  Whole warp.
__device__ __forceinline__ bool spec_plan_holds(const SchedParams &s, int lane, int2 seen) {
  if (s.B > 64) return false;
  const int b0 = lane, b1 = 32 + lane;
  const int L0 = b0 < s.B ? __ldg(s.seq_lens + b0) : -1;
  const int L1 = b1 < s.B ? __ldg(s.seq_lens + b1) : -1;
  auto clean = [&](int L) {
    const bool appends = s.append && append_ok(L, s.Nmax);
    const int Lraw = appends ? L + 1 : L;
    return Lraw > 0 && Lraw <= s.Nmax && (!s.append || appends);
  };
  const bool ok = L0 == seen.x && L1 == seen.y && (b0 >= s.B || clean(L0)) && (b1 >= s.B || clean(L1));
  return __all_sync(0xffffffffu, ok);
}

// One segment: tiles [t0, t1) of unit (b, uib) where uib = g*HC + hc.
struct Segment {
  int b, uib;
  int t0, t1;
  int tiles;             // tiles of every unit of row b
  long long unit_first;  // global (virtual) index of the unit's first real tile
};

// Walks the segments of a range; every thread that calls next() with the
// same cursor sees the same sequence.
struct SegmentCursor {
  long long pos, end, pre_b;
  int b, tiles_b, cost;

  __device__ __forceinline__ void init(const SchedParams &s, const CtaRange &r) {
    pos = r.begin;
    end = r.end;
    pre_b = r.pre_b;
    b = r.b;
    cost = r.cost;
    tiles_b = pos < end ? r.tiles_b : 0;
  }

  __device__ __forceinline__ bool next(const SchedParams &s, Segment &seg) {
    for (;;) {
      if (pos >= end) return false;
      long long span = unit_span(tiles_b, cost);
      while (pos >= pre_b + span * s.units_per_b) {
        // pos starts a row here, so a unit's charge comes first: with no
        // more than that left in the range there is no real tile, and the
        // next row's length is not read (after a CTA's last segment the
        // cursor reads no length)
        if (end - pos <= cost) return false;
        pre_b += span * s.units_per_b;
        ++b;
        tiles_b = row_tiles(s, b);
        span = unit_span(tiles_b, cost);
      }
      const long long off = pos - pre_b;
      // (32-bit division whenever the values allow: a 64-bit one is a long
      // software sequence, and this runs on every warp's start-up path)
      int uib, v0;
      if (off < 0x7fffffffLL && span < 0x7fffffffLL) {
        uib = (int)off / (int)span;
        v0 = (int)off - uib * (int)span;
      } else {
        uib = (int)(off / span);
        v0 = (int)(off % span);
      }
      const long long left = end - pos;
      const int v1 = left < span - v0 ? v0 + (int)left : (int)span;
      pos += v1 - v0;
      if (v1 <= cost) continue;  // only the unit's charge lies in the range
      seg.b = b;
      seg.uib = uib;
      seg.t0 = v0 > cost ? v0 - cost : 0;
      seg.t1 = v1 - cost;
      seg.tiles = tiles_b;
      seg.unit_first = pre_b + (long long)uib * span + cost;
      return true;
    }
  }
};

// Workspace slot of the partial of this CTA's segment number seg_index
// (only its first and last segments can be partial).
__device__ __forceinline__ int partial_slot(int seg_index) {
  return 2 * (int)blockIdx.x + (seg_index == 0 ? 0 : 1);
}

}  // namespace gqa
