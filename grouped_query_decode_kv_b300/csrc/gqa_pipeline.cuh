// K/V streaming pipeline of the split kernels.
//
// One producer thread issues TMA tile copies of K and V (128-byte swizzled
// boxes of `block_n` positions) into a ring of STAGES shared-memory stages;
// the consumer warps wait on a per-stage "full" mbarrier (completed by the
// copies' transaction bytes) and release the stage through an "empty"
// mbarrier that counts one arrival per consumer warp.  The ring runs on
// across the units a persistent CTA visits, so the next unit's tiles stream
// in while the consumers finish the previous one.  Every wait is bounded
// (see mbar_wait).  Each K/V byte of the CTA's range is read from HBM once.
#pragma once

#include "gqa_device.cuh"
#include "gqa_params.cuh"
#include "gqa_schedule.cuh"

namespace gqa {

template <int NBOX_, int BLOCK_N_, int STAGES_, int CONSUMER_WARPS_>
struct KVPipe {
  static constexpr int NBOX = NBOX_;              // 128-byte boxes per row (d * elt / 128)
  static constexpr int BLOCK_N = BLOCK_N_;        // positions per stage
  static constexpr int STAGES = STAGES_;
  static constexpr int CONSUMER_WARPS = CONSUMER_WARPS_;
  static constexpr int BOX_BYTES = BLOCK_N * 128;
  static constexpr int TILE_BYTES = NBOX * BOX_BYTES;  // K (or V) part of a stage
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int PIPE_BYTES = STAGES * STAGE_BYTES;
  static_assert(BOX_BYTES % 1024 == 0, "swizzled boxes need 1024-byte alignment");

  uint32_t base;    // shared address of stage 0 (1024-byte aligned)
  uint32_t full0;   // shared address of full[0]; full[i] = full0 + 8*i
  uint32_t empty0;  // empty[i] = empty0 + 8*i

  __device__ __forceinline__ uint32_t k_tile(int st) const { return base + st * STAGE_BYTES; }
  __device__ __forceinline__ uint32_t v_tile(int st) const { return base + st * STAGE_BYTES + TILE_BYTES; }
  __device__ __forceinline__ uint32_t full(int st) const { return full0 + 8 * st; }
  __device__ __forceinline__ uint32_t empty(int st) const { return empty0 + 8 * st; }

  __device__ __forceinline__ void init() const {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(full(i), 1);
      mbar_init(empty(i), CONSUMER_WARPS);
    }
    fence_barrier_init();
  }

  // Producer side (one thread).  Ring slot r (counted across the whole
  // CTA) lives in stage r % STAGES; before refilling a stage the producer
  // waits until every consumer warp released its previous use.  Returns
  // false when that wait timed out.
  __device__ __forceinline__ bool acquire(int r) const {
    return r < STAGES || mbar_wait(empty(r % STAGES), ((r / STAGES) - 1) & 1);
  }

  // Copies the K and V rows [n0, n0 + BLOCK_N) of K/V head `bg` into ring
  // slot r; the stage's full barrier completes when all bytes landed.
  // Rows past the tensor's end arrive as zeros.
  __device__ __forceinline__ void load(int r, const CUtensorMap *tmK, const CUtensorMap *tmV, int box_elems,
                                       int bg, int n0, uint64_t pol) const {
    const int st = r % STAGES;
    mbar_arrive_expect_tx(full(st), STAGE_BYTES);
#pragma unroll
    for (int bx = 0; bx < NBOX; ++bx) {
      tma_load_3d(k_tile(st) + bx * BOX_BYTES, tmK, bx * box_elems, n0, bg, full(st), pol);
      tma_load_3d(v_tile(st) + bx * BOX_BYTES, tmV, bx * box_elems, n0, bg, full(st), pol);
    }
  }

  // The last tile of a unit with only `rows` (< BLOCK_N) cached positions:
  // ceil(rows / TAIL) boxes of TAIL positions from the short-box maps, so
  // that the rest of the tile is not read from HBM.  The stage's other rows
  // keep stale data: the consumers mask those positions (and clear their V
  // rows), as they do for any position past L.  Returns false (nothing
  // issued) when the whole box is as cheap.
  template <int TAIL>
  __device__ __forceinline__ bool load_tail(int r, const CUtensorMap *tmK, const CUtensorMap *tmV, int box_elems,
                                            int bg, int n0, int rows, uint64_t pol) const {
    const int n = (rows + TAIL - 1) / TAIL;
    if (n * TAIL > BLOCK_N - 2 * TAIL) return false;
    const int st = r % STAGES;
    mbar_arrive_expect_tx(full(st), 2 * NBOX * n * TAIL * 128);
    for (int j = 0; j < n; ++j) {
#pragma unroll
      for (int bx = 0; bx < NBOX; ++bx) {
        tma_load_3d(k_tile(st) + bx * BOX_BYTES + j * TAIL * 128, tmK, bx * box_elems, n0 + j * TAIL, bg, full(st), pol);
        tma_load_3d(v_tile(st) + bx * BOX_BYTES + j * TAIL * 128, tmV, bx * box_elems, n0 + j * TAIL, bg, full(st), pol);
      }
    }
    return true;
  }

  // Waits (bounded) for the last min(issued, STAGES) copies to land, so that
  // no copy is in flight when the block exits.
  __device__ __forceinline__ void drain(int issued) const {
    for (int r = (issued > STAGES ? issued - STAGES : 0); r < issued; ++r)
      if (!mbar_wait(full(r % STAGES), (r / STAGES) & 1)) break;
  }

  // Consumer side: wait until ring slot r holds its tile / release it.
  __device__ __forceinline__ bool wait_full(int r) const { return mbar_wait(full(r % STAGES), (r / STAGES) & 1); }
  __device__ __forceinline__ void release(int r) const { mbar_arrive(empty(r % STAGES)); }
};

// Fused decode step, whole producer warp: copies the new token's K and V
// rows of KV head bg (batch row b) into cache row L_b.  The CTA that loads a
// unit's last tile is the only one that reads the row, and it copies the row
// before that load (after a fence.proxy.async for the TMA to see it).
__device__ __forceinline__ void append_rows(const SplitParams &p, int b, int bg, int lane) {
  const int L = __ldg(p.seq_lens + b);
  if (!append_ok(L, p.Nmax) || !GQA_CACHE_OK(p, bg, L)) return;
  const uint4 *kn = reinterpret_cast<const uint4 *>(p.k_new) + (size_t)bg * p.row_chunks;
  const uint4 *vn = reinterpret_cast<const uint4 *>(p.v_new) + (size_t)bg * p.row_chunks;
  uint4 *kc = reinterpret_cast<uint4 *>(p.k_cache) + ((size_t)bg * p.Nmax + L) * p.row_chunks;
  uint4 *vc = reinterpret_cast<uint4 *>(p.v_cache) + ((size_t)bg * p.Nmax + L) * p.row_chunks;
  for (int i = lane; i < 2 * p.row_chunks; i += 32) {
    if (i < p.row_chunks)
      kc[i] = __ldg(kn + i);
    else
      vc[i - p.row_chunks] = __ldg(vn + i - p.row_chunks);
  }
}

__device__ __forceinline__ void fence_global_for_async_proxy() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// The producer warp's whole job: stream the K/V tiles of every segment of
// this CTA's range, in order, through the ring (lane 0 issues the copies).
// Unit u = (b, g*HC + hc) reads K/V head b*G + g.  In a fused step the warp
// also writes the appended rows: the rows of units whose last tile falls in
// the ring's first STAGES loads right before that load, all the others in one
// batch once those first loads are in flight (their latency then overlaps).
// tmK16 / tmV16 (or null): maps of the same caches with 16-position boxes,
// for the last tile of each unit (see KVPipe::load_tail).
template <class Pipe>
__device__ __forceinline__ void produce_range(const Pipe &pipe, const SchedParams &s, const CtaRange &range,
                                              const CUtensorMap *tmK, const CUtensorMap *tmV, int box_elems, int G,
                                              int HC, const SplitParams &p, int lane,
                                              const CUtensorMap *tmK16 = nullptr,
                                              const CUtensorMap *tmV16 = nullptr) {
  const uint64_t pol = l2_policy_evict_first();
  SegmentCursor cur;
  cur.init(s, range);
  Segment seg;
  int r = 0;
  bool ok = true;
  bool batch_done = !p.append;
  while (ok && cur.next(s, seg)) {
    const int bg = seg.b * G + seg.uib / HC;
    for (int t = seg.t0; t < seg.t1; ++t) {
      if (!batch_done && r == Pipe::STAGES) {
        // every remaining unit of the range whose last tile is this CTA's
        SegmentCursor rest = cur;
        Segment rs = seg;
        bool more = true;
        while (more) {
          if (rs.t1 == rs.tiles) append_rows(p, rs.b, rs.b * G + rs.uib / HC, lane);
          more = rest.next(s, rs);
        }
        fence_global_for_async_proxy();
        batch_done = true;
      }
      if (!batch_done && t == seg.tiles - 1) {
        append_rows(p, seg.b, bg, lane);
        fence_global_for_async_proxy();
      }
      __syncwarp();
      if (lane == 0) {
        ok = pipe.acquire(r);
        if (ok) {
          const int rows =
              tmK16 && t == seg.tiles - 1 ? attn_len(p.seq_lens, seg.b, p.Nmax, p.append) - t * Pipe::BLOCK_N : 0;
          if (!(rows > 0 && pipe.template load_tail<16>(r, tmK16, tmV16, box_elems, bg, t * Pipe::BLOCK_N, rows, pol)))
            pipe.load(r, tmK, tmV, box_elems, bg, t * Pipe::BLOCK_N, pol);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      ++r;
    }
  }
  if (lane == 0) pipe.drain(r);
  __syncwarp();
}

// Before the kernel may read what earlier kernels wrote (ahead of
// griddepcontrol.wait), one lane asks L2 for the first `n` tiles of the
// range a speculative plan gives this CTA, so that the first loads after
// the wait find them there.  Only a hint: a stale plan costs some bandwidth,
// never a wrong result (the real loads still come from global memory).
__device__ __forceinline__ void prefetch_first_tiles(const SchedParams &s, const CtaRange &range,
                                                     const CUtensorMap *tmK, const CUtensorMap *tmV, int box_elems,
                                                     int nbox, int G, int HC, int n) {
  SegmentCursor cur;
  cur.init(s, range);
  Segment seg;
  while (n > 0 && cur.next(s, seg)) {
    const int bg = seg.b * G + seg.uib / HC;
    for (int t = seg.t0; t < seg.t1 && n > 0; ++t, --n) {
      for (int bx = 0; bx < nbox; ++bx) {
        tma_prefetch_l2_3d(tmK, bx * box_elems, t * s.block_n, bg);
        tma_prefetch_l2_3d(tmV, bx * box_elems, t * s.block_n, bg);
      }
    }
  }
}

__device__ __forceinline__ void consumer_bar_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// Named barrier 1 over the consumer threads that also ANDs `ok` across
// them, so that every consumer warp takes the same decision after a timed
// out wait (and they keep meeting at the same barriers).
__device__ __forceinline__ bool consumer_bar_and(int nthreads, bool ok) {
  uint32_t res;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(res)
      : "r"((uint32_t)ok), "r"(nthreads)
      : "memory");
  return res != 0;
}

// Rounds the dynamic shared-memory base up to 1024 bytes.
__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
  const uint32_t a = smem_u32(p);
  return p + (((a + 1023u) & ~1023u) - a);
}

}  // namespace gqa
