// K/V streaming pipeline of the split kernels.
//
// One producer thread issues TMA tile copies of K and V (128-byte swizzled
// boxes of `block_n` positions) into a ring of STAGES shared-memory stages;
// the consumer warps wait on a per-stage "full" mbarrier (completed by the
// copies' transaction bytes) and release the stage through an "empty"
// mbarrier that counts one arrival per consumer warp.  Every wait is bounded
// (see mbar_wait).  Each K/V byte of the split is read from HBM once.
#pragma once

#include "gqa_device.cuh"

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

  // Producer (one thread): copies tiles [0, ntiles) of K/V head `bg`
  // starting at position n_start.  Returns after the last copy it issued has
  // landed (bounded), so that no copy is in flight when the block exits.
  __device__ __forceinline__ void produce(const CUtensorMap *tmK, const CUtensorMap *tmV, int box_elems,
                                          int bg, int n_start, int ntiles) const {
    const uint64_t pol = l2_policy_evict_first();
    int issued = 0;
    for (int t = 0; t < ntiles; ++t) {
      const int st = t % STAGES;
      if (t >= STAGES && !mbar_wait(empty(st), ((t / STAGES) - 1) & 1)) break;
      mbar_arrive_expect_tx(full(st), STAGE_BYTES);
      const int n0 = n_start + t * BLOCK_N;
#pragma unroll
      for (int bx = 0; bx < NBOX; ++bx) {
        tma_load_3d(k_tile(st) + bx * BOX_BYTES, tmK, bx * box_elems, n0, bg, full(st), pol);
        tma_load_3d(v_tile(st) + bx * BOX_BYTES, tmV, bx * box_elems, n0, bg, full(st), pol);
      }
      issued = t + 1;
    }
    // drain: the last min(issued, STAGES) copies
    for (int t = (issued > STAGES ? issued - STAGES : 0); t < issued; ++t)
      if (!mbar_wait(full(t % STAGES), (t / STAGES) & 1)) break;
  }
};

__device__ __forceinline__ void consumer_bar_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// Rounds the dynamic shared-memory base up to 1024 bytes.
__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
  const uint32_t a = smem_u32(p);
  return p + (((a + 1023u) & ~1023u) - a);
}

}  // namespace gqa
