// Self-test of the bounded waits: one warp waits, through the same bounded
// waits the split kernels use, on a condition that nothing will satisfy, so
// that each wait gives up after its time limit (about one second), sets
// GQA_DEVERR_TIMEOUT in the error word and returns; the kernel then ends and
// the context stays usable.  Not part of the method: it checks the error
// path that a stalled pipeline would take, without a fault or a trap.
#pragma once

#include "gqa_device.cuh"
#include "gqa_merge.cuh"
#include "gqa_split_tc.cuh"

namespace gqa {

// which = 0: the single-thread mbarrier wait (TMA producers, CUDA-core and
// warp-MMA consumers); 1: the whole-warp wait of the tcgen05 kernel's softmax
// and converter warps; 2: a fused step's producer waiting for its warps'
// signals before it counts the block (no count word, no rows to advance).
// One block of one warp.
__global__ void __launch_bounds__(32) gqa_wait_selftest_kernel(int which) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ UnitMerge um;
  const int lane = threadIdx.x & 31;
  const uint32_t b = smem_u32(&bar);
  if (lane == 0) {
    mbar_init(b, 1);  // one arrival completes phase 0, and none comes
    um.reads_done = 0;
  }
  fence_barrier_init();
  __syncwarp();
  if (which == 0) {
    if (lane == 0) mbar_wait(b, 0);
  } else if (which == 1) {
    warp_wait(b, 0);
  } else {
    SplitParams p = {};
    p.B = 0;              // no lengths to advance
    p.done_cnt = nullptr;  // a one-block grid: no count word
    arrive_step_early(p, &um, 1, lane);
  }
}

}  // namespace gqa
