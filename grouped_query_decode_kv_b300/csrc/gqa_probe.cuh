// Read-only streaming probes: the ceiling the decode kernels' K/V streams are
// measured against.  Not part of the method: a decode-attention call reads
// its K/V bytes once and writes almost nothing, so the bound that matters is
// how fast this GPU can stream bytes out of device memory and discard them,
// not a copy (which also writes every byte).  Two forms, the two ways the
// split kernels read:
//   mode 0  16-byte loads from every thread, eight in flight per thread;
//   mode 1  bulk asynchronous copies (the TMA engine, as the K/V pipeline
//           uses) of 32 KB chunks into a ring of shared-memory stages, one
//           CTA per SM.
// Every byte is folded into one 32-bit XOR word, so the reads cannot be
// dropped, and the word is a checksum a test can verify.
#pragma once

#include "gqa_device.cuh"

namespace gqa {

__device__ __forceinline__ uint4 ldg_stream(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// XOR of the block's values into *sink (one atomic per block).
__device__ __forceinline__ void block_xor_to(uint32_t v, uint32_t *sink, uint32_t *red) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v ^= __shfl_xor_sync(0xffffffffu, v, off);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t t = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t ^= red[w];
    atomicXor(sink, t);
  }
}

constexpr int kProbeLdgThreads = 512;

__global__ void __launch_bounds__(kProbeLdgThreads) gqa_read_ldg_kernel(const uint4 *buf, size_t n16, uint32_t *sink) {
  __shared__ uint32_t red[kProbeLdgThreads / 32];
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  uint32_t acc = 0;
  for (; i + 7 * stride < n16; i += 8 * stride) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = ldg_stream(buf + i + u * stride);
#pragma unroll
    for (int u = 0; u < 8; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  for (; i < n16; i += stride) {
    const uint4 v = ldg_stream(buf + i);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  block_xor_to(acc, sink, red);
}

constexpr int kProbeChunk = 32768;   // bytes per bulk copy
constexpr int kProbeStages = 6;
constexpr int kProbeBulkThreads = 256;
constexpr int kProbeBulkSmem = 1024 + kProbeStages * kProbeChunk + kProbeStages * 8 + 64;

__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// CTA c streams chunks c, c + P, c + 2P, ... through the ring; every thread
// folds 128 bytes of each landed chunk.  Waits are bounded: after a timeout
// the CTA stops issuing, drains what is in flight (bounded too) and leaves.
__global__ void __launch_bounds__(kProbeBulkThreads, 1) gqa_read_bulk_kernel(const uint8_t *buf, size_t chunks,
                                                                            uint32_t *sink) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base0 = smem_u32(smem_raw);
  const uint32_t base = (base0 + 1023u) & ~1023u;
  const uint32_t bars = base + kProbeStages * kProbeChunk;
  __shared__ uint32_t red[kProbeBulkThreads / 32];
  __shared__ int stop;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kProbeStages; ++s) mbar_init(bars + 8 * s, 1);
    fence_barrier_init();
    stop = 0;
  }
  __syncthreads();
  const size_t mine = chunks > blockIdx.x ? (chunks - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  auto issue = [&](size_t j) {
    const int s = (int)(j % kProbeStages);
    mbar_arrive_expect_tx(bars + 8 * s, kProbeChunk);
    bulk_load(base + s * kProbeChunk, buf + (blockIdx.x + j * gridDim.x) * (size_t)kProbeChunk, kProbeChunk,
              bars + 8 * s);
  };
  if (threadIdx.x == 0)
    for (size_t j = 0; j < mine && j < (size_t)kProbeStages; ++j) issue(j);
  uint32_t acc = 0;
  size_t j = 0;
  for (; j < mine; ++j) {
    const int s = (int)(j % kProbeStages);
    if (threadIdx.x == 0 && !mbar_wait(bars + 8 * s, (uint32_t)((j / kProbeStages) & 1))) stop = 1;
    __syncthreads();
    if (stop) break;
    const uint32_t a = base + s * kProbeChunk + threadIdx.x * 16;
#pragma unroll
    for (int q = 0; q < kProbeChunk / (kProbeBulkThreads * 16); ++q) {
      const uint4 v = lds128(a + q * kProbeBulkThreads * 16);
      acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
    __syncthreads();  // stage s is read: it may be refilled
    if (threadIdx.x == 0 && j + kProbeStages < mine) issue(j + kProbeStages);
  }
  if (threadIdx.x == 0 && stop) {
    // copies issued after j may still land: wait for them (bounded) before
    // the block leaves
    for (size_t jj = j; jj < mine && jj < j + kProbeStages; ++jj)
      if (!mbar_wait(bars + 8 * (int)(jj % kProbeStages), (uint32_t)((jj / kProbeStages) & 1))) break;
  }
  block_xor_to(acc, sink, red);
}

}  // namespace gqa
