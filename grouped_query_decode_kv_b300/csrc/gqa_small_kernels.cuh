// The small kernels of the path: the KV-cache append of one decode step and
// the MHA -> GQA mean-pool of projection weights.
#pragma once

#include "gqa_device.cuh"
#include "gqa_params.cuh"

namespace gqa {

// One block per batch row b: copy k_new[b,g,:], v_new[b,g,:] (16-byte
// chunks, bit-exact) into row L_b of every KV head, then L_b += 1.
__global__ void __launch_bounds__(256) gqa_kv_append_kernel(const uint4 *__restrict__ k_new,
                                                            const uint4 *__restrict__ v_new,
                                                            uint4 *__restrict__ k_cache,
                                                            uint4 *__restrict__ v_cache, int32_t *seq_lens,
                                                            int G, int Nmax, int chunks_per_row) {
  griddep_wait();  // launched as a programmatic dependent: earlier kernels' writes are visible
  griddep_launch_dependents();
  const int b = blockIdx.x;
  const int L = seq_lens[b];
  __syncthreads();  // every thread has read L before thread 0 may update it
  if (L < 0 || L >= Nmax) {
    if (threadIdx.x == 0) flag_error(GQA_DEVERR_APPEND_LEN);
    return;
  }
  const int per_cache = G * chunks_per_row;
  for (int i = threadIdx.x; i < 2 * per_cache; i += blockDim.x) {
    const int which = i / per_cache, rem = i % per_cache;
    const int g = rem / chunks_per_row, c = rem % chunks_per_row;
    const size_t src = ((size_t)b * G + g) * chunks_per_row + c;
    const size_t dst = (((size_t)b * G + g) * Nmax + L) * chunks_per_row + c;
    if (which == 0)
      k_cache[dst] = k_new[src];
    else
      v_cache[dst] = v_new[src];
  }
  __syncthreads();
  if (threadIdx.x == 0) seq_lens[b] = L + 1;
}

// FP8 cache append, one block per batch row b: each thread turns 16 bf16
// values of k_new[b,g,:] (or v_new) into 16 E4M3 codes, x / scale[g] in fp32
// (IEEE division) rounded to nearest even and saturated, and stores them in
// row L_b; then L_b += 1.
__global__ void __launch_bounds__(256) gqa_kv_append_fp8_kernel(const __nv_bfloat16 *__restrict__ k_new,
                                                                const __nv_bfloat16 *__restrict__ v_new,
                                                                uint8_t *__restrict__ k_cache,
                                                                uint8_t *__restrict__ v_cache,
                                                                const float *__restrict__ k_scale,
                                                                const float *__restrict__ v_scale,
                                                                int32_t *seq_lens, int G, int Nmax, int d) {
  griddep_wait();
  griddep_launch_dependents();
  const int b = blockIdx.x;
  const int L = seq_lens[b];
  __syncthreads();  // every thread has read L before thread 0 may update it
  if (L < 0 || L >= Nmax) {
    if (threadIdx.x == 0) flag_error(GQA_DEVERR_APPEND_LEN);
    return;
  }
  const int chunks = d / 16, per_cache = G * chunks;
  for (int i = threadIdx.x; i < 2 * per_cache; i += blockDim.x) {
    const int which = i / per_cache, rem = i % per_cache;
    const int g = rem / chunks, c = rem % chunks;
    const __nv_bfloat16 *src = (which == 0 ? k_new : v_new) + ((size_t)b * G + g) * d + c * 16;
    const float sc = __ldg((which == 0 ? k_scale : v_scale) + g);
    const uint4 lo = __ldg(reinterpret_cast<const uint4 *>(src)), hi = __ldg(reinterpret_cast<const uint4 *>(src) + 1);
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    uint32_t packed[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t p0 = float2_to_e4m3x2(__fdiv_rn(bf16_lo(w[2 * k]), sc), __fdiv_rn(bf16_hi(w[2 * k]), sc));
      const uint32_t p1 =
          float2_to_e4m3x2(__fdiv_rn(bf16_lo(w[2 * k + 1]), sc), __fdiv_rn(bf16_hi(w[2 * k + 1]), sc));
      packed[k] = p0 | (p1 << 16);
    }
    uint8_t *dst = (which == 0 ? k_cache : v_cache) + (((size_t)b * G + g) * Nmax + L) * d + c * 16;
    *reinterpret_cast<uint4 *>(dst) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  }
  __syncthreads();
  if (threadIdx.x == 0) seq_lens[b] = L + 1;
}

// w_out[g, e] = mean_{j < n_rep} w[g*n_rep + j, e], fp32 accumulation.
template <typename T>
__global__ void __launch_bounds__(256) gqa_meanpool_kernel(const T *__restrict__ w, T *__restrict__ w_out,
                                                           int G, int n_rep, long long per_head) {
  const long long total = (long long)G * per_head;
  const float inv = 1.f / (float)n_rep;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const long long g = i / per_head, e = i % per_head;
    float s = 0.f;
    for (int j = 0; j < n_rep; ++j) s += to_float<T>(w[(g * n_rep + j) * per_head + e]);
    w_out[i] = from_float<T>(s * inv);
  }
}

}  // namespace gqa
