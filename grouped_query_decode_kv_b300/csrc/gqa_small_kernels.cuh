// The small kernels of the path: log-sum-exp combine of the split partials,
// the KV-cache append of one decode step, and the MHA -> GQA mean-pool of
// projection weights.
#pragma once

#include "gqa_device.cuh"
#include "gqa_params.cuh"

namespace gqa {

template <typename T>
__device__ __forceinline__ T from_float(float x);
template <>
__device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }
template <>
__device__ __forceinline__ float from_float<float>(float x) { return x; }

template <typename T>
__device__ __forceinline__ float to_float(T x);
template <>
__device__ __forceinline__ float to_float<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }
template <>
__device__ __forceinline__ float to_float<float>(float x) { return x; }

// One warp per (b, h): merge the partial softmax states of the unit that
// holds head h when the stream-K split cut that unit between CTAs:
//   out = sum_k 2^(m_k - M) o_k / sum_k 2^(m_k - M) l_k,  M = max_k m_k,
// over the unit's partials (slot info.x of its first CTA, then slot 2c of
// every later CTA c up to info.y).  Units finished inside one CTA
// (info.y < 0) and empty sequences were written by the split kernel.
// Launched as a programmatic dependent of the split kernel: it waits for
// that grid to finish before reading the workspace.
template <typename T, int D>
__global__ void __launch_bounds__(128) gqa_combine_kernel(const CombineParams p) {
  constexpr int PER_LANE = D / 32;
  griddep_wait();
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long bh = (long long)blockIdx.x * 4 + warp;
  if (bh >= (long long)p.B * p.H) return;
  const int b = (int)(bh / p.H), h = (int)(bh % p.H);
  const int L = max(0, min(p.seq_lens[b], p.Nmax));
  if (L == 0) return;
  const int g = h / p.n_rep, rr = h % p.n_rep;
  const int hc = rr / p.heads_per_cta, hl = rr % p.heads_per_cta;
  const int2 info = p.unit_info[((size_t)b * p.G + g) * p.head_chunks + hc];
  if (info.y < 0) return;
  const int c_lo = info.x >> 1;
  const int n = info.y - c_lo + 1;  // number of partials
  const float2 *ml = reinterpret_cast<const float2 *>(p.ml_part);
  auto slot_of = [&](int k) { return k == 0 ? info.x : 2 * (c_lo + k); };
  float M = -INFINITY;
  for (int k = lane; k < n; k += 32) M = fmaxf(M, ml[(size_t)slot_of(k) * p.heads_per_cta + hl].x);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float acc[PER_LANE];
#pragma unroll
  for (int e = 0; e < PER_LANE; ++e) acc[e] = 0.f;
  float l = 0.f;
  for (int k = 0; k < n; ++k) {
    const size_t ps = (size_t)slot_of(k) * p.heads_per_cta + hl;
    const float2 mls = ml[ps];
    const float w = merge_weight(mls.x, M);
    l += w * mls.y;
    const float *op = p.o_part + ps * D + lane * PER_LANE;
    if constexpr (PER_LANE == 4) {
      const float4 v = *reinterpret_cast<const float4 *>(op);
      acc[0] += w * v.x; acc[1] += w * v.y; acc[2] += w * v.z; acc[3] += w * v.w;
    } else {
      const float2 v = *reinterpret_cast<const float2 *>(op);
      acc[0] += w * v.x; acc[1] += w * v.y;
    }
  }
  const float inv = 1.f / l;
  T *o = reinterpret_cast<T *>(p.out) + (size_t)bh * D + lane * PER_LANE;
#pragma unroll
  for (int e = 0; e < PER_LANE; ++e) o[e] = from_float<T>(acc[e] * inv);
}

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
