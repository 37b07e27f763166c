// Q/K/V projections of the decode token on the 5th-generation tensor cores.
//
//   q[b,h,:] = x[b,:] . P_q[h]     (every query head its own weights)
//   k[b,g,:] = x[b,:] . P_k[g]     (one K and one V head per group)
//   v[b,g,:] = x[b,:] . P_v[g]
// with x [B, A] and P [heads, A, d], the per-line einsums of the CSDN blog
// on MQA/GQA, section "MQA 的推导" ('ba,had->bhd' for Q, the head axis of
// P_k / P_v shrinking to G), and the 2kiu.com explainer, section 3.2,
// steps 2-3.  With a decode batch of B <= 256 rows this is a GEMM whose M is
// tiny: its cost is reading the weights once, (H + 2G)*A*d*2 bytes.  So the
// output features are the MMA's M and the batch its N (swap-AB):
//   D^T[j, b] = sum_a P[h][a][j] * x[b][a]   M = 128 output features, N = NB
//                                            (batch padded to 16..256), K = A
//   A operand: a 64-feature (a) x 128-feature (j) tile of P exactly as TMA
//              lands it from the [heads, A, d] layout (MN-major: j runs along
//              the 128-byte rows, two boxes of 64 features; for d = 64 the
//              two boxes are two consecutive heads)
//   B operand: the matching 64-column slice of x, K-major, zeros past B
// The accumulator lives in TMEM (double-buffered across segments).
//
// Work: items = projection heads (128 output features each), each A/64
// tiles; the flat tile space is split over a persistent grid exactly as the
// attention kernels split theirs (contiguous ranges, cta_start), so every CTA
// streams the same weight bytes.  An item cut between CTAs leaves fp32
// partial sums in two workspace slots per CTA; the last of its CTAs to
// finish adds them in a fixed order and writes the bf16 result.
//
// Warp roles (192 threads, one CTA per SM): warp 0 TMA producer, warp 1 MMA
// issuer and TMEM owner, warps 2..5 epilogue.  Every wait is bounded.
#pragma once

#include "gqa_device.cuh"
#include "gqa_merge.cuh"
#include "gqa_pipeline.cuh"
#include "gqa_schedule.cuh"
#include "gqa_tcgen05.cuh"

namespace gqa {

struct ProjParams {
  void *out[3];                  // q [B,H,d], k [B,G,d], v [B,G,d], bf16
  int heads[3];                  // H, G, G
  int item_start[4];             // first item of each output; item_start[3] = all items
  int ktiles;                    // A / KT
  int B;                         // batch rows of this launch (<= NB)
  int d;                         // 64 or 128
  float *part;                   // [2P][NB][128] partial sums (null with one CTA)
  unsigned long long *item_cnt;  // [items] merge counters, (epoch << 32) | CTAs done
  unsigned epoch;
};

template <int NB_, int KT_>
struct ProjCfg {
  static constexpr int NB = NB_;                 // batch columns: N of the MMA
  static_assert(NB == 16 || NB == 32 || NB == 64 || NB == 128 || NB == 256, "batch tile");
  static constexpr int KT = KT_;                 // input features per tile
  static_assert(KT == 64 || KT == 128 || KT == 256, "tile depth");
  static constexpr int W_BOX = KT * 128;         // 64 output features x KT inputs
  static constexpr int W_TILE = 2 * W_BOX;       // 128 output features
  static constexpr int X_BOX = NB * 128;         // NB rows x 64 inputs (one 128-byte swizzle atom)
  static constexpr int X_TILE = (KT / 64) * X_BOX;
  static constexpr int STAGE_BYTES = W_TILE + X_TILE;
  static constexpr int STAGES = 196608 / STAGE_BYTES > 10 ? 10 : 196608 / STAGE_BYTES;
  static constexpr int THREADS = 192;
  static constexpr int TM_COLS = 2 * NB < 32 ? 32 : 2 * NB;  // two accumulators
  static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
  static constexpr int BAR_OFF = RING_BYTES;     // full[ST], empty[ST], acc_full[2], acc_free[2], mma_done
  static constexpr int NBAR = 2 * STAGES + 5;
  static constexpr int SLOT_OFF = BAR_OFF + NBAR * 8;  // TMEM address, merge flag
  static constexpr int SMEM_BYTES = 1024 + SLOT_OFF + 16;
  static_assert(SMEM_BYTES > 116 * 1024 && SMEM_BYTES <= 227 * 1024, "one resident CTA per SM");
};

// Item -> (output 0/1/2, index within it).
__device__ __forceinline__ int proj_output(const ProjParams &p, int item, int &idx) {
  const int s = item < p.item_start[1] ? 0 : (item < p.item_start[2] ? 1 : 2);
  idx = item - p.item_start[s];
  return s;
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    gqa_qkv_proj_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmWq,
                        const __grid_constant__ CUtensorMap tmWk, const __grid_constant__ CUtensorMap tmWv,
                        const ProjParams p) {
  constexpr int ST = C::STAGES, NB = C::NB;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t base = smem_u32(smem);
  const uint32_t full0 = base + C::BAR_OFF, empty0 = full0 + 8 * ST;
  const uint32_t acc_full0 = empty0 + 8 * ST, acc_free0 = acc_full0 + 16, mma_done = acc_free0 + 16;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::SLOT_OFF);
  volatile int *merge_flag = reinterpret_cast<volatile int *>(smem + C::SLOT_OFF + 8);
  auto full = [&](int i) { return full0 + 8 * i; };
  auto empty = [&](int i) { return empty0 + 8 * i; };

  const long long T = (long long)p.item_start[3] * p.ktiles;
  const int P = gridDim.x, c = blockIdx.x;
  const long long begin = cta_start(c, T, P), end = cta_start(c + 1, T, P);

  if (threadIdx.x == 0) {
    for (int i = 0; i < ST; ++i) {
      mbar_init(full(i), 1);
      mbar_init(empty(i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(acc_full0 + 8 * i, 1);
      mbar_init(acc_free0 + 8 * i, 4);
    }
    mbar_init(mma_done, 1);
    fence_barrier_init();
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmWq);
    tma_prefetch_desc(&tmWk);
    tma_prefetch_desc(&tmWv);
    // The weights are parameters, not results of the previous kernel: ask L2
    // for this CTA's first ring-full of weight tiles while that kernel ends
    // (a hint only; the copies after the wait read global memory).
    int item = (int)(begin / p.ktiles), t = (int)(begin % p.ktiles);
    for (long long pos = begin; pos < end && pos < begin + ST; ++pos) {
      int idx;
      const int s = proj_output(p, item, idx);
      const CUtensorMap *tm = s == 0 ? &tmWq : (s == 1 ? &tmWk : &tmWv);
      if (p.d == 128) {
        tma_prefetch_l2_3d(tm, 0, t * C::KT, idx);
        tma_prefetch_l2_3d(tm, 64, t * C::KT, idx);
      } else {
        tma_prefetch_l2_3d(tm, 0, t * C::KT, 2 * idx);
        tma_prefetch_l2_3d(tm, 0, t * C::KT, 2 * idx + 1);
      }
      if (++t == p.ktiles) {
        t = 0;
        ++item;
      }
    }
  }
  if (warp == 1) {
    tc::tmem_alloc(smem_u32(tmem_slot), C::TM_COLS);
    tc::tmem_relinquish();
  }
  griddep_wait();  // x written by an earlier kernel is visible
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  griddep_launch_dependents();
  const uint32_t tmem = *tmem_slot;

  if (begin < end) {
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        const uint64_t pol = l2_policy_evict_first();
        int item = (int)(begin / p.ktiles), t = (int)(begin % p.ktiles), idx;
        int s = proj_output(p, item, idx);
        const CUtensorMap *tm = s == 0 ? &tmWq : (s == 1 ? &tmWk : &tmWv);
        int r = 0;
        for (long long pos = begin; pos < end; ++pos, ++r) {
          const int st = r % ST;
          if (r >= ST && !mbar_wait(empty(st), ((r / ST) - 1) & 1)) break;
          mbar_arrive_expect_tx(full(st), C::STAGE_BYTES);
          const uint32_t wt = base + st * C::STAGE_BYTES;
          if (p.d == 128) {
            tma_load_3d(wt, tm, 0, t * C::KT, idx, full(st), pol);
            tma_load_3d(wt + C::W_BOX, tm, 64, t * C::KT, idx, full(st), pol);
          } else {  // two heads of 64 features; past the last head the box reads zeros
            tma_load_3d(wt, tm, 0, t * C::KT, 2 * idx, full(st), pol);
            tma_load_3d(wt + C::W_BOX, tm, 0, t * C::KT, 2 * idx + 1, full(st), pol);
          }
#pragma unroll
          for (int xb = 0; xb < C::KT / 64; ++xb)
            tma_load_2d(wt + C::W_TILE + xb * C::X_BOX, &tmX, t * C::KT + xb * 64, 0, full(st));
          if (++t == p.ktiles) {
            t = 0;
            ++item;
            s = proj_output(p, item, idx);
            tm = s == 0 ? &tmWq : (s == 1 ? &tmWk : &tmWv);
          }
        }
        // copies still in flight land before the CTA may end (bounded)
        for (int q = (r > ST ? r - ST : 0); q < r; ++q)
          if (!mbar_wait(full(q % ST), (q / ST) & 1)) break;
      }
      __syncwarp();
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        constexpr uint32_t IDESC = tc::idesc_bf16_f32(128, NB, true, false);
        int r = 0, seg = 0;
        bool ok = true;
        long long pos = begin;
        while (ok && pos < end) {
          const int item = (int)(pos / p.ktiles), t0 = (int)(pos % p.ktiles);
          const int t1 = (int)min((long long)p.ktiles, t0 + (end - pos));
          const int buf = seg & 1;
          if (seg >= 2 && !mbar_wait(acc_free0 + 8 * buf, ((seg >> 1) - 1) & 1)) break;
          tc::fence_after();
          for (int t = t0; t < t1; ++t, ++r) {
            const int st = r % ST;
            if (!mbar_wait(full(st), (r / ST) & 1)) {
              ok = false;
              break;
            }
            tc::fence_after();
            const uint32_t wt = base + st * C::STAGE_BYTES, xt = wt + C::W_TILE;
#pragma unroll
            for (int ks = 0; ks < C::KT / 16; ++ks) {
              const uint64_t a = tc::smem_desc_sw128(wt + ks * 2048, C::W_BOX, 1024);
              const uint64_t b = tc::smem_desc_sw128(xt + (ks >> 2) * C::X_BOX + (ks & 3) * 32, 16, 1024);
              tc::mma_ss(tmem + buf * NB, a, b, IDESC, t > t0 || ks > 0);
            }
            tc::commit(empty(st));
          }
          if (!ok) break;
          tc::commit(acc_full0 + 8 * buf);
          pos += t1 - t0;
          ++seg;
          (void)item;
        }
        // nothing of this thread's may still run when TMEM is freed
        tc::commit(mma_done);
        mbar_wait(mma_done, 0);
      }
      __syncwarp();
    } else {
      // ------------------------------------------------------------ epilogue
      const int sub = warp & 3;       // TMEM lane quarter of this warp
      const int R = 32 * sub + lane;  // TMEM lane: output feature of the 128-feature tile
      const uint32_t trow = tmem + ((uint32_t)(32 * sub) << 16);
      bool dead = false;
      int seg = 0;
      long long pos = begin;
      if (R == 0 && p.item_cnt) {
        // only the range's first and last items can be cut: tag their
        // counters now, off the path of the end-of-range arrival
        const int i0 = (int)(begin / p.ktiles), i1 = (int)((end - 1) / p.ktiles);
        const int t0 = (int)(begin - (long long)i0 * p.ktiles), e1 = (int)(end - (long long)i1 * p.ktiles);
        if (t0 != 0 || (i0 == i1 && e1 != p.ktiles)) tag_unit_counter(p.item_cnt + i0, p.epoch);
        if (i1 != i0 && e1 != p.ktiles) tag_unit_counter(p.item_cnt + i1, p.epoch);
      }
      while (pos < end) {
        const int item = (int)(pos / p.ktiles), t0 = (int)(pos % p.ktiles);
        const int t1 = (int)min((long long)p.ktiles, t0 + (end - pos));
        const int buf = seg & 1;
        if (!dead && !__all_sync(0xffffffffu, mbar_wait(acc_full0 + 8 * buf, (seg >> 1) & 1))) dead = true;
        tc::fence_after();
        int idx;
        const int s = proj_output(p, item, idx);
        // feature R of the tile: head idx (d = 128) or 2*idx + R/64 (d = 64)
        const int head = p.d == 128 ? idx : 2 * idx + (R >> 6);
        const int j = p.d == 128 ? R : (R & 63);
        const bool real = head < p.heads[s];
        __nv_bfloat16 *out = reinterpret_cast<__nv_bfloat16 *>(p.out[s]);
        const bool whole = t0 == 0 && t1 == p.ktiles;
        const int slot = 2 * c + (seg == 0 ? 0 : 1);
#pragma unroll 1
        for (int n0 = 0; n0 < NB; n0 += 16) {
          uint32_t v[32];
          tc::ld_32x32b_x16(trow + buf * NB + n0, v);
          tc::wait_ld();
#pragma unroll
          for (int n = 0; n < 16; ++n) {
            const int b = n0 + n;
            if (b < p.B) {
              const float f = __uint_as_float(v[n]);
              if (whole) {
                if (real) out[((size_t)b * p.heads[s] + head) * p.d + j] = __float2bfloat16_rn(f);
              } else {
                p.part[((size_t)slot * NB + b) * 128 + R] = f;
              }
            }
          }
        }
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_free0 + 8 * buf);
        if (!whole) {
          // the last CTA of a cut item adds its partials in a fixed order
          __threadfence();
          asm volatile("bar.sync 2, 128;" ::: "memory");
          const long long first = (long long)item * p.ktiles;
          const int c_lo = cta_of_tile(first, T, P), c_hi = cta_of_tile(first + p.ktiles - 1, T, P);
          if (R == 0) {
            const bool last = add_unit_arrival(p.item_cnt + item) == (unsigned)(c_hi - c_lo + 1);
            if (last) {
              __threadfence();
              atomicExch(p.item_cnt + item, (unsigned long long)p.epoch << 32);
            }
            *merge_flag = last;
          }
          asm volatile("bar.sync 2, 128;" ::: "memory");
          if (*merge_flag) {
            // 16 batch rows of up to four partials at a time, so that their
            // 64 independent L2 loads are in flight together; the partials
            // are still added in slot order
            const int slot0 = cta_start(c_lo, T, P) == first ? 2 * c_lo : 2 * c_lo + 1;
            const int nparts = c_hi - c_lo + 1;
            for (int b0 = 0; b0 < p.B; b0 += 16) {
              float acc[16];
#pragma unroll
              for (int n = 0; n < 16; ++n) acc[n] = 0.f;
              for (int k0 = 0; k0 < nparts; k0 += 4) {
                float v[4][16];
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                  const int k = k0 + kk;
                  const float *src = p.part + ((size_t)(k == 0 ? slot0 : 2 * (c_lo + k)) * NB + b0) * 128 + R;
#pragma unroll
                  for (int n = 0; n < 16; ++n) v[kk][n] = k < nparts && b0 + n < p.B ? __ldcg(src + (size_t)n * 128) : 0.f;
                }
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                  for (int n = 0; n < 16; ++n)
                    if (k0 + kk < nparts) acc[n] += v[kk][n];
              }
#pragma unroll
              for (int n = 0; n < 16; ++n)
                if (real && b0 + n < p.B)
                  out[((size_t)(b0 + n) * p.heads[s] + head) * p.d + j] = __float2bfloat16_rn(acc[n]);
            }
          }
          asm volatile("bar.sync 2, 128;" ::: "memory");  // merge_flag is reused
        }
        pos += t1 - t0;
        ++seg;
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    tc::tmem_dealloc(tmem, C::TM_COLS);
  }
}

}  // namespace gqa
