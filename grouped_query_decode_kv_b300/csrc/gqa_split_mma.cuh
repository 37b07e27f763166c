// Split-KV GQA decode kernel on warp-level bf16 tensor-core MMA
// (mma.sync m16n8k16), for groups of n_rep >= 3 query heads.
//
// The group's query heads are the MMA's M dimension (16 rows per fragment,
// padded when n_rep is not a multiple of 16), cached positions are N for
// S = Q.K^T and K for O += P.V, and the head dimension is K for S and N for
// O.  Each K/V tile that TMA lands in shared memory is read once by every
// warp that owns part of it and multiplies all n_rep query rows at once:
// this reuse of one K/V head by the whole group is what makes GQA cheaper
// than MHA per decode step (GQA paper, section 2.2; fogdragon's CSDN blog on
// MQA/GQA, section "MQA 的推导": the arithmetic is unchanged, the cache bytes
// shrink by n_rep).
//
// Softmax is online in fp32 and base 2: the logits are scaled by
// scale*log2(e) after the MMA, and a row's running max is only raised when a
// new tile exceeds it by more than 8 (a factor 256), so that the
// accumulator is rarely rescaled; out = O / l at the end is exact whatever
// max was used.
#pragma once

#include "gqa_params.cuh"
#include "gqa_pipeline.cuh"

namespace gqa {

template <int D_, int MFW_, int WH_, int BLOCK_N_, int STAGES_>
struct MmaCfg {
  static constexpr int D = D_;
  static constexpr int MFW = MFW_;  // 16-row head fragments per warp
  static constexpr int WH = WH_;    // warp groups along heads (4 warps each, split along positions)
  static constexpr int CONSUMER_WARPS = 4 * WH;
  static constexpr int THREADS = (CONSUMER_WARPS + 1) * 32;
  static constexpr int HEADS = 16 * MFW * WH;  // query heads per CTA
  using Pipe = KVPipe<D * 2 / 128, BLOCK_N_, STAGES_, CONSUMER_WARPS>;
  static constexpr int BLOCK_N = BLOCK_N_;
  static constexpr int ROWS_PER_WARP = BLOCK_N / 4;
  static constexpr int SUB = ROWS_PER_WARP / 16;  // 16-position sub-tiles per warp per stage
  static constexpr int NF = D / 8;                // n8 fragments of O
  static constexpr int KS = D / 16;               // k16 steps of S
  static constexpr int SLOT_WORDS = (MFW * NF * 4 + MFW * 2 * 2) * 32;
  static constexpr int EPI_BYTES = WH * 3 * SLOT_WORDS * 4;
  static constexpr int BODY_BYTES = Pipe::PIPE_BYTES > EPI_BYTES ? Pipe::PIPE_BYTES : EPI_BYTES;
  static constexpr int SMEM_BYTES = 1024 + BODY_BYTES + 2 * Pipe::STAGES * 8;
  static_assert(ROWS_PER_WARP % 16 == 0, "each warp takes whole 16-position sub-tiles");
  static_assert(D == 64 || D == 128, "head dimension");
};

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    gqa_split_mma_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                         const SplitParams p) {
  using Pipe = typename C::Pipe;
  constexpr int D = C::D, MFW = C::MFW, NF = C::NF, KS = C::KS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);

  const int s = blockIdx.x, b = blockIdx.z;
  const int g = blockIdx.y / p.head_chunks, hc = blockIdx.y % p.head_chunks;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h_first = g * p.n_rep + hc * C::HEADS;
  const int nh = min(C::HEADS, p.n_rep - hc * C::HEADS);

  int L = p.seq_lens[b];
  if ((L <= 0 || L > p.Nmax) && s == 0 && hc == 0 && threadIdx.x == 0) flag_error(GQA_DEVERR_ATTN_LEN);
  L = max(0, min(L, p.Nmax));
  if (L == 0) {  // empty sequence: out = 0
    if (s == 0) {
      __nv_bfloat16 *o = reinterpret_cast<__nv_bfloat16 *>(p.out) + ((size_t)b * p.H + h_first) * D;
      for (int i = threadIdx.x; i < nh * D; i += C::THREADS) o[i] = __float2bfloat16_rn(0.f);
    }
    return;
  }
  const int start = s * p.chunk;
  if (start >= L) return;
  const int end = min(start + p.chunk, L);
  const int ntiles = (end - start + C::BLOCK_N - 1) / C::BLOCK_N;
  const bool direct = (L + p.chunk - 1) / p.chunk == 1;

  Pipe pipe;
  pipe.base = smem_u32(smem);
  pipe.full0 = pipe.base + C::BODY_BYTES;
  pipe.empty0 = pipe.full0 + 8 * Pipe::STAGES;
  if (threadIdx.x == 0) pipe.init();
  __syncthreads();

  if (warp == C::CONSUMER_WARPS) {  // producer warp
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      pipe.produce(&tmK, &tmV, 64, b * p.G + g, start, ntiles);
    }
    return;
  }

  const int wh = warp >> 2, wn = warp & 3;
  const int gq = lane >> 2, tq = lane & 3;

  // Q fragments (A operand, row-major 16x16 per k-step), kept in registers.
  uint32_t qa[MFW][KS][4];
  {
    const uint32_t *q32 = reinterpret_cast<const uint32_t *>(p.q);
#pragma unroll
    for (int mf = 0; mf < MFW; ++mf)
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int hl = wh * 16 * MFW + mf * 16 + gq + 8 * half;
        const bool ok = hl < nh;
        const size_t row = ((size_t)b * p.H + h_first + (ok ? hl : 0)) * (D / 2);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          qa[mf][ks][half] = ok ? __ldg(q32 + row + ks * 8 + tq) : 0u;
          qa[mf][ks][2 + half] = ok ? __ldg(q32 + row + ks * 8 + 4 + tq) : 0u;
        }
      }
  }

  float o[MFW][NF][4];
  float m_run[MFW][2], l_run[MFW][2];
#pragma unroll
  for (int mf = 0; mf < MFW; ++mf) {
#pragma unroll
    for (int nf = 0; nf < NF; ++nf) o[mf][nf][0] = o[mf][nf][1] = o[mf][nf][2] = o[mf][nf][3] = 0.f;
    m_run[mf][0] = m_run[mf][1] = -INFINITY;
    l_run[mf][0] = l_run[mf][1] = 0.f;
  }

  for (int t = 0; t < ntiles; ++t) {
    const int st = t % Pipe::STAGES;
    if (!mbar_wait(pipe.full(st), (t / Pipe::STAGES) & 1)) break;
    const uint32_t kt = pipe.k_tile(st), vt = pipe.v_tile(st);
    const int n0 = start + t * C::BLOCK_N;
    const bool tail = n0 + C::BLOCK_N > end;
#pragma unroll
    for (int sub = 0; sub < C::SUB; ++sub) {
      const int r0 = wn * C::ROWS_PER_WARP + sub * 16;  // first row of this sub-tile in the stage
      const int tok0 = n0 + r0;
      if (tok0 >= end) break;  // warp-uniform
      if (tok0 + 16 > L) {
        // Rows at or past L may hold anything (NaN included); P is 0 there
        // but 0 * NaN is NaN inside the MMA, so clear those V rows first.
        const int first_bad = L - tok0;  // >= 1
        for (int i = lane; i < (16 - first_bad) * Pipe::NBOX * 8; i += 32) {
          const int row = r0 + first_bad + i / (Pipe::NBOX * 8);
          const int rest = i % (Pipe::NBOX * 8);
          const uint32_t a = vt + (rest >> 3) * Pipe::BOX_BYTES + row * 128 + (rest & 7) * 16;
          asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(a), "r"(0u) : "memory");
        }
        __syncwarp();
      }

      // S = Q . K^T for 16 positions: two n8 fragments per head fragment.
      float sacc[MFW][2][4];
#pragma unroll
      for (int mf = 0; mf < MFW; ++mf)
#pragma unroll
        for (int nf = 0; nf < 2; ++nf) sacc[mf][nf][0] = sacc[mf][nf][1] = sacc[mf][nf][2] = sacc[mf][nf][3] = 0.f;
      {
        const int row = r0 + (lane & 7) + ((lane >> 4) << 3);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          const int c16 = 2 * ks + ((lane >> 3) & 1);
          uint32_t k0, k1, k2, k3;
          ldsm_x4(swz128(kt + (c16 >> 3) * Pipe::BOX_BYTES, row, c16 & 7), k0, k1, k2, k3);
#pragma unroll
          for (int mf = 0; mf < MFW; ++mf) {
            mma_bf16_16816(sacc[mf][0], qa[mf][ks], k0, k1);
            mma_bf16_16816(sacc[mf][1], qa[mf][ks], k2, k3);
          }
        }
      }

      // scale to log2 units, mask positions outside [start, end), row max
      float tmax[MFW][2];
#pragma unroll
      for (int mf = 0; mf < MFW; ++mf) {
        tmax[mf][0] = tmax[mf][1] = -INFINITY;
#pragma unroll
        for (int nf = 0; nf < 2; ++nf)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float x = sacc[mf][nf][e] * p.scale_log2;
            if (tail) {
              const int tok = tok0 + nf * 8 + 2 * tq + (e & 1);
              x = tok < end ? x : -INFINITY;
            }
            sacc[mf][nf][e] = x;
            tmax[mf][e >> 1] = fmaxf(tmax[mf][e >> 1], x);
          }
#pragma unroll
        for (int rh = 0; rh < 2; ++rh) {
          tmax[mf][rh] = fmaxf(tmax[mf][rh], __shfl_xor_sync(0xffffffffu, tmax[mf][rh], 1));
          tmax[mf][rh] = fmaxf(tmax[mf][rh], __shfl_xor_sync(0xffffffffu, tmax[mf][rh], 2));
        }
      }
      bool need = false;
#pragma unroll
      for (int mf = 0; mf < MFW; ++mf)
#pragma unroll
        for (int rh = 0; rh < 2; ++rh) need |= tmax[mf][rh] > m_run[mf][rh] + 8.f;
      if (__any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int mf = 0; mf < MFW; ++mf)
#pragma unroll
          for (int rh = 0; rh < 2; ++rh) {
            if (tmax[mf][rh] > m_run[mf][rh] + 8.f) {
              const float corr = merge_weight(m_run[mf][rh], tmax[mf][rh]);
              m_run[mf][rh] = tmax[mf][rh];
              l_run[mf][rh] *= corr;
#pragma unroll
              for (int nf = 0; nf < NF; ++nf) {
                o[mf][nf][2 * rh] *= corr;
                o[mf][nf][2 * rh + 1] *= corr;
              }
            }
          }
      }

      // P = exp2(S - m), packed to bf16 as the A operand of O += P.V
      uint32_t pa[MFW][4];
#pragma unroll
      for (int mf = 0; mf < MFW; ++mf) {
        const float m0 = m_run[mf][0] == -INFINITY ? 0.f : m_run[mf][0];
        const float m1 = m_run[mf][1] == -INFINITY ? 0.f : m_run[mf][1];
        float pv[2][4];
#pragma unroll
        for (int nf = 0; nf < 2; ++nf) {
          pv[nf][0] = exp2f(sacc[mf][nf][0] - m0);
          pv[nf][1] = exp2f(sacc[mf][nf][1] - m0);
          pv[nf][2] = exp2f(sacc[mf][nf][2] - m1);
          pv[nf][3] = exp2f(sacc[mf][nf][3] - m1);
          l_run[mf][0] += pv[nf][0] + pv[nf][1];
          l_run[mf][1] += pv[nf][2] + pv[nf][3];
        }
        pa[mf][0] = pack_bf16x2(pv[0][0], pv[0][1]);
        pa[mf][1] = pack_bf16x2(pv[0][2], pv[0][3]);
        pa[mf][2] = pack_bf16x2(pv[1][0], pv[1][1]);
        pa[mf][3] = pack_bf16x2(pv[1][2], pv[1][3]);
      }

      // O += P . V ; V fragments through ldmatrix.trans
      {
        const int row = r0 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
        for (int dn = 0; dn < D / 16; ++dn) {
          const int c16 = 2 * dn + (lane >> 4);
          uint32_t v0, v1, v2, v3;
          ldsm_x4_trans(swz128(vt + (c16 >> 3) * Pipe::BOX_BYTES, row, c16 & 7), v0, v1, v2, v3);
#pragma unroll
          for (int mf = 0; mf < MFW; ++mf) {
            mma_bf16_16816(o[mf][2 * dn], pa[mf], v0, v1);
            mma_bf16_16816(o[mf][2 * dn + 1], pa[mf], v2, v3);
          }
        }
      }
    }
    if (tail) fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(pipe.empty(st));
  }

  // ---- epilogue: merge the four position slices of each head group
#pragma unroll
  for (int mf = 0; mf < MFW; ++mf)
#pragma unroll
    for (int rh = 0; rh < 2; ++rh) {
      l_run[mf][rh] += __shfl_xor_sync(0xffffffffu, l_run[mf][rh], 1);
      l_run[mf][rh] += __shfl_xor_sync(0xffffffffu, l_run[mf][rh], 2);
    }
  consumer_bar_sync(C::CONSUMER_WARPS * 32);  // all stages consumed: reuse them as scratch
  float *scratch = reinterpret_cast<float *>(smem);
  if (wn > 0) {
    float *slot = scratch + (wh * 3 + (wn - 1)) * C::SLOT_WORDS + lane;
    int i = 0;
#pragma unroll
    for (int mf = 0; mf < MFW; ++mf)
#pragma unroll
      for (int nf = 0; nf < NF; ++nf)
#pragma unroll
        for (int e = 0; e < 4; ++e) slot[32 * i++] = o[mf][nf][e];
#pragma unroll
    for (int mf = 0; mf < MFW; ++mf)
#pragma unroll
      for (int rh = 0; rh < 2; ++rh) {
        slot[32 * i++] = m_run[mf][rh];
        slot[32 * i++] = l_run[mf][rh];
      }
  }
  consumer_bar_sync(C::CONSUMER_WARPS * 32);
  if (wn != 0) return;

  const float *slots[3];
#pragma unroll
  for (int k = 0; k < 3; ++k) slots[k] = scratch + (wh * 3 + k) * C::SLOT_WORDS + lane;
  constexpr int ML_BASE = MFW * NF * 4;
#pragma unroll
  for (int mf = 0; mf < MFW; ++mf)
#pragma unroll
    for (int rh = 0; rh < 2; ++rh) {
      const int mi = ML_BASE + (mf * 2 + rh) * 2;
      float mk[3], lk[3];
      float M = m_run[mf][rh];
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        mk[k] = slots[k][32 * mi];
        lk[k] = slots[k][32 * (mi + 1)];
        M = fmaxf(M, mk[k]);
      }
      const float ws = merge_weight(m_run[mf][rh], M);
      float wk[3];
      float l = l_run[mf][rh] * ws;
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        wk[k] = merge_weight(mk[k], M);
        l += lk[k] * wk[k];
      }
#pragma unroll
      for (int nf = 0; nf < NF; ++nf)
#pragma unroll
        for (int e = 2 * rh; e < 2 * rh + 2; ++e) {
          const int oi = (mf * NF + nf) * 4 + e;
          float v = o[mf][nf][e] * ws;
#pragma unroll
          for (int k = 0; k < 3; ++k) v += slots[k][32 * oi] * wk[k];
          o[mf][nf][e] = v;
        }
      m_run[mf][rh] = M;
      l_run[mf][rh] = l;
    }

#pragma unroll
  for (int mf = 0; mf < MFW; ++mf)
#pragma unroll
    for (int rh = 0; rh < 2; ++rh) {
      const int hl = wh * 16 * MFW + mf * 16 + gq + 8 * rh;
      if (hl >= nh) continue;
      const size_t bh = (size_t)b * p.H + h_first + hl;
      if (direct) {
        const float inv = 1.f / l_run[mf][rh];
        uint32_t *orow = reinterpret_cast<uint32_t *>(p.out) + bh * (D / 2);
#pragma unroll
        for (int nf = 0; nf < NF; ++nf)
          orow[nf * 4 + tq] = pack_bf16x2(o[mf][nf][2 * rh] * inv, o[mf][nf][2 * rh + 1] * inv);
      } else {
        float2 *prow = reinterpret_cast<float2 *>(p.o_part + (bh * p.S_max + s) * D);
#pragma unroll
        for (int nf = 0; nf < NF; ++nf) prow[nf * 4 + tq] = make_float2(o[mf][nf][2 * rh], o[mf][nf][2 * rh + 1]);
        if (tq == 0)
          reinterpret_cast<float2 *>(p.ml_part)[bh * p.S_max + s] = make_float2(m_run[mf][rh], l_run[mf][rh]);
      }
    }
}

}  // namespace gqa
