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
// Persistent grid: each CTA walks its stream-K range of tiles (see
// gqa_schedule.cuh) unit by unit; at the end of a unit the four warps that
// split its positions merge their states through shared memory (their o
// slices, scaled to a common max, are summed in a fixed order).
//
// Softmax is online in fp32 and base 2: the logits are scaled by
// scale*log2(e) after the MMA, and a row's running max is only raised when a
// new tile exceeds it by more than 8 (a factor 256), so that the
// accumulator is rarely rescaled; out = O / l at the end is exact whatever
// max was used.
#pragma once

#include "gqa_merge.cuh"
#include "gqa_params.cuh"
#include "gqa_pipeline.cuh"

namespace gqa {

template <int D_, int MFW_, int WH_, int BLOCK_N_, int STAGES_, int MIN_BLOCKS_ = 1>
struct MmaCfg {
  static constexpr int D = D_;
  static constexpr int MFW = MFW_;  // 16-row head fragments per warp
  static constexpr int WH = WH_;    // warp groups along heads (4 warps each, split along positions)
  static constexpr int CONSUMER_WARPS = 4 * WH;
  static constexpr int THREADS = (CONSUMER_WARPS + 1) * 32;
  static constexpr int HEADS = 16 * MFW * WH;  // query heads per CTA
  static constexpr int UNIT_COST = 2;          // stream-K charge per unit, in tiles (gqa_schedule.cuh)
  static constexpr bool FP8 = false;           // bf16 caches only
  static constexpr int MIN_BLOCKS = MIN_BLOCKS_;  // resident CTAs per SM the register budget must allow
  using Pipe = KVPipe<D * 2 / 128, BLOCK_N_, STAGES_, CONSUMER_WARPS>;
  static constexpr int BLOCK_N = BLOCK_N_;
  static constexpr int ROWS_PER_WARP = BLOCK_N / 4;
  static constexpr int SUB = ROWS_PER_WARP / 16;  // 16-position sub-tiles per warp per stage
  static constexpr int NF = D / 8;                // n8 fragments of O
  static constexpr int KS = D / 16;               // k16 steps of S
  // per-unit merge scratch: o summed over the 4 position slices, the (m, l)
  // of each slice, and the merged (M, l) of each head
  static constexpr int OSUM_LD = D + 8;  // padded row: the fragment-ordered adds hit distinct banks
  static constexpr int OSUM_OFF = Pipe::PIPE_BYTES;
  static constexpr int ML_OFF = OSUM_OFF + HEADS * OSUM_LD * 4;
  static constexpr int FIN_OFF = ML_OFF + 4 * HEADS * 8;
  static constexpr int BAR_OFF = FIN_OFF + HEADS * 8;
  static constexpr int RANGE_OFF = BAR_OFF + 2 * Pipe::STAGES * 8;
  static constexpr int MERGE_OFF = RANGE_OFF + 64;
  static constexpr int SMEM_BYTES = 1024 + MERGE_OFF + (int)sizeof(UnitMerge);
  static_assert(ROWS_PER_WARP % 16 == 0, "each warp takes whole 16-position sub-tiles");
  static_assert(D == 64 || D == 128, "head dimension");
};

// STEP: the instantiation for the fused decode step, whose CTAs count on the
// step word as soon as no thread will read the lengths again (the others,
// compiled without that code, count after all of their work when asked to).
template <class C, bool MULTI, bool STEP = false>
__global__ void __launch_bounds__(C::THREADS, C::MIN_BLOCKS)
    gqa_split_mma_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                         const SplitParams p) {
  using Pipe = typename C::Pipe;
  constexpr int D = C::D, MFW = C::MFW, NF = C::NF, KS = C::KS;
  constexpr int NCONS = C::CONSUMER_WARPS * 32;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  Pipe pipe;
  pipe.base = smem_u32(smem);
  pipe.full0 = pipe.base + C::BAR_OFF;
  pipe.empty0 = pipe.full0 + 8 * Pipe::STAGES;
  CtaRange *range_smem = reinterpret_cast<CtaRange *>(smem + C::RANGE_OFF);
  UnitMerge *um = reinterpret_cast<UnitMerge *>(smem + C::MERGE_OFF);
  float *osum = reinterpret_cast<float *>(smem + C::OSUM_OFF);    // [HEADS][OSUM_LD]
  float2 *ml_s = reinterpret_cast<float2 *>(smem + C::ML_OFF);    // [4][HEADS]
  float2 *fin_s = reinterpret_cast<float2 *>(smem + C::FIN_OFF);  // [HEADS]
  SchedParams sp;
  sp.seq_lens = p.seq_lens;
  sp.B = p.B;
  sp.Nmax = p.Nmax;
  sp.units_per_b = p.G * p.head_chunks;
  sp.block_n = C::BLOCK_N;
  sp.append = p.append;
  sp.unit_cost = C::UNIT_COST;

  if (threadIdx.x == 0) pipe.init();
  int2 spec_lens = make_int2(-1, -1);  // warp 0: the lengths the speculative plan read
  if (warp == 0) {
    // Ahead of the wait for earlier kernels: fetch the tensor maps and ask
    // L2 for the first tiles of a speculative plan (a hint only).
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
    }
    SchedParams spx = sp;
    spx.spec = 1;
    const CtaRange r0 = warp_plan_range<true>(spx, lane, nullptr, 0, &spec_lens);
    // kept in shared memory, not registers, across the wait
    if (lane == 0) *range_smem = r0;
    if (lane == 0 && r0.begin < r0.end)
      prefetch_first_tiles(spx, r0, &tmK, &tmV, 64, Pipe::NBOX, p.G, p.head_chunks, Pipe::STAGES);
  }
  griddep_wait();  // lengths and cache rows written by earlier kernels are visible
  if (warp == 0) {
    if (!spec_plan_holds(sp, lane, spec_lens)) {
      const CtaRange r = warp_plan_range(sp, lane, p.out, (size_t)p.H * D * sizeof(__nv_bfloat16));
      if (lane == 0) *range_smem = r;
    }
  }
  if (STEP && threadIdx.x == 0) um->reads_done = 0;
  __syncthreads();
  griddep_launch_dependents();
  const CtaRange range = *range_smem;
  if (warp == C::CONSUMER_WARPS) {
    if (range.begin < range.end) produce_range(pipe, sp, range, &tmK, &tmV, 64, p.G, p.head_chunks, p, lane);
    if (STEP && p.append) arrive_step_early(p, um, C::CONSUMER_WARPS, lane);
  }
  bool lens_read = !STEP || !p.append || warp == C::CONSUMER_WARPS;  // this warp has signalled (or need not)
  if (range.begin < range.end && warp != C::CONSUMER_WARPS) {

  const int wh = warp >> 2, wn = warp & 3;
  const int gq = lane >> 2, tq = lane & 3;
  SegmentCursor cur;
  cur.init(sp, range);
  Segment seg;
  int r = 0;
  bool alive = true;
  for (int seg_index = 0; alive && cur.next(sp, seg); ++seg_index) {
    const int g = seg.uib / p.head_chunks, hc = seg.uib % p.head_chunks;
    const int b = seg.b;
    const int h_first = g * p.n_rep + hc * C::HEADS;
    const int nh = min(C::HEADS, p.n_rep - hc * C::HEADS);
    const int L = attn_len(p.seq_lens, b, p.Nmax, p.append);
    if (STEP && !lens_read && cur.end - cur.pos <= cur.cost) {
      // a fused step, and the CTA's last segment: the cursor now ends on a
      // unit boundary (or the range's end) with at most a unit's charge
      // left, so no real tile follows and it reads no more lengths
      signal_lengths_read(um, lane);
      lens_read = true;
    }

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
          const size_t row = query_row<MULTI>(p, b, h_first + (ok ? hl : 0)) * (D / 2);
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            qa[mf][ks][half] = ok ? __ldg(q32 + row + ks * 8 + tq) : 0u;
            qa[mf][ks][2 + half] = ok ? __ldg(q32 + row + ks * 8 + 4 + tq) : 0u;
          }
        }
    }

    // positions n < lim of each of this thread's rows are visible to it
    // (L, less the later tokens of the row's own run)
    int lim[MFW][2];
#pragma unroll
    for (int mf = 0; mf < MFW; ++mf)
#pragma unroll
      for (int rh = 0; rh < 2; ++rh) {
        const int hl = wh * 16 * MFW + mf * 16 + gq + 8 * rh;
        lim[mf][rh] = L - query_lag<MULTI>(p, h_first + (hl < nh ? hl : 0));
      }
    const int L_all = L - (p.tokens - 1);  // positions below this are visible to every row

    float o[MFW][NF][4];
    float m_run[MFW][2], l_run[MFW][2];
#pragma unroll
    for (int mf = 0; mf < MFW; ++mf) {
#pragma unroll
      for (int nf = 0; nf < NF; ++nf) o[mf][nf][0] = o[mf][nf][1] = o[mf][nf][2] = o[mf][nf][3] = 0.f;
      m_run[mf][0] = m_run[mf][1] = -INFINITY;
      l_run[mf][0] = l_run[mf][1] = 0.f;
    }

    for (int t = seg.t0; t < seg.t1; ++t, ++r) {
      if (!pipe.wait_full(r)) {
        alive = false;
        break;
      }
      const int st = r % Pipe::STAGES;
      const uint32_t kt = pipe.k_tile(st), vt = pipe.v_tile(st);
      const int n0 = t * C::BLOCK_N;
      const int end = min(n0 + C::BLOCK_N, L);
      const bool tail = n0 + C::BLOCK_N > (MULTI ? L_all : end);
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

        // scale to log2 units, mask positions a row may not see, row max
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
                x = tok < (MULTI ? lim[mf][e >> 1] : end) ? x : -INFINITY;
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
      if (lane == 0) pipe.release(r);
    }

    // ---- epilogue: merge the four position slices of each head group
#pragma unroll
    for (int mf = 0; mf < MFW; ++mf)
#pragma unroll
      for (int rh = 0; rh < 2; ++rh) {
        l_run[mf][rh] += __shfl_xor_sync(0xffffffffu, l_run[mf][rh], 1);
        l_run[mf][rh] += __shfl_xor_sync(0xffffffffu, l_run[mf][rh], 2);
        if (tq == 0) {
          const int hl = wh * 16 * MFW + mf * 16 + gq + 8 * rh;
          ml_s[wn * C::HEADS + hl] = make_float2(m_run[mf][rh], l_run[mf][rh]);
        }
      }
    alive = consumer_bar_and(NCONS, alive);
    float w[MFW][2];
#pragma unroll
    for (int mf = 0; mf < MFW; ++mf)
#pragma unroll
      for (int rh = 0; rh < 2; ++rh) {
        const int hl = wh * 16 * MFW + mf * 16 + gq + 8 * rh;
        float M = -INFINITY;
#pragma unroll
        for (int k = 0; k < 4; ++k) M = fmaxf(M, ml_s[k * C::HEADS + hl].x);
        w[mf][rh] = merge_weight(m_run[mf][rh], M);
        if (wn == 0 && tq == 0) {
          float l = 0.f;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 mk = ml_s[k * C::HEADS + hl];
            l += mk.y * merge_weight(mk.x, M);
          }
          fin_s[hl] = make_float2(M, l);
        }
      }
    // the four position slices add their scaled o into osum in a fixed order
    // (slice 0 stores, slices 1..3 add), so that results are reproducible
#pragma unroll 1
    for (int k = 0; k < 4; ++k) {
      if (wn == k) {
#pragma unroll
        for (int mf = 0; mf < MFW; ++mf)
#pragma unroll
          for (int rh = 0; rh < 2; ++rh) {
            float *orow = osum + (wh * 16 * MFW + mf * 16 + gq + 8 * rh) * C::OSUM_LD + 2 * tq;
#pragma unroll
            for (int nf = 0; nf < NF; ++nf) {
              float2 v = make_float2(o[mf][nf][2 * rh] * w[mf][rh], o[mf][nf][2 * rh + 1] * w[mf][rh]);
              if (k > 0) {
                const float2 prev = *reinterpret_cast<const float2 *>(orow + nf * 8);
                v.x += prev.x;
                v.y += prev.y;
              }
              *reinterpret_cast<float2 *>(orow + nf * 8) = v;
            }
          }
      }
      consumer_bar_sync(NCONS);
    }

    // ---- write the unit's result (whole unit) or its partial state
    const bool whole = seg.t0 == 0 && seg.t1 == seg.tiles;
    const int slot = partial_slot(seg_index);
    for (int i = threadIdx.x; i < nh * (D / 8); i += NCONS) {
      const int hl = i / (D / 8), d0 = (i % (D / 8)) * 8;
      const float *src = osum + hl * C::OSUM_LD + d0;
      const float4 a = *reinterpret_cast<const float4 *>(src);
      const float4 c = *reinterpret_cast<const float4 *>(src + 4);
      if (whole) {
        const float inv = (!MULTI || fin_s[hl].y > 0.f) ? 1.f / fin_s[hl].y : 0.f;
        uint4 pk;
        pk.x = pack_bf16x2(a.x * inv, a.y * inv);
        pk.y = pack_bf16x2(a.z * inv, a.w * inv);
        pk.z = pack_bf16x2(c.x * inv, c.y * inv);
        pk.w = pack_bf16x2(c.z * inv, c.w * inv);
        if (GQA_ROW_OK(p, query_row<MULTI>(p, b, h_first + hl)))
          *reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(p.out) +
                                     query_row<MULTI>(p, b, h_first + hl) * D + d0) = pk;
      } else {
        float *dst = p.o_part + ((size_t)slot * p.heads_per_cta + hl) * D + d0;
        if (GQA_SLOT_OK(p, slot, hl)) {
          *reinterpret_cast<float4 *>(dst) = a;
          *reinterpret_cast<float4 *>(dst + 4) = c;
        }
      }
    }
    if (!whole)
      for (int hl = threadIdx.x; hl < nh; hl += NCONS)
        reinterpret_cast<float2 *>(p.ml_part)[(size_t)slot * p.heads_per_cta + hl] = fin_s[hl];
    if (threadIdx.x == 0) record_unit(p, seg, whole, slot, range, b);
    if (!whole && p.unit_cnt)
      finish_split_unit<__nv_bfloat16, D, MULTI>(p, seg, range, b, h_first, nh, threadIdx.x, NCONS, um,
                                          [] { consumer_bar_sync(NCONS); });
    consumer_bar_sync(NCONS);  // scratch free for the next unit
  }
  }
  if constexpr (STEP) {
    if (!lens_read) signal_lengths_read(um, lane);  // empty range, or a timed-out wait ended the loop
  } else if (p.append) {
    __syncthreads();
    finish_step(p, threadIdx.x, blockDim.x, &um->last);
  }
}

}  // namespace gqa
