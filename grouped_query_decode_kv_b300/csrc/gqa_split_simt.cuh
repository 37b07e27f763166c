// Split-KV GQA decode kernel on CUDA cores (fp32 FMA), for groups of one or
// two query heads in bf16 (MHA-like shapes, where a K/V row is used by too few
// heads to fill an MMA tile) and for every shape in fp32.
//
// Persistent grid: each CTA walks its stream-K range of tiles (see
// gqa_schedule.cuh) unit by unit, with the same TMA pipeline as the MMA
// kernel running on across units.  Inside a warp, 8 lanes share one
// cached position: lane j holds the 16-byte chunk j of every 128-byte box of
// the row (so a quarter-warp reads one full 128-byte line of the swizzled
// tile, free of bank conflicts), the q.k partial sums are reduced over the 8
// lanes with shuffles, and each 8-lane group keeps its own online-softmax
// state (running max, sum, output slice) over the positions it visits.
// The four groups of a warp and the four consumer warps are merged by
// log-sum-exp at the end of every unit, in a scratch area of its own so that
// the ring keeps filling meanwhile.
#pragma once

#include "gqa_merge.cuh"
#include "gqa_params.cuh"
#include "gqa_pipeline.cuh"

namespace gqa {

// T: cache element type; TQ: q and out element type (T unless the cache is
// FP8 E4M3, whose q and out are bf16).
template <typename T, int D_, int NH_, int BLOCK_N_, int STAGES_, typename TQ = T>
struct SimtCfg {
  using Elem = T;
  using QElem = TQ;
  static constexpr bool FP8 = sizeof(T) == 1;
  static constexpr int D = D_;
  static constexpr int NH = NH_;  // query heads per CTA
  static constexpr int ELT = sizeof(T);
  static constexpr int NBOX = D * ELT / 128;
  static constexpr int BOX_ELEMS = 128 / ELT;
  static constexpr int EPC = 16 / ELT;      // elements per 16-byte chunk
  static constexpr int EPL = NBOX * EPC;    // elements of a row held by one lane
  static_assert(EPL % 2 == 0, "pairs of elements for the packed FMA");
  static constexpr int CONSUMER_WARPS = 4;
  static constexpr int THREADS = (CONSUMER_WARPS + 1) * 32;
  static constexpr int HEADS = NH;
  static constexpr int UNIT_COST = 2;  // stream-K charge per unit, in tiles (gqa_schedule.cuh)
  using Pipe = KVPipe<NBOX, BLOCK_N_, STAGES_, CONSUMER_WARPS>;
  static constexpr int BLOCK_N = BLOCK_N_;
  static constexpr int ROWS_PER_WARP = BLOCK_N / 4;
  static constexpr int SLOT_WORDS = NH * (EPL + 2) * 8;
  static constexpr int EPI_BYTES = 3 * SLOT_WORDS * 4;
  static constexpr int EPI_OFF = Pipe::PIPE_BYTES;            // merge scratch
  static constexpr int BAR_OFF = EPI_OFF + EPI_BYTES;         // full[], empty[] mbarriers
  static constexpr int RANGE_OFF = BAR_OFF + 2 * Pipe::STAGES * 8;
  static constexpr int MERGE_OFF = RANGE_OFF + 64;
  static constexpr int SMEM_BYTES = 1024 + MERGE_OFF + (int)sizeof(UnitMerge);
  static_assert(ROWS_PER_WARP % 4 == 0, "four 8-lane groups per warp");
  static_assert(NBOX >= 1, "a row spans at least one 128-byte box");
};

// Widen the EPC elements of one 16-byte chunk to fp32.
template <typename T>
__device__ __forceinline__ void widen_chunk(const uint4 &c, float *f);

template <>
__device__ __forceinline__ void widen_chunk<__nv_bfloat16>(const uint4 &c, float *f) {
  f[0] = bf16_lo(c.x); f[1] = bf16_hi(c.x);
  f[2] = bf16_lo(c.y); f[3] = bf16_hi(c.y);
  f[4] = bf16_lo(c.z); f[5] = bf16_hi(c.z);
  f[6] = bf16_lo(c.w); f[7] = bf16_hi(c.w);
}

template <>
__device__ __forceinline__ void widen_chunk<e4m3_t>(const uint4 &c, float *f) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    e4m3x2_to_float(w[i] & 0xffffu, f[4 * i], f[4 * i + 1]);
    e4m3x2_to_float(w[i] >> 16, f[4 * i + 2], f[4 * i + 3]);
  }
}

// N consecutive elements of type T (N * sizeof(T) a multiple of 16 bytes,
// 16-byte aligned) to fp32, and back.
template <typename T, int N>
__device__ __forceinline__ void load_elems(const T *src, float *f) {
  constexpr int PER = 16 / (int)sizeof(T);
#pragma unroll
  for (int c = 0; c < N / PER; ++c) widen_chunk<T>(__ldg(reinterpret_cast<const uint4 *>(src) + c), f + c * PER);
}

template <typename T>
__device__ __forceinline__ void store_chunk(T *dst, const float *f);

template <typename T, int N>
__device__ __forceinline__ void store_elems(T *dst, const float *f) {
  constexpr int PER = 16 / (int)sizeof(T);
#pragma unroll
  for (int c = 0; c < N / PER; ++c) store_chunk<T>(dst + c * PER, f + c * PER);
}

template <>
__device__ __forceinline__ void widen_chunk<float>(const uint4 &c, float *f) {
  f[0] = __uint_as_float(c.x); f[1] = __uint_as_float(c.y);
  f[2] = __uint_as_float(c.z); f[3] = __uint_as_float(c.w);
}

// Round EPC fp32 values to T and store them as one 16-byte chunk.

template <>
__device__ __forceinline__ void store_chunk<__nv_bfloat16>(__nv_bfloat16 *dst, const float *f) {
  uint4 c;
  c.x = pack_bf16x2(f[0], f[1]);
  c.y = pack_bf16x2(f[2], f[3]);
  c.z = pack_bf16x2(f[4], f[5]);
  c.w = pack_bf16x2(f[6], f[7]);
  *reinterpret_cast<uint4 *>(dst) = c;
}

template <>
__device__ __forceinline__ void store_chunk<float>(float *dst, const float *f) {
  *reinterpret_cast<float4 *>(dst) = make_float4(f[0], f[1], f[2], f[3]);
}


// STEP: the instantiation for the fused decode step, whose CTAs count on the
// step word as soon as no thread will read the lengths again (the others,
// compiled without that code, count after all of their work when asked to).
template <class C, bool MULTI, bool STEP = false>
__global__ void __launch_bounds__(C::THREADS)
    gqa_split_simt_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                          const SplitParams p) {
  using T = typename C::Elem;
  using TQ = typename C::QElem;
  using Pipe = typename C::Pipe;
  constexpr int D = C::D, NH = C::NH, EPC = C::EPC, EPL = C::EPL, NBOX = C::NBOX;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  Pipe pipe;
  pipe.base = smem_u32(smem);
  pipe.full0 = pipe.base + C::BAR_OFF;
  pipe.empty0 = pipe.full0 + 8 * Pipe::STAGES;
  CtaRange *range_smem = reinterpret_cast<CtaRange *>(smem + C::RANGE_OFF);
  UnitMerge *um = reinterpret_cast<UnitMerge *>(smem + C::MERGE_OFF);
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
      prefetch_first_tiles(spx, r0, &tmK, &tmV, C::BOX_ELEMS, NBOX, p.G, p.head_chunks, Pipe::STAGES);
  }
  griddep_wait();  // lengths and cache rows written by earlier kernels are visible
  if (warp == 0) {
    if (!spec_plan_holds(sp, lane, spec_lens)) {
      const CtaRange r = warp_plan_range(sp, lane, p.out, (size_t)p.H * D * sizeof(TQ));
      if (lane == 0) *range_smem = r;
    }
  }
  if (STEP && threadIdx.x == 0) um->reads_done = 0;
  __syncthreads();
  griddep_launch_dependents();
  const CtaRange range = *range_smem;
  if (warp == C::CONSUMER_WARPS) {
    if (range.begin < range.end) produce_range(pipe, sp, range, &tmK, &tmV, C::BOX_ELEMS, p.G, p.head_chunks, p, lane);
    if (STEP && p.append) arrive_step_early(p, um, C::CONSUMER_WARPS, lane);
  }
  bool lens_read = !STEP || !p.append || warp == C::CONSUMER_WARPS;  // this warp has signalled (or need not)
  if (range.begin < range.end && warp != C::CONSUMER_WARPS) {

  const int tg = lane >> 3, j = lane & 7;
  float *scratch = reinterpret_cast<float *>(smem + C::EPI_OFF);
  SegmentCursor cur;
  cur.init(sp, range);
  Segment seg;
  int r = 0;  // ring slot of the next tile
  bool alive = true;
  for (int seg_index = 0; alive && cur.next(sp, seg); ++seg_index) {
    const int g = seg.uib / p.head_chunks, hc = seg.uib % p.head_chunks;
    const int b = seg.b;
    const int h_first = g * p.n_rep + hc * NH;
    const int nh = min(NH, p.n_rep - hc * NH);
    const int L = attn_len(p.seq_lens, b, p.Nmax, p.append);
    if (STEP && !lens_read && cur.end - cur.pos <= cur.cost) {
      // a fused step, and the CTA's last segment: the cursor now ends on a
      // unit boundary (or the range's end) with at most a unit's charge
      // left, so no real tile follows and it reads no more lengths
      signal_lengths_read(um, lane);
      lens_read = true;
    }
    // FP8 cache: K's per-head scale joins the logit scale, V's multiplies the
    // unit's result
    const float sl2 = C::FP8 ? p.scale_log2 * __ldg(p.k_scale + g) : p.scale_log2;
    const float vscale = C::FP8 ? __ldg(p.v_scale + g) : 1.f;

    // this lane's slice of q: element e of box bx is d = bx*BOX_ELEMS + j*EPC + e
    float qf[NH][EPL];
    int lim[NH];  // positions n < lim[h] are visible to row h
    const int L_all = L - (p.tokens - 1);  // ... and all positions below L_all to every row
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      const int hh = h_first + (h < nh ? h : 0);
      lim[h] = L - query_lag<MULTI>(p, hh);
      const TQ *qrow = reinterpret_cast<const TQ *>(p.q) + query_row<MULTI>(p, b, hh) * D;
#pragma unroll
      for (int bx = 0; bx < NBOX; ++bx) load_elems<TQ, EPC>(qrow + bx * C::BOX_ELEMS + j * EPC, &qf[h][bx * EPC]);
    }

    float acc[NH][EPL], m_run[NH], l_run[NH];
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      m_run[h] = -INFINITY;
      l_run[h] = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[h][e] = 0.f;
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
#pragma unroll 2
      for (int i = tg; i < C::ROWS_PER_WARP; i += 4) {
        const int row = warp * C::ROWS_PER_WARP + i;
        const int tok = n0 + row;
        if (n0 + warp * C::ROWS_PER_WARP + (i - tg) >= end) break;  // warp-uniform: no position of this step left
        const bool valid = tok < end;
        float kf[EPL];
#pragma unroll
        for (int bx = 0; bx < NBOX; ++bx)
          widen_chunk<T>(lds128(swz128(kt + bx * Pipe::BOX_BYTES, row, j)), &kf[bx * EPC]);
        float x[NH];
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          // bf16 / fp32: the packed two-lane fp32 FMA, even and odd elements
          // in two partial sums (measured: sweep G=32 332.6 -> 315.6 us; the
          // E4M3 instantiation measured 2 % slower with it and keeps one sum)
          float dot;
          if constexpr (C::FP8) {
            dot = 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) dot = fmaf(qf[h][e], kf[e], dot);
          } else {
            float2 d2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < EPL; e += 2)
              d2 = __ffma2_rn(make_float2(qf[h][e], qf[h][e + 1]), make_float2(kf[e], kf[e + 1]), d2);
            dot = d2.x + d2.y;
          }
          dot += __shfl_xor_sync(0xffffffffu, dot, 1);
          dot += __shfl_xor_sync(0xffffffffu, dot, 2);
          dot += __shfl_xor_sync(0xffffffffu, dot, 4);
          x[h] = dot * sl2;
        }
        if (valid) {
          const bool lagged = tok >= L_all;  // only with several tokens
          float vf[EPL];
#pragma unroll
          for (int bx = 0; bx < NBOX; ++bx)
            widen_chunk<T>(lds128(swz128(vt + bx * Pipe::BOX_BYTES, row, j)), &vf[bx * EPC]);
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            if constexpr (MULTI) {
              if (lagged && tok >= lim[h]) continue;  // a later token of row h's own run
            }
            if (x[h] > m_run[h]) {
              const float corr = merge_weight(m_run[h], x[h]);
              m_run[h] = x[h];
              l_run[h] *= corr;
#pragma unroll
              for (int e = 0; e < EPL; ++e) acc[h][e] *= corr;
            }
            const float pw = exp2f(x[h] - m_run[h]);
            l_run[h] += pw;
            if constexpr (C::FP8) {
#pragma unroll
              for (int e = 0; e < EPL; ++e) acc[h][e] = fmaf(pw, vf[e], acc[h][e]);
            } else {
              // the same FMA per element, two elements per instruction
              const float2 pw2 = make_float2(pw, pw);
#pragma unroll
              for (int e = 0; e < EPL; e += 2) {
                const float2 a = __ffma2_rn(pw2, make_float2(vf[e], vf[e + 1]), make_float2(acc[h][e], acc[h][e + 1]));
                acc[h][e] = a.x;
                acc[h][e + 1] = a.y;
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) pipe.release(r);
    }

    // ---- merge the four 8-lane groups of the warp (xor 8, xor 16)
#pragma unroll
    for (int off = 8; off <= 16; off <<= 1) {
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        const float mo = __shfl_xor_sync(0xffffffffu, m_run[h], off);
        const float lo = __shfl_xor_sync(0xffffffffu, l_run[h], off);
        const float M = fmaxf(m_run[h], mo);
        const float ws = merge_weight(m_run[h], M), wo = merge_weight(mo, M);
        l_run[h] = l_run[h] * ws + lo * wo;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          const float ao = __shfl_xor_sync(0xffffffffu, acc[h][e], off);
          acc[h][e] = acc[h][e] * ws + ao * wo;
        }
        m_run[h] = M;
      }
    }

    // ---- merge the four warps through the scratch (lanes 0..7 hold the state)
    alive = consumer_bar_and(C::CONSUMER_WARPS * 32, alive);
    if (warp > 0 && lane < 8) {
      float *slot = scratch + (warp - 1) * C::SLOT_WORDS + lane;
      int i = 0;
#pragma unroll
      for (int h = 0; h < NH; ++h) {
#pragma unroll
        for (int e = 0; e < EPL; ++e) slot[8 * i++] = acc[h][e];
        slot[8 * i++] = m_run[h];
        slot[8 * i++] = l_run[h];
      }
    }
    consumer_bar_sync(C::CONSUMER_WARPS * 32);
    if (warp == 0 && lane < 8) {
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        const int base = h * (EPL + 2);
        float mk[3], lk[3], wk[3];
        float M = m_run[h];
#pragma unroll
        for (int k = 0; k < 3; ++k) {
          const float *slot = scratch + k * C::SLOT_WORDS + lane;
          mk[k] = slot[8 * (base + EPL)];
          lk[k] = slot[8 * (base + EPL + 1)];
          M = fmaxf(M, mk[k]);
        }
        const float ws = merge_weight(m_run[h], M);
        float l = l_run[h] * ws;
#pragma unroll
        for (int k = 0; k < 3; ++k) {
          wk[k] = merge_weight(mk[k], M);
          l += lk[k] * wk[k];
        }
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          float v = acc[h][e] * ws;
#pragma unroll
          for (int k = 0; k < 3; ++k) v += scratch[k * C::SLOT_WORDS + lane + 8 * (base + e)] * wk[k];
          acc[h][e] = v;
        }
        m_run[h] = M;
        l_run[h] = l;
      }

      const bool whole = seg.t0 == 0 && seg.t1 == seg.tiles;
      const int slot = partial_slot(seg_index);
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        if (h >= nh) break;
        const size_t bh = query_row<MULTI>(p, b, h_first + h);
        if (!(whole ? GQA_ROW_OK(p, bh) : GQA_SLOT_OK(p, slot, h))) continue;
        if (whole) {
          // a row with no visible position (several tokens only) is 0
          float inv = (!MULTI || l_run[h] > 0.f) ? 1.f / l_run[h] : 0.f;
          if (C::FP8) inv *= vscale;
          TQ *orow = reinterpret_cast<TQ *>(p.out) + bh * D;
#pragma unroll
          for (int bx = 0; bx < NBOX; ++bx) {
            float f[EPC];
#pragma unroll
            for (int e = 0; e < EPC; ++e) f[e] = acc[h][bx * EPC + e] * inv;
            store_elems<TQ, EPC>(orow + bx * C::BOX_ELEMS + j * EPC, f);
          }
        } else {
          const size_t ps = (size_t)slot * p.heads_per_cta + h;
          float *prow = p.o_part + ps * D;
          if (C::FP8) {
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[h][e] *= vscale;
          }
#pragma unroll
          for (int bx = 0; bx < NBOX; ++bx)
#pragma unroll
            for (int e = 0; e < EPC; e += 4)
              *reinterpret_cast<float4 *>(prow + bx * C::BOX_ELEMS + j * EPC + e) =
                  make_float4(acc[h][bx * EPC + e], acc[h][bx * EPC + e + 1], acc[h][bx * EPC + e + 2],
                              acc[h][bx * EPC + e + 3]);
          if (j == 0) reinterpret_cast<float2 *>(p.ml_part)[ps] = make_float2(m_run[h], l_run[h]);
        }
      }
    }
    const bool whole = seg.t0 == 0 && seg.t1 == seg.tiles;
    if (threadIdx.x == 0) record_unit(p, seg, whole, partial_slot(seg_index), range, b);
    if (!whole && p.unit_cnt)
      finish_split_unit<TQ, D, MULTI>(p, seg, range, b, h_first, nh, threadIdx.x, C::CONSUMER_WARPS * 32, um,
                              [] { consumer_bar_sync(C::CONSUMER_WARPS * 32); });
    consumer_bar_sync(C::CONSUMER_WARPS * 32);  // scratch free for the next unit
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
