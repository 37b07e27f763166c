// Split-KV GQA decode kernel on the 5th-generation tensor cores (tcgen05,
// accumulators in tensor memory), bf16, head dimension 128, for groups of
// n_rep >= 8 query heads per KV head (GQA-8 and coarser, MQA).
//
// Per tile of 128 cached positions of one unit (batch b, KV head g), with
// the group's query heads (up to 64 per unit, padded to N = 16, 32 or 64) as
// N:
//   S^T  = K_tile . Q^T     M = 128 positions, N = heads, K = d = 128
//                           A = K tile as TMA landed it (K-major, 128-byte
//                           swizzle), B = Q (K-major, swizzled by the kernel)
//   O^T += V_tile^T . P^T   M = d = 128, N = heads, K = 128 positions
//                           A = V tile as TMA landed it (MN-major: d runs
//                           along the 128-byte rows), B = P^T written by the
//                           softmax threads (MN-major: one row of N heads
//                           per position, swizzled to the row's width)
// Each K/V byte read from HBM serves every query head of the group (the
// point of GQA: GQA paper, section 2.2), and the MMA work per tile is the
// 2 x 128 x 128 x 2 x N flop, well under the tensor pipe's rate.
//
// Softmax: thread R of a group of four softmax warps owns TMEM lane R, which
// is cached position R of the tile in S^T and output dimension R in O^T.
// A configuration may give the head columns to two such groups (half each;
// the host does so for the several-token kernel with 32 rows per unit), so
// that two warps per sub-partition share the softmax.  For each of its heads
// h a thread keeps its own partial sum l_R[h]; the running max m[h] (base-2
// units) is shared by the group through shared memory.  A tile first votes
// whether any logit exceeds m[h] + 8; only then (always on a unit's first
// tile) the tile's per-head maxima are reduced across the group's 128
// threads and m moves (to the tile's maximum, or P_LIFT below it), with O^T
// rescaled in TMEM.  P = 2^(S - m) is written
// to shared memory as bf16 (double-buffered where shared memory allows, so
// that the softmax of tile t+1 need not wait for the P.V of tile t); the
// l_R[h] are summed across threads once per unit.
//
// Warp roles (one CTA per SM):
//   warp 0     TMA producer of the CTA's stream-K range (gqa_pipeline.cuh)
//   warp 1     S^T MMA issuer (one thread) and TMEM owner
//   warp 2     P.V MMA issuer (one thread)
//   warps 3..  softmax and output, in SG groups of four (group 0 also
//              loads Q); FP8 with 33-64 heads: then four converter warps
//              (8-32 heads use E4M3 MMAs on the landed tiles, no converters)
// S^T is double-buffered in TMEM so that S of tile t+1 overlaps the softmax
// of tile t; O^T is double-buffered across units.  Every mbarrier wait is
// bounded (about one second), after which the CTA winds down and flags
// GQA_DEVERR_TIMEOUT.
#pragma once

#include "gqa_merge.cuh"
#include "gqa_params.cuh"
#include "gqa_pipeline.cuh"
#include "gqa_tcgen05.cuh"

namespace gqa {

// FP8_: the cache holds E4M3 codes; four more warps convert each landed
// tile to f16 (exact): the K tile into tensor memory, where the S^T MMA
// reads it as its A operand, the V tile into one of VSTG shared-memory
// staging buffers that the P.V MMA reads; Q and P are f16 too (one operand
// type per MMA).
// F8N_ (with FP8_): no conversion at all.  Both MMAs are kind::f8f6f4 with
// E4M3 operands and K = 32 per instruction, half the instructions of the f16
// path: S^T reads the K tile as TMA landed it (K-major), P.V the V tile as
// landed (MN-major: d runs along the 128-byte rows).  Q and P, which are not
// E4M3 values, enter as two E4M3 terms each, a head's columns doubled:
//   Q[h] = (Q_hi + Q_lo / 16) / qs_h   (qs_h a power of two per head that
//                                        puts max |Q[h]| in [128, 256))
//   P    =  P_hi + P_lo / 32           (P in f16 first; both terms E4M3)
// so S^T and O^T have 2*NR columns, term 0 in [0, NR) and term 1 in
// [NR, 2*NR), combined by one FMA per head after the MMA.  The two Q terms
// hold every bf16 query exactly (4 + 4 significant bits) while qs_h keeps a
// head's elements in the E4M3 normal range.  P's range is set by where the
// running max sits: when it moves, it moves to P_LIFT = 2 (log2 units) below
// the tile's maximum, so the largest P is 2^2 and may grow to 2^8 before the
// next move.  The two terms keep 8 significant bits (bf16 P in the bf16
// path has 8) for P >= 2^-6 and reach down to P = 2^-15: a probability under
// 2^-17 of the largest one is dropped.  (A larger lift reaches further but
// leaves less room before the next move: measured, 6 made the rescales
// frequent and the calls 10-30 % slower; 2 costs nothing measurable.)
template <int NR_, int STAGES_, int PB_, bool FP8_ = false, int SG_ = 1, int VSTG_ = 2, bool F8N_ = false>
struct TcCfg {
  static constexpr bool FP8 = FP8_;
  static constexpr bool F8N = FP8_ && F8N_;          // native E4M3 MMAs, no converter warps
  static constexpr bool CONV = FP8_ && !F8N_;        // converter warps (K to TMEM, V to f16 staging)
  static constexpr int NM = F8N ? 2 * NR_ : NR_;     // N of both MMAs (two terms per head with F8N)
  static constexpr int P_LIFT = F8N ? 2 : 0;         // where a moved running max sits below the tile max
  static constexpr int VSTG = VSTG_;  // FP8: f16 V staging buffers
  static_assert(VSTG >= 2 && VSTG <= 3, "V staging buffers");
  static constexpr int D = 128;
  static constexpr int BLOCK_N = 128;  // positions per tile: M of S^T, K of P.V
  static constexpr int STAGES = STAGES_;
  static constexpr int NR = NR_;       // heads per unit, padded to a multiple of 16: N of both MMAs
  static constexpr int NQ = NR;
  static constexpr int HEADS = NR;
  static constexpr int PB = PB_;       // P^T buffers
  // stream-K charge per unit, in tiles (gqa_schedule.cuh).  A unit's fixed
  // cost takes about the same time on every path, so it is worth more of the
  // native E4M3 path's shorter tiles (FP8 GQA-8 with charge 2, 4, 6, 8:
  // 37.0, 33.0, 31.7, 32.4 us per call; bf16 GQA-8 with 2, 3, 4: 49.0,
  // 49.4, 49.7 us)
  static constexpr int UNIT_COST = F8N ? 6 : 2;
  static_assert(NR == 16 || NR == 32 || NR == 64, "heads per unit");
  static_assert(PB == 1 || PB == 2, "P^T buffers");
  // softmax groups of four warps; group j owns the head columns
  // [j*HG, (j+1)*HG) of S^T, P^T and O^T
  static constexpr int SG = SG_;
  static constexpr int HG = NR / SG;
  static_assert(SG == 1 || (SG == 2 && NR >= 32), "two softmax groups need 16+ heads each");
  static_assert(!F8N || (SG == 1 && NR <= 32), "native E4M3 path: one softmax group, up to 32 heads");
  // one "empty" arrival per tile: the MMA commit (FP8: the 4 converter warps)
  using Pipe = KVPipe<FP8 ? 1 : 2, BLOCK_N, STAGES, CONV ? 4 : 1>;
  static constexpr int SOFT_WARP0 = 3;            // first softmax warp (after producer, two MMA issuers)
  static constexpr int CONV_WARP0 = SOFT_WARP0 + 4 * SG;  // first FP8 converter warp
  static constexpr int THREADS = (CONV_WARP0 + (CONV ? 4 : 0)) * 32;
  // fused step: the signals the producer waits for before it counts the CTA
  // (the two MMA issuer threads, the softmax warps, the converter warps)
  static constexpr int LEN_READERS = 2 + 4 * SG + (CONV ? 4 : 0);
  static constexpr int KV_BOX = BLOCK_N * 128;  // one 128-byte-wide box of a bf16 K or V tile
  // FP8: V staging [2] in f16, two boxes each (d 0-63, 64-127); the f16 K
  // tiles live in tensor memory
  static constexpr int STG_OFF = Pipe::PIPE_BYTES;
  static constexpr int STG_TILE = 2 * KV_BOX;
  static constexpr int STG_BYTES = CONV ? VSTG * STG_TILE : 0;
  static constexpr int SOFT = 128;             // threads of one softmax group
  // TMEM columns: S^T buffers [0, 2*NM), O^T buffers [2*NM, 4*NM); FP8 with
  // converters: two f16 K tiles [4*NM, 4*NM + 128) (lane = position, 64
  // columns of f16 pairs)
  static constexpr int TM_S = 0;
  static constexpr int TM_O = 2 * NM;
  static constexpr int TM_K = 4 * NM;
  static constexpr int TM_USED = 4 * NM + (CONV ? 128 : 0);
  static constexpr int TM_COLS = TM_USED <= 32 ? 32 : TM_USED <= 64 ? 64 : TM_USED <= 128 ? 128 : TM_USED <= 256 ? 256 : 512;
  // shared memory
  // Q: two 128-byte-wide boxes (d 0-63, 64-127) of NR rows per buffer; two
  // buffers where shared memory allows, so that the next unit's Q lands
  // while the current one is still in use
  // F8N: each buffer holds the E4M3 operand (NM rows of 128 codes: term 0
  // of the NR heads, then term 1) and, after it, the bf16 rows as copied
  // (two boxes, as above)
  static constexpr int Q_OFF = STG_OFF + STG_BYTES;
  static constexpr int Q_BOX = NR * 128;
  static constexpr int Q_OP = F8N ? NM * 128 : 0;  // E4M3 operand bytes
  static constexpr int Q_STG = Q_OP;               // offset of the bf16 rows in a buffer
  static constexpr int Q_BYTES = Q_OP + 2 * Q_BOX;
  // P^T buffers, MN-major: one row of NR heads (2*NR bytes: bf16 or f16, or
  // with F8N the two E4M3 terms) per position, stored with the swizzle of the
  // row's width, so that the thread that owns a position writes its heads
  // with 16-byte stores
  static constexpr int P_ROW = 2 * NR;
  static constexpr int P_BYTES = BLOCK_N * P_ROW;
  static constexpr int P_SWZ_SHIFT = NR == 64 ? 0 : (NR == 32 ? 1 : 2);
  static constexpr int P_SWZ_MASK = NR == 64 ? 7 : (NR == 32 ? 3 : 1);
  // pipe full[STAGES], empty[STAGES]; then s_full[2], s_free[2], p_full[2],
  // pv_done[2], o_free[2], q_full[2], mma_done; FP8: conv_full[2], stg_free[3]
  static constexpr int NBAR = 2 * STAGES + 13 + (FP8 ? 5 : 0);
  static constexpr int RANGE_BYTES = ((int)sizeof(CtaRange) + 7) / 8 * 8;
  static constexpr int QSC_BYTES = F8N ? 2 * NQ * 4 + NQ * 4 : 0;  // F8N: 1/qs per Q buffer, logit factor per head
  static constexpr int TAIL_BYTES =
      4 * NQ * 4 + 3 * NQ * 4 + QSC_BYTES + NBAR * 8 + 8 + RANGE_BYTES + (int)sizeof(UnitMerge);
  static constexpr int QB = 1024 + Q_OFF + 2 * Q_BYTES + PB * P_BYTES + TAIL_BYTES <= 227 * 1024 ? 2 : 1;
  static constexpr int P_OFF = Q_OFF + QB * Q_BYTES;
  static constexpr int RED_OFF = P_OFF + PB * P_BYTES;  // [SG][4][HG] cross-warp reduction
  static constexpr int FIN_OFF = RED_OFF + 4 * NQ * 4;   // [NQ] reduced value
  static constexpr int M_OFF = FIN_OFF + NQ * 4;         // [NQ] running max of the unit
  static constexpr int CORR_OFF = M_OFF + NQ * 4;        // [NQ] rescale factor of a tile
  static constexpr int QSC_OFF = CORR_OFF + NQ * 4;      // F8N: [2][NQ] 1/qs_h, then [NQ] logit factor
  static constexpr int BAR_OFF = QSC_OFF + QSC_BYTES;
  static constexpr int TMEM_SLOT_OFF = BAR_OFF + NBAR * 8;
  static constexpr int RANGE_OFF = TMEM_SLOT_OFF + 8;  // 8-byte aligned (barriers before it)
  static constexpr int MERGE_OFF = RANGE_OFF + RANGE_BYTES;
  static constexpr int SMEM_BYTES = 1024 + MERGE_OFF + (int)sizeof(UnitMerge);
  // more than half of an SM's shared memory: one CTA per SM, so the TMEM
  // allocation never waits for another CTA
  static_assert(SMEM_BYTES > 116 * 1024 && SMEM_BYTES <= 227 * 1024, "one resident CTA per SM");
};

struct TcBars {
  uint32_t b0;
  __device__ __forceinline__ uint32_t s_full(int i) const { return b0 + 8 * i; }
  __device__ __forceinline__ uint32_t s_free(int i) const { return b0 + 16 + 8 * i; }
  __device__ __forceinline__ uint32_t p_full(int i) const { return b0 + 32 + 8 * i; }
  __device__ __forceinline__ uint32_t pv_done(int i) const { return b0 + 48 + 8 * i; }
  __device__ __forceinline__ uint32_t o_free(int i) const { return b0 + 64 + 8 * i; }
  __device__ __forceinline__ uint32_t q_full(int i) const { return b0 + 80 + 8 * i; }
  __device__ __forceinline__ uint32_t mma_done() const { return b0 + 96; }
  __device__ __forceinline__ uint32_t conv_full(int i) const { return b0 + 104 + 8 * i; }
  __device__ __forceinline__ uint32_t stg_free(int i) const { return b0 + 120 + 8 * i; }
};

// All lanes of a warp wait; a wait that timed out in any lane counts as
// timed out in all of them, so that the warp stays converged for the
// warp-collective tcgen05 loads and stores.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

// Named barrier 2 + j over the 128 threads of softmax group j; the second
// form ORs a flag.
__device__ __forceinline__ void soft_bar(int grp) { asm volatile("bar.sync %0, 128;" ::"r"(2 + grp) : "memory"); }
__device__ __forceinline__ bool soft_bar_or(int grp, bool v) {
  uint32_t res;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(res)
      : "r"((uint32_t)v), "r"(2 + grp)
      : "memory");
  return res != 0;
}

// Reduces v[h] (h < NR) across the 32 lanes of a warp (a butterfly that
// halves the values kept per lane at each step while more than one is left,
// then combines single values).  Afterwards lane L holds the result for head
// j + K*(L >> SHIFT) in v[j], j < K = max(1, NR/32).
template <int NR>
struct TransposeReduce {
  static constexpr int K = NR > 32 ? NR / 32 : 1;
  static constexpr int HALVINGS = NR >= 32 ? 5 : (NR == 16 ? 4 : 3);
  static constexpr int SHIFT = 5 - HALVINGS;
};

template <int NR, bool MAX>
__device__ __forceinline__ void warp_transpose_reduce(float (&v)[NR], int lane) {
#pragma unroll
  for (int s = 0; s < 5; ++s) {
    const int o = 16 >> s, n = NR >> s;
    if (n > TransposeReduce<NR>::K) {
      const bool upper = (lane & o) != 0;
#pragma unroll
      for (int j = 0; j < n / 2; ++j) {
        const float give = upper ? v[j] : v[j + n / 2];
        const float keep = upper ? v[j + n / 2] : v[j];
        const float got = __shfl_xor_sync(0xffffffffu, give, o);
        v[j] = MAX ? fmaxf(keep, got) : keep + got;
      }
    } else {
#pragma unroll
      for (int j = 0; j < TransposeReduce<NR>::K; ++j) {
        const float got = __shfl_xor_sync(0xffffffffu, v[j], o);
        v[j] = MAX ? fmaxf(v[j], got) : v[j] + got;
      }
    }
  }
}

// Per-head reduction of v (group grp's HG heads) over the group's 128
// threads (v is clobbered); afterwards every thread of the group can read
// the result of its head h from fin[grp*HG + h].  `red` holds [SG][4][HG].
template <class C, bool MAX>
__device__ __forceinline__ void soft_reduce(float (&v)[C::HG], int grp, int sub, int lane, float *red, float *fin,
                                            int R) {
  using TR = TransposeReduce<C::HG>;
  constexpr int HG = C::HG;
  warp_transpose_reduce<HG, MAX>(v, lane);
  float *rg = red + grp * 4 * HG;
#pragma unroll
  for (int j = 0; j < TR::K; ++j) rg[sub * HG + j + TR::K * (lane >> TR::SHIFT)] = v[j];
  soft_bar(grp);
  if (R < HG) {
    const float a = rg[R], b2 = rg[HG + R], c = rg[2 * HG + R], d = rg[3 * HG + R];
    fin[grp * HG + R] = MAX ? fmaxf(fmaxf(a, b2), fmaxf(c, d)) : (a + b2) + (c + d);
  }
  soft_bar(grp);
}

// Per-head maximum of v (group grp's HG heads) over the group's 128 threads:
// one warp-wide redux per head (every lane gets its warp's maximum), lane 0
// of each warp stores its warp's HG maxima, and thread R < HG combines the
// four warps'; afterwards every thread of the group can read the maximum of
// its head h from fin[grp*HG + h].  Exact (a maximum does not depend on the
// order); NaN inputs are ignored as by fmaxf.  With m_first (a unit's first
// tile) thread R also sets the running max of its head, m_first[grp*HG + R],
// to that maximum, or keeps `floor` when the maximum does not exceed it by
// more than 8, before the same final barrier.
template <class C>
__device__ __forceinline__ void soft_reduce_max(float (&v)[C::HG], int grp, int sub, int lane, float *red, float *fin,
                                                int R, float *m_first = nullptr, float floor = 0.f) {
  constexpr int HG = C::HG;
#pragma unroll
  for (int h = 0; h < HG; ++h) asm volatile("redux.sync.max.f32 %0, %0, 0xffffffff;" : "+f"(v[h]));
  float *rg = red + grp * 4 * HG;
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < HG; h += 4)
      *reinterpret_cast<float4 *>(rg + sub * HG + h) = make_float4(v[h], v[h + 1], v[h + 2], v[h + 3]);
  }
  soft_bar(grp);
  if (R < HG) {
    const float t = fmaxf(fmaxf(rg[R], rg[HG + R]), fmaxf(rg[2 * HG + R], rg[3 * HG + R]));
    fin[grp * HG + R] = t;
    if (m_first) m_first[grp * HG + R] = t > floor + 8.f ? t : floor;
  }
  soft_bar(grp);
}

// 4x4 transpose across the four lanes of each quad (lanes 4k..4k+3): lane j
// of a quad holds v[i] = M[j][i] before and v[i] = M[i][j] after (two
// butterfly stages, each swapping one pair of values with the partner lane).
__device__ __forceinline__ void quad_transpose(float (&v)[4], int lane) {
  const bool b0 = (lane & 1) != 0, b1 = (lane & 2) != 0;
  float r;
  r = __shfl_xor_sync(0xffffffffu, b0 ? v[0] : v[1], 1);
  v[0] = b0 ? r : v[0];
  v[1] = b0 ? v[1] : r;
  r = __shfl_xor_sync(0xffffffffu, b0 ? v[2] : v[3], 1);
  v[2] = b0 ? r : v[2];
  v[3] = b0 ? v[3] : r;
  r = __shfl_xor_sync(0xffffffffu, b1 ? v[0] : v[2], 2);
  v[0] = b1 ? r : v[0];
  v[2] = b1 ? v[2] : r;
  r = __shfl_xor_sync(0xffffffffu, b1 ? v[1] : v[3], 2);
  v[1] = b1 ? r : v[1];
  v[3] = b1 ? v[3] : r;
}

// Merge of the unit whose k pieces the k CTAs of this cluster (ranks 0..k-1,
// CTAs c0 .. c0+k-1) left in workspace slots 2*(c0+j) (none for an empty
// piece): this CTA writes heads [r*hpr, min(nh, (r+1)*hpr)), hpr =
// ceil(nh / k), r its rank,
//   out = sum_j 2^(m_j - M) O_j / sum_j 2^(m_j - M) l_j,  M = max_j m_j,
// over the non-empty pieces j = 0 .. k-1 in order.  A thread takes 16
// dimensions of one head and issues all of its loads before it uses any.
template <class C, bool MULTI>
__device__ __forceinline__ void merge_cluster_unit(const SplitParams &p, const CtaRange &range, int tid, int nthr) {
  constexpr int D = C::D, KMAX = 4, SEG = 16;  // at most 4 CTAs per cluster (host)
  const int k = p.cluster_k;
  const int r = (int)cluster_rank();
  const int c0 = (int)blockIdx.x - r;
  // the unit, from the range (a CTA with an empty piece has no segment);
  // piece j is empty when it starts where piece j + 1 does
  const int tiles = range.tiles_b;
  const long long uoff = range.begin - range.pre_b;
  const int uib = uoff < 0x7fffffffLL ? (int)uoff / tiles : (int)(uoff / tiles);
  bool has[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) has[j] = j < k && piece_start(j + 1, tiles, k) > piece_start(j, tiles, k);
  const int b = range.b, g = uib / p.head_chunks, hc = uib % p.head_chunks;
  const int h_first = g * p.n_rep + hc * p.heads_per_cta;
  const int nh = min(p.heads_per_cta, p.n_rep - hc * p.heads_per_cta);
  const int hpr = (nh + k - 1) / k;
  const int h_lo = r * hpr, h_hi = min(nh, h_lo + hpr);
  const float2 *ml = reinterpret_cast<const float2 *>(p.ml_part);
  for (int it = tid; it < (h_hi - h_lo) * (D / SEG); it += nthr) {
    const int h = h_lo + it / (D / SEG), d0 = (it % (D / SEG)) * SEG;
    float2 mlj[KMAX];
    float4 oj[KMAX][SEG / 4];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (has[j]) {
        if (!GQA_SLOT_OK(p, 2 * (c0 + j), h)) continue;
        const size_t ps = (size_t)2 * (c0 + j) * p.heads_per_cta + h;
        mlj[j] = __ldcg(ml + ps);
        const float4 *o = reinterpret_cast<const float4 *>(p.o_part + ps * D + d0);
#pragma unroll
        for (int q = 0; q < SEG / 4; ++q) oj[j][q] = __ldcg(o + q);
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (!has[j]) mlj[j] = make_float2(-INFINITY, 0.f);
      M = fmaxf(M, mlj[j].x);
    }
    float L = 0.f, a[SEG];
#pragma unroll
    for (int e = 0; e < SEG; ++e) a[e] = 0.f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (has[j]) {
        const float w = merge_weight(mlj[j].x, M);
        L += w * mlj[j].y;
#pragma unroll
        for (int q = 0; q < SEG / 4; ++q) {
          a[4 * q + 0] += w * oj[j][q].x;
          a[4 * q + 1] += w * oj[j][q].y;
          a[4 * q + 2] += w * oj[j][q].z;
          a[4 * q + 3] += w * oj[j][q].w;
        }
      }
    }
    const float inv = (!MULTI || L > 0.f) ? 1.f / L : 0.f;  // 0: a query row that sees no position
    uint4 pk[2];
    uint32_t *pw = reinterpret_cast<uint32_t *>(pk);
#pragma unroll
    for (int e = 0; e < SEG / 2; ++e) pw[e] = pack_bf16x2(a[2 * e] * inv, a[2 * e + 1] * inv);
    const size_t orow = query_row<MULTI>(p, b, h_first + h);
    if (!GQA_ROW_OK(p, orow)) continue;
    uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(p.out) + orow * D + d0);
    dst[0] = pk[0];
    dst[1] = pk[1];
  }
}

// Floor of the running max (log2 units): far below any logit, finite so
// that 2^(x - floor) is 0 for x = -inf.  A partial left with it (a row with
// no visible position in its segment) gets weight 0 in the merge unless every
// partial of the row has it, and a row whose sum stays 0 is written as 0.
constexpr float kNoMax = -1e30f;

// STEP: the instantiation for the fused decode step, whose CTAs count on the
// step word as soon as no thread will read the lengths again (the others,
// compiled without that code, count after all of their work when asked to).
template <class C, bool MULTI, bool STEP = false>
__global__ void __launch_bounds__(C::THREADS, 1)
    gqa_split_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                        const __grid_constant__ CUtensorMap tmK16, const __grid_constant__ CUtensorMap tmV16,
                        const SplitParams p) {
  using Pipe = typename C::Pipe;
  constexpr int D = C::D, BN = C::BLOCK_N, ST = C::STAGES, NR = C::NR, HG = C::HG;
  constexpr int HCH = HG < 32 ? HG : 32;  // TMEM columns per tcgen05.ld of the softmax
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  Pipe pipe;
  pipe.base = smem_u32(smem);
  pipe.full0 = pipe.base + C::BAR_OFF;
  pipe.empty0 = pipe.full0 + 8 * ST;
  TcBars bars{pipe.empty0 + 8 * ST};
  const uint32_t qbase = pipe.base + C::Q_OFF;
  const uint32_t pbase = pipe.base + C::P_OFF;
  float *red = reinterpret_cast<float *>(smem + C::RED_OFF);
  float *fin = reinterpret_cast<float *>(smem + C::FIN_OFF);
  float *m_s = reinterpret_cast<float *>(smem + C::M_OFF);
  float *corr_s = reinterpret_cast<float *>(smem + C::CORR_OFF);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::TMEM_SLOT_OFF);
  CtaRange *range_smem = reinterpret_cast<CtaRange *>(smem + C::RANGE_OFF);
  UnitMerge *um = reinterpret_cast<UnitMerge *>(smem + C::MERGE_OFF);
  SchedParams sp;
  sp.seq_lens = p.seq_lens;
  sp.B = p.B;
  sp.Nmax = p.Nmax;
  sp.units_per_b = p.G * p.head_chunks;
  sp.block_n = BN;
  sp.append = p.append;
  sp.unit_cost = C::UNIT_COST;
  sp.cluster_k = p.cluster_k;

  if (threadIdx.x == 0) {
    pipe.init();
    for (int i = 0; i < 2; ++i) {
      mbar_init(bars.s_full(i), 1);
      mbar_init(bars.s_free(i), 4 * C::SG);  // one arrival per softmax warp
      mbar_init(bars.o_free(i), 4 * C::SG);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bars.p_full(i), 4 * C::SG);
      mbar_init(bars.pv_done(i), 1);
    }
    mbar_init(bars.q_full(0), 4);  // one arrival per warp of softmax group 0
    mbar_init(bars.q_full(1), 4);
    mbar_init(bars.mma_done(), 2);  // the commits of both MMA issuers
    if (C::CONV) {
      for (int i = 0; i < 2; ++i) mbar_init(bars.conv_full(i), 4);  // one arrival per converter warp
      for (int i = 0; i < C::VSTG; ++i) mbar_init(bars.stg_free(i), 1);  // the MMA commit after the tile's P.V
    }
    fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(smem_u32(tmem_slot), C::TM_COLS);
    tc::tmem_relinquish();
  }
  int2 spec_lens = make_int2(-1, -1);  // warp 0: the lengths the speculative plan read
  if (warp == 0) {
    // Ahead of the wait for earlier kernels: fetch the tensor maps and ask
    // L2 for the first tiles of a speculative plan (a hint only).
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmK16);
      tma_prefetch_desc(&tmV16);
    }
    SchedParams spx = sp;
    spx.spec = 1;
    const CtaRange r0 = warp_plan_range<true>(spx, lane, nullptr, 0, &spec_lens);
    // kept in shared memory, not registers, across the wait
    if (lane == 0) *range_smem = r0;
    if (lane == 0 && r0.begin < r0.end) prefetch_first_tiles(spx, r0, &tmK, &tmV, C::FP8 ? 128 : 64, C::FP8 ? 1 : 2, p.G, p.head_chunks, ST);
    if (!MULTI && r0.begin < r0.end) {
      // and for the query rows of the first unit (a hint too: the copy
      // after the wait still reads global memory)
      SegmentCursor c0;
      c0.init(spx, r0);
      Segment s0;
      if (c0.next(spx, s0)) {
        const int g = s0.uib / p.head_chunks, hc = s0.uib % p.head_chunks;
        const int hf = g * p.n_rep + hc * p.heads_per_cta;
        const int nh = min(p.heads_per_cta, p.n_rep - hc * p.heads_per_cta);
        const char *qb = reinterpret_cast<const char *>(p.q) + ((size_t)s0.b * p.H + hf) * D * 2;
        for (int ln = lane; ln < nh * D * 2 / 128; ln += 32)
          asm volatile("prefetch.global.L2 [%0];" ::"l"(qb + (size_t)ln * 128));
      }
    }
  }
  griddep_wait();  // lengths, q and cache rows written by earlier kernels are visible
  if (warp == 0) {
    if (!spec_plan_holds(sp, lane, spec_lens)) {
      const CtaRange r = warp_plan_range(sp, lane, p.out, (size_t)p.H * D * sizeof(__nv_bfloat16));
      if (lane == 0) *range_smem = r;
    }
  }
  if (STEP && threadIdx.x == 0) um->reads_done = 0;
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  griddep_launch_dependents();
  const CtaRange range = *range_smem;
  const uint32_t tmem = *tmem_slot;

  if (range.begin < range.end) {
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      // (a unit's last tile, when short, through the 16-position boxes)
      produce_range(pipe, sp, range, &tmK, &tmV, C::FP8 ? 128 : 64, p.G, p.head_chunks, p, lane, &tmK16, &tmV16);
    } else if (warp == 1 || warp == 2) {
      // ------------------------------------------------------------ MMA issuers
      // Two threads issue the MMAs, each walking the CTA's tiles on its own:
      // lane 0 of warp 1 the S^T of every tile (once its K tile is ready, its
      // S buffer free and, on a unit's first tile, the unit's Q in place),
      // lane 0 of warp 2 the P.V (once its P^T is written and, on a unit's
      // first tile, its O buffer free).  Issuing a tile's eight MMAs takes
      // a few hundred nanoseconds; with one thread for both chains the S^T of
      // the next tile waited behind the P.V of the previous one.  The chains
      // meet only through the softmax (S -> P), and each commits its own
      // MMAs to its barriers.
      if (lane == 0) {
        // FP8 cache: all operands are f16 (exact for the E4M3 values)
        constexpr uint32_t IDESC_S = C::F8N   ? tc::idesc_e4m3_f32(BN, C::NM, false, false)
                                     : C::FP8 ? tc::idesc_f16_f32(BN, NR, false, false)
                                              : tc::idesc_bf16_f32(BN, NR, false, false);
        constexpr uint32_t IDESC_PV = C::F8N   ? tc::idesc_e4m3_f32(D, C::NM, true, true)
                                      : C::FP8 ? tc::idesc_f16_f32(D, NR, true, true)
                                               : tc::idesc_bf16_f32(D, NR, true, true);
        SegmentCursor cur;
        cur.init(sp, range);
        Segment seg;
        int tg = 0;
        bool ok = true;
        bool lens_read = !STEP || !p.append;
        for (int unit = 0; ok && cur.next(sp, seg); ++unit) {
          if (STEP && !lens_read && cur.end - cur.pos <= cur.cost) {  // the last segment: no more reads
            signal_lengths_read_thread(um);
            lens_read = true;
          }
          for (int i = 0; ok && i < seg.t1 - seg.t0; ++i, ++tg) {
            if (warp == 1) {
              const int st = tg % ST;
              // unit u's Q is in buffer u % QB, its (u / QB)-th use
              const int qb = unit % C::QB;
              ok = (i != 0 || mbar_wait(bars.q_full(qb), (unit / C::QB) & 1)) &&
                   (C::CONV ? mbar_wait(bars.conv_full(tg & 1), (tg >> 1) & 1)
                           : mbar_wait(pipe.full(st), (tg / ST) & 1)) &&
                   (tg < 2 || mbar_wait(bars.s_free(tg & 1), ((tg >> 1) - 1) & 1));
              if (!ok) break;
              tc::fence_after();
              // descriptors of the tile's first K step; the others are
              // constant offsets from them (one add each)
              const uint64_t b0 = tc::smem_desc_sw128(qbase + qb * C::Q_BYTES, 16, 1024);
              const uint64_t a0 = C::CONV ? 0 : tc::smem_desc_sw128(pipe.k_tile(st), 16, 1024);
              const uint32_t dS = tmem + C::TM_S + (tg & 1) * C::NM;
              if constexpr (C::F8N) {
                // E4M3 K tile (one 128-byte row of codes per position) times
                // the two-term E4M3 Q: 32 K elements (32 bytes) per step
#pragma unroll
                for (int ks = 0; ks < D / 32; ++ks)
                  tc::mma_ss_f8(dS, tc::desc_add(a0, ks * 32), tc::desc_add(b0, ks * 32), IDESC_S, ks > 0);
              }
#pragma unroll
              for (int ks = 0; ks < (C::F8N ? 0 : D / 16); ++ks) {
                const uint64_t b = tc::desc_add(b0, (ks >> 2) * C::Q_BOX + (ks & 3) * 32);
                if constexpr (C::CONV) {
                  // A = the f16 K tile in tensor memory: 16 K elements = 8 columns
                  tc::mma_ts(dS, tmem + C::TM_K + (tg & 1) * 64 + ks * 8, b, IDESC_S, ks > 0);
                } else {
                  tc::mma_ss(dS, tc::desc_add(a0, (ks >> 2) * C::KV_BOX + (ks & 3) * 32), b, IDESC_S, ks > 0);
                }
              }
              tc::commit(bars.s_full(tg & 1));
            } else {
              const int ob = unit & 1, pb = tg % C::PB, use = tg / C::PB;
              ok = mbar_wait(bars.p_full(pb), use & 1) &&
                   (i != 0 || unit < 2 || mbar_wait(bars.o_free(ob), ((unit >> 1) - 1) & 1));
              if (!ok) break;
              tc::fence_after();
              const uint32_t vt =
                  C::CONV ? pipe.base + C::STG_OFF + (tg % C::VSTG) * C::STG_TILE : pipe.v_tile(tg % ST);
              const uint64_t a0 = tc::smem_desc_sw128(vt, C::KV_BOX, 1024);
              const uint64_t b0 = tc::smem_desc_mn_rows(pbase + pb * C::P_BYTES, C::P_ROW);
              const uint32_t dO = tmem + C::TM_O + ob * C::NM;
              if constexpr (C::F8N) {
                // E4M3 V tile, MN-major (128 d codes per position row): 32
                // positions (32 rows of 128 bytes) per step
#pragma unroll
                for (int ks = 0; ks < BN / 32; ++ks)
                  tc::mma_ss_f8(dO, tc::desc_add(a0, ks * 4096), tc::desc_add(b0, ks * 32 * C::P_ROW), IDESC_PV,
                                i > 0 || ks > 0);
              } else {
#pragma unroll
                for (int ks = 0; ks < BN / 16; ++ks)
                  tc::mma_ss(dO, tc::desc_add(a0, ks * 2048), tc::desc_add(b0, ks * 16 * C::P_ROW), IDESC_PV,
                             i > 0 || ks > 0);
              }
              // the tile's K and V are no longer read: free its ring stage
              // (FP8 with converters: its staging buffer; the converters free
              // the stage)
              tc::commit(C::CONV ? bars.stg_free(tg % C::VSTG) : pipe.empty(tg % ST));
              tc::commit(bars.pv_done(pb));
            }
          }
        }
        if (STEP && !lens_read) signal_lengths_read_thread(um);
        // nothing of either thread's may still run when TMEM is freed (the
        // barrier counts both threads' commits)
        tc::commit(bars.mma_done());
        mbar_wait(bars.mma_done(), 0);
      }
      __syncwarp();
    } else if (warp < C::CONV_WARP0) {  // (warp >= SOFT_WARP0)
      // ------------------------------------------------------------ softmax
      const int sub = warp & 3;       // TMEM lane quarter of this warp
      const int R = 32 * sub + lane;  // TMEM lane: tile position (S^T) / output dim (O^T)
      const int grp = C::SG == 1 ? 0 : (warp - C::SOFT_WARP0) >> 2;  // softmax group: head columns [hg0, hg0 + HG)
      const int hg0 = grp * HG;
      const uint32_t trow = tmem + ((uint32_t)(32 * sub) << 16);
      // the logits' scale-and-shift and the row sums two heads per
      // instruction (packed fp32 FMA / add): measured faster with 64 heads
      // (sweep G=1 19.95 -> 19.78 us) and with E4M3 operands (GQA-8 32.37 ->
      // 31.78 us), slower with 32 bf16 heads (MQA 15.00 -> 15.15 us)
      constexpr bool PACK = C::F8N || HG == 64;
      SegmentCursor cur;
      cur.init(sp, range);
      Segment seg;
      bool have = cur.next(sp, seg);
      auto unit_heads = [&](const Segment &s, int &h_first, int &nh) {
        const int g = s.uib / p.head_chunks, hc = s.uib % p.head_chunks;
        h_first = g * p.n_rep + hc * p.heads_per_cta;
        nh = min(p.heads_per_cta, p.n_rep - hc * p.heads_per_cta);
      };
      // Q rows of a unit go to buffer u % QB: thread R copies the 128-byte
      // half R & 1 of row R >> 1 (zeros for padding rows) with cp.async, so
      // the copy runs while the thread works on.  With two buffers unit
      // u + 2's copy is issued at the end of unit u and completed (wait,
      // proxy fence, arrival on q_full) at the end of unit u + 1, a whole
      // unit later; with one buffer it is issued and completed at the end of
      // the previous unit.
      auto issue_q = [&](const Segment &s, int buf) {
        int h_first, nh;
        unit_heads(s, h_first, nh);
        const int row = R >> 1, half = R & 1;
        const size_t qrow = query_row<MULTI>(p, s.b, h_first + min(row, nh - 1));
        if (row < NR && GQA_ROW_OK(p, qrow)) {
          const uint4 *src = reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(p.q) +
                                                             qrow * D + half * 64);
          const uint32_t dst = qbase + buf * C::Q_BYTES + C::Q_STG + half * C::Q_BOX + row * 128;
          const uint32_t bytes = row < nh ? 16u : 0u;
#pragma unroll
          for (int c = 0; c < 8; ++c) cp_async_16(dst + ((c ^ (row & 7)) << 4), src + c, bytes);
        }
        cp_async_commit();
      };
      // `later`: another unit's copy was issued after this one
      auto complete_q = [&](int buf, bool later) {
        if (later)
          cp_async_wait<1>();
        else
          cp_async_wait<0>();
        if constexpr (C::F8N) {
          // (the rows were copied by other threads of the group: every copy
          // of this buffer has landed once all of them passed their wait)
          soft_bar(0);
          // E4M3 operand: eight threads per row (R & 7 = part: d 16*part ..
          // 16*part + 15, chunks 2*(part & 3) and + 1 of box part >> 2 of the
          // copied bf16 row); the row's eight lanes agree on its scale qs (a
          // power of two: max |Q[h]| * qs in [128, 256)), then each writes
          // its 16 codes of term 0 (operand row h) and of term 1 (row NR + h)
          const int part = R & 7;
#pragma unroll
          for (int it = 0; it < NR / 16; ++it) {
            const int row = 16 * it + (R >> 3);
            const uint32_t src = qbase + buf * C::Q_BYTES + C::Q_STG + (part >> 2) * C::Q_BOX + row * 128;
            uint4 v[2];
            float mx = 0.f;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const int c = 2 * (part & 3) + j;
              v[j] = lds128(src + ((c ^ (row & 7)) << 4));
              const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
              for (int i = 0; i < 4; ++i) mx = fmaxf(mx, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
            }
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            // qs = 2^(7 - floor(log2 mx)), from the exponent field (clamped
            // to the normal range; 1 for an all-zero row)
            const int e = (int)((__float_as_uint(mx) >> 23) & 0xffu) - 127;
            const int f = mx > 0.f ? min(254, max(1, 127 + 7 - e)) : 127;
            const float qs = __uint_as_float((uint32_t)f << 23);
            if (part == 0) reinterpret_cast<float *>(smem + C::QSC_OFF)[buf * C::NQ + row] = 1.f / qs;
            uint32_t t0[4], t1[4];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
              for (int i = 0; i < 4; i += 2) {
                const float x0 = bf16_lo(w[i]) * qs, x1 = bf16_hi(w[i]) * qs;
                const float x2 = bf16_lo(w[i + 1]) * qs, x3 = bf16_hi(w[i + 1]) * qs;
                const uint32_t a = float2_to_e4m3x2(x0, x1), b = float2_to_e4m3x2(x2, x3);
                float a0, a1, b0, b1;
                e4m3x2_to_float(a, a0, a1);
                e4m3x2_to_float(b, b0, b1);
                const uint32_t la = float2_to_e4m3x2((x0 - a0) * 16.f, (x1 - a1) * 16.f);
                const uint32_t lb = float2_to_e4m3x2((x2 - b0) * 16.f, (x3 - b1) * 16.f);
                t0[2 * j + i / 2] = a | (b << 16);
                t1[2 * j + i / 2] = la | (lb << 16);
              }
            }
            const uint32_t op = qbase + buf * C::Q_BYTES;
            const int r0 = row, r1 = NR + row;
            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(op + r0 * 128 + ((part ^ (r0 & 7)) << 4)),
                         "r"(t0[0]), "r"(t0[1]), "r"(t0[2]), "r"(t0[3])
                         : "memory");
            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(op + r1 * 128 + ((part ^ (r1 & 7)) << 4)),
                         "r"(t1[0]), "r"(t1[1]), "r"(t1[2]), "r"(t1[3])
                         : "memory");
          }
        } else if constexpr (C::FP8) {
          // f16 operands: this thread's bf16 chunks become f16 in place
          const int row = R >> 1, half = R & 1;
          if (row < NR) {
            const uint32_t dst = qbase + buf * C::Q_BYTES + half * C::Q_BOX + row * 128;
            bool big = false;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint32_t a = dst + ((c ^ (row & 7)) << 4);
              const uint4 v = lds128(a);
              const uint32_t w[4] = {v.x, v.y, v.z, v.w};
              uint32_t o[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float lo = bf16_lo(w[i]), hi = bf16_hi(w[i]);
                big |= fabsf(lo) > 65504.f || fabsf(hi) > 65504.f;
                o[i] = pack_f16x2(lo, hi);
              }
              asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(o[0]), "r"(o[1]), "r"(o[2]),
                           "r"(o[3])
                           : "memory");
            }
            if (big) flag_error(GQA_DEVERR_RANGE);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.q_full(buf));
      };
      // softmax group 0 alone loads Q
      if (have && grp == 0) {
        issue_q(seg, 0);
        SegmentCursor la = cur;
        Segment s1;
        const bool has1 = C::QB == 2 && la.next(sp, s1);
        if (has1) issue_q(s1, 1);
        complete_q(0, has1);
      }
      // After a wait that timed out the thread is "dead": its later waits
      // return at once, but it keeps the same control flow, so the four
      // warps of its softmax group still meet at every named barrier and
      // finish (the error word already holds GQA_DEVERR_TIMEOUT).
      bool dead = false;
      auto wait = [&](uint32_t bar, uint32_t parity) {
        if (!dead && !warp_wait(bar, parity)) dead = true;
      };
      int t = 0;
      bool lens_read = !STEP || !p.append;
      for (int unit = 0; have; ++unit) {
        int h_first, nh;
        unit_heads(seg, h_first, nh);
        const int b = seg.b;
        const int L = attn_len(p.seq_lens, b, p.Nmax, p.append);
        if (STEP && !lens_read && cur.end - cur.pos <= cur.cost) {
          // the last unit: the cursor reads no more lengths (nor do the Q
          // look-aheads, which stand at or past it)
          signal_lengths_read(um, lane);
          lens_read = true;
        }
        const int ob = unit & 1;
        const int ntl = seg.t1 - seg.t0;
        // FP8 cache: K's per-head scale joins the logit scale, V's the result
        const int g_unit = seg.uib / p.head_chunks;
        const float sl2 = C::FP8 ? p.scale_log2 * __ldg(p.k_scale + g_unit) : p.scale_log2;
        const float vscale = C::FP8 ? __ldg(p.v_scale + g_unit) : 1.f;
        float lp[HG];
#pragma unroll
        for (int h = 0; h < HG; ++h) lp[h] = 0.f;
        // The running max starts at a finite floor rather than -inf, so that
        // a row that has seen no visible position yet (a query token whose
        // whole view lies in later tiles) gets 2^(-inf - floor) = 0, not NaN.
        // Padding rows (zero queries, so zero logits) are computed like real
        // ones and never written out.
        if (R < HG) m_s[hg0 + R] = kNoMax;
        // F8N: head h's logit factor, the logit scale over the head's Q scale
        // (this unit's Q buffer was completed by this group before the unit)
        float *cf_s = reinterpret_cast<float *>(smem + C::QSC_OFF) + 2 * C::NQ;
        if (C::F8N && R < HG)
          cf_s[hg0 + R] = sl2 * reinterpret_cast<const float *>(smem + C::QSC_OFF)[(unit % C::QB) * C::NQ + hg0 + R];
        soft_bar(grp);
        // Row h of the unit is query token t(h) = (row0 + h) / rep_kv of its
        // run and sees positions n < L_all + t(h); positions below L_all are
        // visible to every row.
        const int L_all = L - (p.tokens - 1);
        const int row0 = h_first % p.n_rep + hg0;  // the group's first row
        const int t_first = row0 / p.rep_kv, k_first = row0 % p.rep_kv;
        const float4 *m4 = reinterpret_cast<const float4 *>(m_s + hg0);
        for (int i = 0; i < ntl; ++i) {
          const int tg = t + i, sb = tg & 1, st = tg % ST;
          const bool valid = (seg.t0 + i) * BN + R < L;
          // a tile that reaches L_all needs the per-row limits of a run of
          // several tokens; before it every position is visible to every row
          const bool edge = (seg.t0 + i + 1) * BN > L_all;
          const int pos = (seg.t0 + i) * BN + R;
          // -inf where the row may not see this position: past L (the cache
          // row may hold NaN), or a later token of the row's own run
          auto mask = [&](float(&v)[HG]) {
            if (__any_sync(0xffffffffu, !valid)) {
#pragma unroll
              for (int h = 0; h < HG; ++h) v[h] = valid ? v[h] : -INFINITY;
            }
            if (MULTI && edge) {
              int tk = t_first, kk = k_first;
#pragma unroll
              for (int h = 0; h < HG; ++h) {
                if (pos >= L_all + tk) v[h] = -INFINITY;
                const bool wrap = ++kk == p.rep_kv;
                kk = wrap ? 0 : kk;
                tk += wrap ? 1 : 0;
              }
            }
          };
          // this position's raw logits S of the group's heads (every column
          // chunk asked for before the one wait); F8N: the two Q terms'
          // columns, combined (term 0 + term 1 / 16; the head's Q scale is in
          // its logit factor)
          auto load_s = [&](float(&x)[HG]) {
            uint32_t r[HG];
#pragma unroll
            for (int c0 = 0; c0 < HG; c0 += HCH) {
              if constexpr (HCH == 32) {
                tc::ld_32x32b_x32(trow + C::TM_S + sb * C::NM + hg0 + c0, r + c0);
              } else {
                tc::ld_32x32b_x16(trow + C::TM_S + sb * C::NM + hg0 + c0, r + c0);
              }
            }
            if constexpr (C::F8N) {
              uint32_t r1[HG];
#pragma unroll
              for (int c0 = 0; c0 < HG; c0 += HCH) {
                if constexpr (HCH == 32) {
                  tc::ld_32x32b_x32(trow + C::TM_S + sb * C::NM + NR + hg0 + c0, r1 + c0);
                } else {
                  tc::ld_32x32b_x16(trow + C::TM_S + sb * C::NM + NR + hg0 + c0, r1 + c0);
                }
              }
              tc::wait_ld();
#pragma unroll
              for (int h = 0; h < HG; ++h) x[h] = fmaf(__uint_as_float(r1[h]), 0.0625f, __uint_as_float(r[h]));
            } else {
              tc::wait_ld();
#pragma unroll
              for (int h = 0; h < HG; ++h) x[h] = __uint_as_float(r[h]);
            }
          };
          const float4 *cf4 = reinterpret_cast<const float4 *>(cf_s + hg0);
          // y = S * scale_log2 - m (F8N: S * factor[h] - m), masked
          auto compute_y = [&](float(&y)[HG]) {
            float x[HG];
            load_s(x);
#pragma unroll
            for (int h4 = 0; h4 < HG; h4 += 4) {
              const float4 mm = m4[h4 >> 2];
              const float4 cf = C::F8N ? cf4[h4 >> 2] : make_float4(sl2, sl2, sl2, sl2);
              if constexpr (PACK) {
                const float2 y01 = __ffma2_rn(make_float2(x[h4 + 0], x[h4 + 1]), make_float2(cf.x, cf.y),
                                              make_float2(-mm.x, -mm.y));
                const float2 y23 = __ffma2_rn(make_float2(x[h4 + 2], x[h4 + 3]), make_float2(cf.z, cf.w),
                                              make_float2(-mm.z, -mm.w));
                y[h4 + 0] = y01.x;
                y[h4 + 1] = y01.y;
                y[h4 + 2] = y23.x;
                y[h4 + 3] = y23.y;
              } else {
                y[h4 + 0] = fmaf(x[h4 + 0], cf.x, -mm.x);
                y[h4 + 1] = fmaf(x[h4 + 1], cf.y, -mm.y);
                y[h4 + 2] = fmaf(x[h4 + 2], cf.z, -mm.z);
                y[h4 + 3] = fmaf(x[h4 + 3], cf.w, -mm.w);
              }
            }
            mask(y);
          };
          wait(bars.s_full(sb), (tg >> 1) & 1);
          tc::fence_after();
          float y[HG];
          // Lazy running max: it starts at a unit's first tile's maximum and
          // then moves only where a logit beats it by more than 8 (log2
          // units).  On the first tile one read of S serves both the maximum
          // and y, and there is neither a vote nor a rescale.  Measured, this
          // pays on the bf16 groups of 32 heads (sweep G=2 26.5 -> 26.2 us,
          // MQA 15.7 -> 15.2 us) but costs the 16-head and E4M3 kernels
          // (their larger code slows the steady tile: FP8 GQA-8 32.0 -> 32.9
          // us) and gains nothing with 64 heads, which keep the general path.
          constexpr bool FIRST_FAST = !C::FP8 && HG == 32;
          bool rare;
          if constexpr (FIRST_FAST) {
            if (i == 0) {
              float x[HG];
              load_s(x);
#pragma unroll
              for (int h = 0; h < HG; ++h) x[h] *= sl2;
              mask(x);
#pragma unroll
              for (int h = 0; h < HG; ++h) y[h] = x[h];
              soft_reduce_max<C>(x, grp, sub, lane, red, fin, R, m_s, kNoMax);
#pragma unroll
              for (int h4 = 0; h4 < HG; h4 += 4) {
                const float4 mm = m4[h4 >> 2];
                y[h4 + 0] -= mm.x;
                y[h4 + 1] -= mm.y;
                y[h4 + 2] -= mm.z;
                y[h4 + 3] -= mm.w;
              }
              rare = false;
            } else {
              compute_y(y);
              float ymax = y[0];
#pragma unroll
              for (int h = 1; h < HG; ++h) ymax = fmaxf(ymax, y[h]);
              rare = soft_bar_or(grp, ymax > 8.f);
            }
          } else {
            compute_y(y);
            float ymax = y[0];
#pragma unroll
            for (int h = 1; h < HG; ++h) ymax = fmaxf(ymax, y[h]);
            rare = soft_bar_or(grp, i == 0 || ymax > 8.f);
          }
          if (rare) {
            {
              float x[HG];
              load_s(x);
#pragma unroll
              for (int h = 0; h < HG; ++h) x[h] *= C::F8N ? cf_s[hg0 + h] : sl2;
              mask(x);
              soft_reduce_max<C>(x, grp, sub, lane, red, fin, R);
            }
            bool moved_mine = false;
            if (R < HG) {
              const float tmax = fin[hg0 + R], mo = m_s[hg0 + R];
              float corr = 1.f;
              if (tmax > mo + 8.f) {
                const float mn = tmax - (float)C::P_LIFT;
                corr = merge_weight(mo, mn);
                m_s[hg0 + R] = mn;
                moved_mine = true;
              }
              corr_s[hg0 + R] = corr;
            }
            const bool moved = soft_bar_or(grp, moved_mine);
            if (i > 0) {  // (on a unit's first tile the sums are still 0)
#pragma unroll
              for (int h = 0; h < HG; ++h) lp[h] *= corr_s[hg0 + h];
            }
            compute_y(y);  // against the moved maxima
            if (i > 0 && moved) {
              // O^T holds P.V of the unit's tiles so far: rescale it once the
              // last of them landed (the same decision in every thread)
              wait(bars.pv_done((tg - 1) % C::PB), ((tg - 1) / C::PB) & 1);
              tc::fence_after();
#pragma unroll 1
              for (int cc = 0; cc < (C::F8N ? 2 : 1) * HG; cc += HCH) {  // rare: kept small
                // (F8N: the columns of both P terms of the group's heads)
                const int c0 = cc % HG;
                const uint32_t ta = trow + C::TM_O + ob * C::NM + (cc / HG) * NR + hg0 + c0;
                uint32_t r[32];
                if constexpr (HCH == 32) {
                  tc::ld_32x32b_x32(ta, r);
                } else {
                  tc::ld_32x32b_x16(ta, r);
                }
                tc::wait_ld();
#pragma unroll
                for (int c = 0; c < HCH; ++c)
                  r[c] = __float_as_uint(__uint_as_float(r[c]) * corr_s[hg0 + c0 + c]);
                if constexpr (HCH == 32) {
                  tc::st_32x32b_x32(ta, r);
                } else {
                  tc::st_32x32b_x16(ta, r);
                }
              }
              tc::wait_st();
            }
          }
          // row R of P^T (position R; the group's heads): 2^y, packed in
          // pairs; F8N: P in f16, then its two E4M3 terms P_hi = e4m3(P) and
          // P_lo = e4m3(32 (P - P_hi)) (P <= 2^8 under the lazy max, so
          // |P - P_hi| <= 8 and neither saturates), HG codes of each
          uint32_t pk[HG / 2];
#pragma unroll
          for (int h = 0; h < HG; h += 2) {
            const float p0 = tc::ex2(y[h]), p1 = tc::ex2(y[h + 1]);
            if constexpr (PACK) {
              const float2 l2 = __fadd2_rn(make_float2(lp[h], lp[h + 1]), make_float2(p0, p1));
              lp[h] = l2.x;
              lp[h + 1] = l2.y;
            } else {
              lp[h] += p0;
              lp[h + 1] += p1;
            }
            if constexpr (C::F8N) {
              const uint32_t ph = pack_f16x2(p0, p1);
              const uint32_t c_hi = f16x2_to_e4m3x2(ph);
              const uint32_t c_lo = f16x2_to_e4m3x2(hmul2_32(hsub2_u32(ph, e4m3x2_to_f16x2(c_hi))));
              // hi codes fill the first HG/4 words, lo codes the next HG/4
              const int w = h >> 2, sh = (h & 2) * 8;
              if ((h & 2) == 0) {
                pk[w] = c_hi;
                pk[HG / 4 + w] = c_lo;
              } else {
                pk[w] |= c_hi << sh;
                pk[HG / 4 + w] |= c_lo << sh;
              }
            } else {
              pk[h >> 1] = C::FP8 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
            }
          }
          // the P buffer was last read by the P.V of tile tg - PB
          const int pb = tg % C::PB;
          if (tg >= C::PB) wait(bars.pv_done(pb), ((tg / C::PB) - 1) & 1);
          {
            const uint32_t row = pbase + pb * C::P_BYTES + R * C::P_ROW;
            const int swz = (R >> C::P_SWZ_SHIFT) & C::P_SWZ_MASK;
#pragma unroll
            for (int c = 0; c < HG / 8; ++c) {
              // F8N: chunks [0, HG/16) hold the hi codes, the next HG/16 the
              // lo codes (the row is NR hi codes, then NR lo codes; HG = NR)
              const int chunk = (hg0 >> 3) + c;
              asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(row + ((chunk ^ swz) << 4)),
                           "r"(pk[4 * c]), "r"(pk[4 * c + 1]), "r"(pk[4 * c + 2]), "r"(pk[4 * c + 3])
                           : "memory");
            }
          }
          if (!C::CONV && grp == 0 && !valid && !dead && mbar_wait(pipe.full(st), (tg / ST) & 1)) {
            // position past L: its V row may hold anything (NaN included) and
            // 0 * NaN = NaN inside the MMA, so clear it (after it landed;
            // bf16: two 128-byte boxes, E4M3: one)
            const uint32_t a = pipe.v_tile(st) + R * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(a + 16 * c), "r"(0u) : "memory");
              if (!C::FP8)
                asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(a + Pipe::BOX_BYTES + 16 * c), "r"(0u)
                             : "memory");
            }
          }
          fence_proxy_async_smem();
          tc::fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(bars.s_free(sb));
            mbar_arrive(bars.p_full(tg % C::PB));
          }
        }
        t += ntl;
        // the S^T of every tile of this unit is done, so Q may take the next unit
        Segment nseg;
        const bool next = cur.next(sp, nseg);
        if (next && grp == 0) {
          if constexpr (C::QB == 2) {
            // unit + 1's Q was issued a unit ago; unit + 2's goes to this
            // unit's buffer, whose S^T MMAs have all completed
            SegmentCursor la = cur;
            Segment s2;
            const bool has2 = la.next(sp, s2);
            if (has2) issue_q(s2, unit & 1);
            complete_q((unit + 1) & 1, has2);
          } else {
            issue_q(nseg, 0);
            complete_q(0, false);
          }
        }
        // ---- epilogue: l[h] summed over the 128 positions' partials
        const float mR = R < HG ? m_s[hg0 + R] : 0.f;  // kNoMax when the row saw no position
        soft_reduce<C, false>(lp, grp, sub, lane, red, fin, R);
        // O^T of this unit is final once the P.V of its last tile landed
        wait(bars.pv_done((t - 1) % C::PB), ((t - 1) / C::PB) & 1);
        tc::fence_after();
        // cluster plan: the cluster merges the partials of its one unit after
        // the barrier at the end (at most one segment per CTA, always a
        // partial, even when the piece is the whole unit)
        const bool clm = range.cl;
        const bool whole = !clm && seg.t0 == 0 && seg.t1 == seg.tiles;
        const int slot = partial_slot(unit);
        const size_t orow_b = MULTI ? (size_t)b * p.tokens * p.heads_q + (size_t)(h_first / p.n_rep) * p.rep_kv
                                    : (size_t)b * p.H + h_first;
        const int d4 = 32 * sub + (lane & ~3);
        // columns [c0, c0 + HCH) of the group's heads of O^T (dimension R):
        // F8N adds the P_lo term's columns / 32
        auto load_o = [&](int c0, float(&o)[32]) {
          uint32_t r[32];
          if constexpr (HCH == 32) {
            tc::ld_32x32b_x32(trow + C::TM_O + ob * C::NM + hg0 + c0, r);
          } else {
            tc::ld_32x32b_x16(trow + C::TM_O + ob * C::NM + hg0 + c0, r);
          }
          if constexpr (C::F8N) {
            uint32_t r1[32];
            if constexpr (HCH == 32) {
              tc::ld_32x32b_x32(trow + C::TM_O + ob * C::NM + NR + hg0 + c0, r1);
            } else {
              tc::ld_32x32b_x16(trow + C::TM_O + ob * C::NM + NR + hg0 + c0, r1);
            }
            tc::wait_ld();
#pragma unroll
            for (int c = 0; c < HCH; ++c) o[c] = fmaf(__uint_as_float(r1[c]), 0.03125f, __uint_as_float(r[c]));
          } else {
            tc::wait_ld();
#pragma unroll
            for (int c = 0; c < HCH; ++c) o[c] = __uint_as_float(r[c]);
          }
        };
        if (!whole) {
          // a cut unit's partial: thread R writes dimension R of every head
          // (consecutive lanes, consecutive words: each warp store is one
          // 128-byte line, and no transpose is needed)
          float *orow = p.o_part + (size_t)slot * p.heads_per_cta * D + R;
#pragma unroll 1
          for (int c0 = 0; c0 < (GQA_SLOT_OK(p, slot, nh - 1) ? HG : 0); c0 += HCH) {
            float o[32];
            load_o(c0, o);
#pragma unroll
            for (int c = 0; c < HCH; ++c)
              if (hg0 + c0 + c < nh) orow[(size_t)(hg0 + c0 + c) * D] = o[c] * vscale;
          }
        }
        // a whole unit goes to out: thread R holds output dimension R of
        // every head; a 4x4 transpose within each quad of lanes gives lane j
        // of a quad four consecutive dimensions d4..d4+3 of head (block + j),
        // written as one 8-byte vector.  One column chunk at a time, the chunk
        // loop not unrolled: this code runs once per unit, and with 64
        // columns its size (instruction fetch), not its loads, is what it costs
#pragma unroll 1
        for (int c0 = 0; c0 < (whole ? HG : 0); c0 += HCH) {
          float o[32];
          load_o(c0, o);
#pragma unroll
          for (int q = 0; q < HCH; q += 4) {
            float v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] = o[q + i] * vscale;
            quad_transpose(v, lane);
            const int h = hg0 + c0 + q + (lane & 3);
            if (h < nh) {
              if (whole) {
                // output row of head h: (b*tokens + t)*heads_q + g*rep_kv + k
                // for row h_first % n_rep + h = t*rep_kv + k of the group
                size_t orow = orow_b + h;
                if constexpr (MULTI) {
                  const int row = h_first % p.n_rep + h;
                  orow = orow_b + (size_t)(row / p.rep_kv) * p.heads_q + row % p.rep_kv;
                }
                const float f = fin[h];
                const bool seen = !MULTI || f > 0.f;  // a row that saw no position is 0
                uint2 pk;
                pk.x = pack_bf16x2(seen ? v[0] / f : 0.f, seen ? v[1] / f : 0.f);
                pk.y = pack_bf16x2(seen ? v[2] / f : 0.f, seen ? v[3] / f : 0.f);
                if (GQA_ROW_OK(p, orow))
                  *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(p.out) + orow * D + d4) = pk;
              }
            }
          }
        }
        if (!whole && R < HG && hg0 + R < nh && GQA_SLOT_OK(p, slot, hg0 + R))
          reinterpret_cast<float2 *>(p.ml_part)[(size_t)slot * p.heads_per_cta + hg0 + R] =
              make_float2(mR, fin[hg0 + R]);
        // merge kernel (no cluster launch): where the unit's partials are
        if (R == 0 && grp == 0) record_unit(p, seg, whole, slot, range, b);
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.o_free(ob));
        soft_bar(grp);  // fin[] is reused by the next unit's reductions
        seg = nseg;
        have = next;
      }
      if (STEP && !lens_read) signal_lengths_read(um, lane);
    } else if constexpr (C::CONV) {
      // ------------------------------------------------------------ FP8 converters
      // Thread R converts position R of every tile (R = the TMEM lane its
      // warp may access): its K row of 128 E4M3 codes (one 128-byte swizzled
      // row as TMA landed it) becomes 64 f16 pairs in TMEM lane R of the
      // tile's K buffer, the A operand of S^T; its V row becomes two 128-byte
      // swizzled rows of f16 in the tile's V staging buffer, zeros at or past
      // L (the codes there may be NaN, and 0 * NaN = NaN in the P.V MMA; a
      // NaN logit is masked by the softmax, so K rows need no clearing).
      // K buffer tg & 1 is free once the S^T of tile tg - 2 has completed,
      // V buffer tg % VSTG once the P.V of tile tg - VSTG has.
      const int R = 32 * (warp & 3) + lane;
      const uint32_t tlane = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
      SegmentCursor cur;
      cur.init(sp, range);
      Segment seg;
      bool dead = false;
      int tg = 0;
      bool lens_read = !STEP || !p.append;
      while (cur.next(sp, seg)) {
        const int L = attn_len(p.seq_lens, seg.b, p.Nmax, p.append);
        if (STEP && !lens_read && cur.end - cur.pos <= cur.cost) {
          signal_lengths_read(um, lane);
          lens_read = true;
        }
        for (int t = seg.t0; t < seg.t1; ++t, ++tg) {
          const int st = tg % ST, cb = tg & 1;
          if (!dead && !warp_wait(pipe.full(st), (tg / ST) & 1)) dead = true;
          // the codes of this position go to registers first, so that the
          // ring stage is released before the conversion (the producer's
          // next copy into it then overlaps the conversion)
          uint4 kw[8], vw[8];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            kw[c] = lds128(swz128(pipe.k_tile(st), R, c));
            vw[c] = lds128(swz128(pipe.v_tile(st), R, c));
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(pipe.empty(st));
          if (tg >= 2 && !dead && !warp_wait(bars.s_full(cb), ((tg >> 1) - 1) & 1)) dead = true;
          {
            uint32_t kr[64];
#pragma unroll
            for (int c = 0; c < 8; ++c) {  // 16 codes -> 8 f16 pairs
              const uint32_t ww[4] = {kw[c].x, kw[c].y, kw[c].z, kw[c].w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                kr[8 * c + 2 * i] = e4m3x2_to_f16x2(ww[i] & 0xffffu);
                kr[8 * c + 2 * i + 1] = e4m3x2_to_f16x2(ww[i] >> 16);
              }
            }
            tc::st_32x32b_x64(tlane + C::TM_K + cb * 64, kr);
          }
          const int vb = tg % C::VSTG;
          if (tg >= C::VSTG && !dead && !warp_wait(bars.stg_free(vb), ((tg / C::VSTG) - 1) & 1)) dead = true;
          const bool valid = t * BN + R < L;
          const uint32_t dst = pipe.base + C::STG_OFF + vb * C::STG_TILE;
#pragma unroll
          for (int c = 0; c < 8; ++c) {  // 16 codes -> 16 f16 (two 16-byte chunks)
            uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
            if (valid) {
              const uint32_t ww[4] = {vw[c].x, vw[c].y, vw[c].z, vw[c].w};
              uint32_t o[8];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                o[2 * i] = e4m3x2_to_f16x2(ww[i] & 0xffffu);
                o[2 * i + 1] = e4m3x2_to_f16x2(ww[i] >> 16);
              }
              lo = make_uint4(o[0], o[1], o[2], o[3]);
              hi = make_uint4(o[4], o[5], o[6], o[7]);
            }
            const uint32_t box = dst + (c >> 2) * C::KV_BOX;
            const int k0 = 2 * (c & 3);
            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(swz128(box, R, k0)), "r"(lo.x), "r"(lo.y),
                         "r"(lo.z), "r"(lo.w)
                         : "memory");
            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(swz128(box, R, k0 + 1)), "r"(hi.x),
                         "r"(hi.y), "r"(hi.z), "r"(hi.w)
                         : "memory");
          }
          tc::wait_st();
          fence_proxy_async_smem();
          tc::fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bars.conv_full(cb));
        }
      }
      if (STEP && !lens_read) signal_lengths_read(um, lane);
    }
  }
  // fused step: the producer, done with its copies, counts the CTA once every
  // reader of the lengths has signalled (an empty range has none)
  if (STEP && warp == 0 && p.append) arrive_step_early(p, um, range.begin < range.end ? C::LEN_READERS : 0, lane);
  // ---- cluster plan: the k CTAs of the cluster wrote the partials of the k
  // pieces of the same unit to their workspace slots (a CTA with an empty
  // piece wrote none); after the barrier (cluster-scope release / acquire,
  // which orders those global writes) the CTA of rank r merges the heads
  // [r*ceil(nh/k), ...) from all of them.  No second launch and no second
  // barrier: nothing is read from the peers' shared memory.  The plan is the
  // same in every CTA, so either every CTA of a cluster comes here or none
  // does.
  if (range.cl) {
    cluster_sync_all();
    if (warp >= C::SOFT_WARP0 && warp < C::CONV_WARP0)
      merge_cluster_unit<C, MULTI>(p, range, threadIdx.x - 32 * C::SOFT_WARP0, C::SG * C::SOFT);
  }
  // ---- teardown: every tcgen05 operation has completed (the MMA threads
  // waited for their last commits); free the tensor memory
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    tc::tmem_dealloc(tmem, C::TM_COLS);
  }
  if (!STEP && p.append) finish_step(p, threadIdx.x, blockDim.x, &um->last);
}

}  // namespace gqa
