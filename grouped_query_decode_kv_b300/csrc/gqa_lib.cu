// libgqa.so: host side of the C ABI declared in include/gqa.h — argument
// checks, the split plan, TMA descriptors and the kernel launches.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <mutex>
#include <utility>

#include "gqa.h"
#include "gqa_device.cuh"
#include "gqa_params.cuh"
#include "gqa_probe.cuh"
#include "gqa_proj_tc.cuh"
#include "gqa_small_kernels.cuh"
#include "gqa_split_mma.cuh"
#include "gqa_split_simt.cuh"
#include "gqa_split_tc.cuh"
#include "gqa_selftest.cuh"

namespace gqa {
namespace {

// ----------------------------------------------------------- kernel configs
// Stages of ~32 KB (K + V tiles).  Ring and per-unit merge scratch are sized
// so that two CTAs fit on one SM where registers allow.
using MmaD128x1 = MmaCfg<128, 1, 1, 64, 3, 2>;  // n_rep 3..16
using MmaD128x2 = MmaCfg<128, 2, 1, 64, 2>;   // n_rep 17..32
using MmaD128x4 = MmaCfg<128, 2, 2, 64, 2>;   // n_rep >= 33 (64 heads per CTA)
using MmaD64x1 = MmaCfg<64, 1, 1, 128, 3, 2>;
using MmaD64x2 = MmaCfg<64, 2, 1, 128, 2>;
using MmaD64x4 = MmaCfg<64, 2, 2, 128, 2>;

template <typename T, int D, int NH>
using SimtFor = SimtCfg<T, D, NH, (32768 / (2 * D * (int)sizeof(T))), 3>;
// FP8 E4M3 cache, bf16 q and out: 64 positions (16 KB of K and V) per stage,
// so that more CTAs share an SM (measured best for MHA: 56 us vs 70 us with 128)
template <int NH>
using SimtFp8 = SimtCfg<e4m3_t, 128, NH, 64, 3, __nv_bfloat16>;

struct KernelChoice {
  const void *func;
  int family;
  int threads;
  int smem;
  int block_n;
  int heads;
  int box_elems;
  cudaError_t (*launch)(dim3, int, const CUtensorMap &, const CUtensorMap &, const CUtensorMap *,
                        const SplitParams &, cudaStream_t);
  // the fused decode step's instantiation, where it has its own (null: the
  // kernel above serves the step too)
  const void *func_step;
  cudaError_t (*launch_step)(dim3, int, const CUtensorMap &, const CUtensorMap &, const CUtensorMap *,
                             const SplitParams &, cudaStream_t);
  int (*clusters)(int);  // max_clusters of the kernel
};

// Launch with programmatic stream serialisation: the kernel may start while
// the previous kernel in the stream finishes; it calls griddepcontrol.wait
// before reading anything that kernel writes.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

enum Family { kSimt = 0, kMma = 1, kTc = 2 };

// MULTI: the instantiation for several query tokens per sequence; the
// one-token kernels are compiled without any of that code.  STEP: the fused
// decode step's instantiation.
template <class C, int F, bool MULTI, bool STEP = false>
auto split_kernel_ptr() {
  if constexpr (F == kMma)
    return &gqa_split_mma_kernel<C, MULTI, STEP>;
  else if constexpr (F == kTc)
    return &gqa_split_tc_kernel<C, MULTI, STEP>;
  else
    return &gqa_split_simt_kernel<C, MULTI, STEP>;
}

// The same in thread-block clusters of `cluster` CTAs along x.
template <typename... Params, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, int cluster,
                               cudaStream_t st, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cluster > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// tail[2]: the caches' maps with 16-position boxes (the tcgen05 kernel reads
// the short last tile of a unit through them; the others take none).
template <class C, int F, bool MULTI, bool STEP = false>
cudaError_t launch_split(dim3 grid, int cluster, const CUtensorMap &k, const CUtensorMap &v, const CUtensorMap *tail,
                         const SplitParams &p, cudaStream_t st) {
  if constexpr (F == kTc)
    return launch_pdl_cluster(split_kernel_ptr<C, F, MULTI, STEP>(), grid, dim3(C::THREADS), C::SMEM_BYTES, cluster,
                              st, k, v, tail[0], tail[1], p);
  else
    return launch_pdl_cluster(split_kernel_ptr<C, F, MULTI, STEP>(), grid, dim3(C::THREADS), C::SMEM_BYTES, cluster,
                              st, k, v, p);
}

// Clusters of `cluster` CTAs of this kernel that can be resident at once (0
// when the query fails); asked once per device and cluster size.
template <class C, int F, bool MULTI>
int max_clusters(int cluster) {
  static std::mutex mu;
  static int cache[64][9];  // [device][cluster], 0 = not asked yet, -1 = failed
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || cluster < 1 || cluster > 8) {
    cudaGetLastError();
    return 0;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev][cluster] != 0) return cache[dev][cluster] > 0 ? cache[dev][cluster] : 0;
  if (cudaFuncSetAttribute(split_kernel_ptr<C, F, MULTI>(), cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::SMEM_BYTES) != cudaSuccess) {
    cudaGetLastError();
    cache[dev][cluster] = -1;
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster * 64);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, split_kernel_ptr<C, F, MULTI>(), &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    cache[dev][cluster] = -1;
    return 0;
  }
  cache[dev][cluster] = n;
  return n;
}

template <class C, int F, bool MULTI>
KernelChoice make_choice() {
  KernelChoice c;
  c.func = reinterpret_cast<const void *>(split_kernel_ptr<C, F, MULTI>());
  c.family = F;
  c.threads = C::THREADS;
  c.smem = C::SMEM_BYTES;
  c.block_n = C::BLOCK_N;
  c.heads = C::HEADS;
  if constexpr (F == kSimt)
    c.box_elems = C::BOX_ELEMS;
  else if constexpr (F == kTc)
    c.box_elems = C::FP8 ? 128 : 64;
  else
    c.box_elems = 64;
  c.launch = &launch_split<C, F, MULTI>;
  // the one-token kernels of the step's dtypes count a fused step's CTAs
  // early (a separate instantiation, so that attention alone keeps its code)
  c.func_step = nullptr;
  c.launch_step = nullptr;
  if constexpr (!MULTI) {
    if constexpr (!C::FP8) {
      c.func_step = reinterpret_cast<const void *>(split_kernel_ptr<C, F, MULTI, true>());
      c.launch_step = &launch_split<C, F, MULTI, true>;
    }
  }
  c.clusters = &max_clusters<C, F, MULTI>;
  return c;
}

// Query heads per KV head from which bf16 d=128 groups go to the tcgen05
// kernel (tensor-core MMAs with TMEM accumulators); smaller groups use the
// warp-level MMA kernel, groups of one or two the CUDA-core kernel.
constexpr int kTcMinNrep = 8;
using TcD128x16 = TcCfg<16, 3, 2>;
using TcD128x32 = TcCfg<32, 3, 2>;
using TcD128x64 = TcCfg<64, 3, 1>;
// several query tokens: the per-row limits make the softmax of a tile
// heavier, and 32 rows per unit are shared by two softmax groups (measured on
// GQA-8 with 4 tokens, B=16, Nmax=8192 ragged: 70.9 -> 64.7 us per call; for
// one token the second group did not pay)
using TcD128x32Multi = TcCfg<32, 3, 2, false, 2>;
// FP8 cache: stages of 32 KB of codes (K and V of 128 positions), two or
// three 32 KB f16 V staging tiles (the f16 K tiles are in tensor memory)
using TcFp8x16 = TcCfg<16, 6, 2, true, 1, 2, true>;
using TcFp8x32 = TcCfg<32, 5, 2, true, 1, 2, true>;
using TcFp8x64 = TcCfg<64, 3, 1, true>;

template <bool M>
KernelChoice choose_kernel(gqa_dtype_t dt, int d, int n_rep) {
  if constexpr (!M) {
    if (dt == GQA_FP8_E4M3) {  // d = 128 (checked by the caller)
      if (n_rep >= kTcMinNrep) {
        if (n_rep <= 16) return make_choice<TcFp8x16, kTc, M>();
        if (n_rep <= 32) return make_choice<TcFp8x32, kTc, M>();
        return make_choice<TcFp8x64, kTc, M>();
      }
      if (n_rep == 1) return make_choice<SimtFp8<1>, kSimt, M>();
      if (n_rep == 2) return make_choice<SimtFp8<2>, kSimt, M>();
      return make_choice<SimtFp8<4>, kSimt, M>();
    }
  }
  if (dt == GQA_BF16) {
    if (d == 128) {
      if (n_rep == 1) return make_choice<SimtFor<__nv_bfloat16, 128, 1>, kSimt, M>();
      if (n_rep == 2) return make_choice<SimtFor<__nv_bfloat16, 128, 2>, kSimt, M>();
      if (n_rep >= kTcMinNrep) {
        if (n_rep <= 16) return make_choice<TcD128x16, kTc, M>();
        if (n_rep <= 32) {
          if constexpr (M) return make_choice<TcD128x32Multi, kTc, M>();
          return make_choice<TcD128x32, kTc, M>();
        }
        return make_choice<TcD128x64, kTc, M>();
      }
      if (n_rep <= 16) return make_choice<MmaD128x1, kMma, M>();
      if (n_rep <= 32) return make_choice<MmaD128x2, kMma, M>();
      return make_choice<MmaD128x4, kMma, M>();
    }
    if (n_rep == 1) return make_choice<SimtFor<__nv_bfloat16, 64, 1>, kSimt, M>();
    if (n_rep == 2) return make_choice<SimtFor<__nv_bfloat16, 64, 2>, kSimt, M>();
    if (n_rep <= 16) return make_choice<MmaD64x1, kMma, M>();
    if (n_rep <= 32) return make_choice<MmaD64x2, kMma, M>();
    return make_choice<MmaD64x4, kMma, M>();
  }
  if (d == 128) {
    if (n_rep == 1) return make_choice<SimtFor<float, 128, 1>, kSimt, M>();
    if (n_rep == 2) return make_choice<SimtFor<float, 128, 2>, kSimt, M>();
    return make_choice<SimtFor<float, 128, 4>, kSimt, M>();
  }
  if (n_rep == 1) return make_choice<SimtFor<float, 64, 1>, kSimt, M>();
  if (n_rep == 2) return make_choice<SimtFor<float, 64, 2>, kSimt, M>();
  return make_choice<SimtFor<float, 64, 4>, kSimt, M>();
}

// ----------------------------------------------------------- split plan
struct Plan {
  KernelChoice k;
  int heads;        // query heads per unit (per CTA segment)
  int head_chunks;  // HC
  int P;            // CTAs of the split kernel
  long long units;  // B * G * HC
  int cluster = 0;  // CTAs per thread-block cluster (0: no clusters)
};

int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

constexpr int kMaxDevices = 64;

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return -1;
  }
  return dev;
}

// SM count of the current device, read once per device (148 without one).
int device_sm_count() {
  static std::atomic<int> cache[kMaxDevices];
  const int dev = current_device();
  if (dev < 0) return 148;
  int sms = cache[dev].load(std::memory_order_relaxed);
  if (sms > 0) return sms;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
    cudaGetLastError();
    return 148;
  }
  cache[dev].store(sms, std::memory_order_relaxed);
  return sms;
}

// Resident CTAs of a split kernel per SM (queried once per kernel; without
// a device, estimated from its shared memory).
int ctas_per_sm(const KernelChoice &kc) {
  static std::mutex mu;
  static const void *funcs[32];
  static int counts[32];
  static int n = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n; ++i)
    if (funcs[i] == kc.func) return counts[i];
  int c = 0;
  if (cudaFuncSetAttribute(kc.func, cudaFuncAttributeMaxDynamicSharedMemorySize, kc.smem) != cudaSuccess ||
      cudaFuncSetAttribute(kc.func, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&c, kc.func, kc.threads, kc.smem) != cudaSuccess || c <= 0) {
    cudaGetLastError();
    return std::max(1, std::min(2, (228 * 1024) / (kc.smem + 1024)));
  }
  if (n < 32) {
    funcs[n] = kc.func;
    counts[n] = c;
    ++n;
  }
  return c;
}

// The split kernel is a persistent grid of one wave (SMs x resident CTAs per
// SM); the stream-K split gives every CTA the same number of tiles whatever
// the lengths.  split_tokens > 0 instead asks for about that many positions
// per CTA when every sequence is full (for tests of the merge and for
// tuning).
// `multi`: the plan of a several-token call (H counts its tokens * heads
// query rows); it picks the kernels compiled for that case.
Plan make_plan(int B, int H, int G, int d, int Nmax, gqa_dtype_t dt, int split_tokens, bool multi = false) {
  Plan pl;
  const int n_rep = H / G;
  // the grid (and so the workspace) is sized from the one-token kernel, so
  // that both instantiations share gqa_decode_workspace_bytes_ex
  const KernelChoice base = choose_kernel<false>(dt, d, n_rep);
  pl.k = multi ? choose_kernel<true>(dt, d, n_rep) : base;
  // the tcgen05 kernel takes a group of up to 64 heads per unit (its MMA N);
  // the others have a fixed number of heads per CTA
  pl.heads = pl.k.family == kTc ? std::min(n_rep, pl.k.heads) : pl.k.heads;
  pl.head_chunks = ceil_div(n_rep, pl.heads);
  pl.units = (long long)B * G * pl.head_chunks;
  const long long tiles_full = pl.units * ceil_div(Nmax, pl.k.block_n);
  long long P;
  if (split_tokens > 0) {
    const long long per_cta = std::max(1, ceil_div(split_tokens, pl.k.block_n));
    P = (tiles_full + per_cta - 1) / per_cta;
  } else {
    P = (long long)device_sm_count() * ctas_per_sm(base);
  }
  P = std::max<long long>(1, std::min<long long>(P, std::min<long long>(tiles_full, 1 << 20)));
  pl.P = (int)P;
  // tcgen05 kernel with room for k = 2..4 CTAs per unit of a full batch:
  // launch in clusters of k, each cluster taking one unit whole, so that a
  // unit's pieces meet in one cluster and are merged by it after a cluster
  // barrier (through the workspace in L2; no merge kernel).  The grid keeps
  // whole clusters and no more of them than can be resident at once.
  if (split_tokens == 0 && pl.k.family == kTc && pl.units > 0) {
    const long long k = P / pl.units;
    if (k >= 2 && k <= 4) {
      const int resident = pl.k.clusters((int)k);
      const long long nclu = std::min<long long>(P / k, resident);
      if (nclu >= pl.units) {
        pl.cluster = (int)k;
        pl.P = (int)(nclu * k);
      }
    }
  }
  return pl;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool plan_fits(const Plan &pl, int B, int G) { return B <= 65535 && pl.units < (1LL << 31); }

// Workspace: a fixed 256-byte head that holds the fused step's arrival
// word, then partial outputs and (m, l) of two slots per CTA, and 8 bytes of
// merge bookkeeping per unit.  The head sits at the same offset for every
// shape, so calls of other shapes (or attention-only calls) that share the
// workspace never write over it.  A single CTA never splits a unit.
constexpr size_t kWsHead = 256;
size_t ws_opart_bytes(const Plan &pl, int d) { return align256((size_t)2 * pl.P * pl.heads * d * sizeof(float)); }
size_t ws_ml_bytes(const Plan &pl) { return align256((size_t)2 * pl.P * pl.heads * 2 * sizeof(float)); }

// A call's epoch tells its counter words from those other calls left in a
// reused workspace; never zero (zero-filled memory reads as a stale word).
unsigned next_epoch() {
  static std::atomic<unsigned> epoch{0};
  unsigned e = epoch.fetch_add(1, std::memory_order_relaxed) + 1;
  if (e == 0) e = epoch.fetch_add(1, std::memory_order_relaxed) + 1;
  return e;
}

size_t ws_book_bytes(const Plan &pl) { return align256((size_t)pl.units * sizeof(unsigned long long)); }

// Every word in it is tagged with the epoch of the call that wrote it, so
// the workspace needs no clearing, ever.
size_t workspace_for(const Plan &pl, int B, int H, int d) {
  (void)B;
  (void)H;
  if (pl.P <= 1) return 0;
  return kWsHead + ws_opart_bytes(pl, d) + ws_ml_bytes(pl) + ws_book_bytes(pl);
}

// ----------------------------------------------------------- workspace allocator
// The workspace of the calls that get their own (gqa_decode_attention,
// gqa_decode_step, ...) comes from the stream-ordered allocator unless the
// caller installed its own with gqa_set_workspace_allocator.
std::atomic<gqa_alloc_fn> g_alloc{nullptr};
std::atomic<gqa_free_fn> g_free{nullptr};
std::atomic<void *> g_alloc_ctx{nullptr};

bool ws_alloc(void **ptr, size_t bytes, cudaStream_t st) {
  *ptr = nullptr;
  if (const gqa_alloc_fn fn = g_alloc.load()) return fn(g_alloc_ctx.load(), ptr, bytes, st) == 0 && *ptr;
  if (cudaMallocAsync(ptr, bytes, st) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return true;
}

// True when the release was accepted (enqueued).
bool ws_free(void *ptr, cudaStream_t st) {
  if (const gqa_free_fn fn = g_free.load()) {
    fn(g_alloc_ctx.load(), ptr, st);
    return true;
  }
  if (cudaFreeAsync(ptr, st) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return true;
}

// ----------------------------------------------------------- TMA descriptors
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// The cache [B*G, Nmax, d] as a 3-D tensor; a box is 128 bytes of one row
// (box_elems elements) by block_n positions, 128-byte swizzled.
bool encode_cache_map(CUtensorMap *map, const void *base, gqa_dtype_t dt, int d, int Nmax, int BG, int block_n,
                      int box_elems) {
  auto fn = encode_fn();
  if (!fn) return false;
  const size_t elt = dt == GQA_FP8_E4M3 ? 1 : (dt == GQA_BF16 ? 2 : 4);
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)Nmax, (cuuint64_t)BG};
  cuuint64_t strides[2] = {(cuuint64_t)(d * elt), (cuuint64_t)((size_t)Nmax * d * elt)};
  cuuint32_t box[3] = {(cuuint32_t)box_elems, (cuuint32_t)block_n, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType ty = dt == GQA_FP8_E4M3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : dt == GQA_BF16   ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                    : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  CUresult r = fn(map, ty, 3,
                  const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_attention_args(const void *q, const void *k, const void *v, const int32_t *sl, const void *out, int B,
                         int H, int G, int d, int Nmax, gqa_dtype_t dt) {
  if (!q || !k || !v || !sl || !out) return GQA_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || G <= 0 || d <= 0 || Nmax <= 0) return GQA_ERR_INVALID_ARG;
  if (H % G != 0) return GQA_ERR_INVALID_ARG;
  if (dt != GQA_F32 && dt != GQA_BF16) return GQA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return GQA_ERR_UNSUPPORTED;
  if (B > 65535) return GQA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return GQA_ERR_INVALID_ARG;
  return GQA_OK;
}

// Opts a split kernel (`func`, of the choice kc) in to its dynamic shared
// memory, once per device.
int ensure_smem_attr(const KernelChoice &kc, const void *func) {
  static std::mutex mu;
  static const void *done_func[256];
  static int done_dev[256];
  static int n = 0;
  const int dev = current_device();
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n; ++i)
    if (done_func[i] == func && done_dev[i] == dev) return GQA_OK;
  if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, kc.smem) != cudaSuccess ||
      cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared) !=
          cudaSuccess) {
    cudaGetLastError();
    return GQA_ERR_CUDA;
  }
  if (n < 256 && dev >= 0) {
    done_func[n] = func;
    done_dev[n] = dev;
    ++n;
  }
  return GQA_OK;
}

// Rows appended by a fused decode step (null for attention alone).
struct StepAppend {
  const void *k_new = nullptr, *v_new = nullptr;
  void *k_cache = nullptr, *v_cache = nullptr;
  int32_t *seq_lens = nullptr;
};

// `tokens` query tokens per sequence: q and out are [B, tokens, H, d] and the
// plan was made for tokens * H query rows.
int run_attention(const void *q, const void *k, const void *v, const int32_t *sl, float scale, void *out, int B,
                  int H, int G, int d, int Nmax, gqa_dtype_t dt, const Plan &pl, void *ws, cudaStream_t st,
                  const StepAppend &app = StepAppend(), int tokens = 1, const float *k_scale = nullptr,
                  const float *v_scale = nullptr) {
  CUtensorMap mk, mv;
  if (!encode_cache_map(&mk, k, dt, d, Nmax, B * G, pl.k.block_n, pl.k.box_elems) ||
      !encode_cache_map(&mv, v, dt, d, Nmax, B * G, pl.k.block_n, pl.k.box_elems))
    return GQA_ERR_CUDA;
  CUtensorMap tail[2];
  if (pl.k.family == kTc && (!encode_cache_map(&tail[0], k, dt, d, Nmax, B * G, 16, pl.k.box_elems) ||
                             !encode_cache_map(&tail[1], v, dt, d, Nmax, B * G, 16, pl.k.box_elems)))
    return GQA_ERR_CUDA;
  const bool own_step = app.k_new != nullptr && pl.k.launch_step != nullptr;
  if (int rc = ensure_smem_attr(pl.k, own_step ? pl.k.func_step : pl.k.func)) return rc;
  SplitParams p;
  p.q = q;
  p.seq_lens = sl;
  p.out = out;
  const bool split = pl.P > 1;
  char *w = reinterpret_cast<char *>(ws);
  p.o_part = split ? reinterpret_cast<float *>(w + kWsHead) : nullptr;
  p.ml_part = split ? reinterpret_cast<float *>(w + kWsHead + ws_opart_bytes(pl, d)) : nullptr;
  // units cut between CTAs merge inside the split kernel for the CUDA-core
  // kernel (the unit's last CTA) and for a cluster launch of the tcgen05
  // kernel (every CTA of the unit's cluster, after a cluster barrier); the
  // rest in the merge kernel, which spreads the (bigger) partials of
  // many-head units over every SM
  void *book = split ? w + kWsHead + ws_opart_bytes(pl, d) + ws_ml_bytes(pl) : nullptr;
  const bool merge_in_kernel = pl.k.family == kSimt || pl.cluster > 1;
  p.unit_cnt = pl.k.family == kSimt ? reinterpret_cast<unsigned long long *>(book) : nullptr;
  p.unit_info = merge_in_kernel ? nullptr : reinterpret_cast<int2 *>(book);
  p.epoch = next_epoch();
  p.cluster_k = pl.cluster;
  p.P = pl.P;
  p.append = app.k_new != nullptr;
  p.k_new = app.k_new;
  p.v_new = app.v_new;
  p.k_cache = app.k_cache;
  p.v_cache = app.v_cache;
  p.seq_lens_w = app.seq_lens;
  p.row_chunks = d * (dt == GQA_FP8_E4M3 ? 1 : (dt == GQA_BF16 ? 2 : 4)) / 16;
  p.done_cnt = split ? reinterpret_cast<unsigned long long *>(w) : nullptr;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.B = B;
  p.H = tokens * H;
  p.G = G;
  p.Nmax = Nmax;
  p.n_rep = tokens * (H / G);
  p.heads_per_cta = pl.heads;
  p.head_chunks = pl.head_chunks;
  p.tokens = tokens;
  p.heads_q = H;
  p.rep_kv = H / G;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  const auto launch = own_step ? pl.k.launch_step : pl.k.launch;
  if (launch(dim3(pl.P), pl.cluster, mk, mv, tail, p, st) != cudaSuccess) {
    cudaGetLastError();
    return GQA_ERR_CUDA;
  }
  if (split && !merge_in_kernel) {
    const dim3 blocks(ceil_div((long long)B * p.H, 4));
    cudaError_t e;
    if (dt == GQA_BF16 || dt == GQA_FP8_E4M3)  // out is bf16 for an FP8 cache too
      e = d == 128 ? launch_pdl(gqa_combine_kernel<__nv_bfloat16, 128>, blocks, dim3(128), 0, st, p)
                   : launch_pdl(gqa_combine_kernel<__nv_bfloat16, 64>, blocks, dim3(128), 0, st, p);
    else
      e = d == 128 ? launch_pdl(gqa_combine_kernel<float, 128>, blocks, dim3(128), 0, st, p)
                   : launch_pdl(gqa_combine_kernel<float, 64>, blocks, dim3(128), 0, st, p);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return GQA_ERR_CUDA;
    }
  }
  return GQA_OK;
}

}  // namespace
}  // namespace gqa

// Fixed split scratch of gqa_decode_attention_noalloc: partial outputs and
// softmax states of one call.  A static device array, so every device that
// loads the library holds it until the process exits; calls on one device
// share it (see gqa.h).
static __device__ __align__(256) unsigned char g_noalloc_scratch[GQA_NOALLOC_SCRATCH_BYTES];

namespace gqa {
namespace {

// Device address of g_noalloc_scratch for the current device.  In host code
// the array's name is only a host-side stand-in, so the real address is
// looked up once per device (with that device current) and cached.
std::mutex g_noalloc_mutex;
void *g_noalloc_ptr[kMaxDevices] = {};

int noalloc_scratch(void **ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return GQA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return GQA_ERR_CUDA;
    }
    g_noalloc_ptr[dev] = p;
  }
  *ptr = g_noalloc_ptr[dev];
  return GQA_OK;
}

}  // namespace
}  // namespace gqa

namespace gqa {
namespace {
// ----------------------------------------------------------- Q/K/V projections
constexpr int kProjMaxBatch = 256;  // batch rows per launch (N of the MMA); larger batches run in chunks
constexpr int kProjKT = 64;         // input features per pipeline stage

int proj_nb(int B) {
  int nb = 16;
  while (nb < B) nb *= 2;
  return nb;
}

struct ProjPlan {
  int nb;      // padded batch columns of one launch
  int items;   // projection items (128 output features each)
  int items_q, items_kv;
  int ktiles;
  int P;       // CTAs
};

ProjPlan make_proj_plan(int B, int A, int H, int G, int d) {
  ProjPlan pl;
  pl.nb = proj_nb(std::min(B, kProjMaxBatch));
  pl.items_q = d == 128 ? H : (H + 1) / 2;
  pl.items_kv = d == 128 ? G : (G + 1) / 2;
  pl.items = pl.items_q + 2 * pl.items_kv;
  pl.ktiles = A / kProjKT;
  const long long T = (long long)pl.items * pl.ktiles;
  pl.P = (int)std::max<long long>(1, std::min<long long>(T, device_sm_count()));
  return pl;
}

size_t proj_part_bytes(const ProjPlan &pl) { return align256((size_t)2 * pl.P * pl.nb * 128 * sizeof(float)); }
size_t proj_workspace(const ProjPlan &pl) {
  if (pl.P <= 1) return 0;
  return proj_part_bytes(pl) + align256((size_t)pl.items * sizeof(unsigned long long));
}

int check_proj_args(const void *x, const void *wq, const void *wk, const void *wv, const void *q, const void *k,
                    const void *v, int B, int A, int H, int G, int d, gqa_dtype_t dt) {
  if (!x || !wq || !wk || !wv || !q || !k || !v) return GQA_ERR_INVALID_ARG;
  if (B <= 0 || A <= 0 || H <= 0 || G <= 0 || d <= 0 || H % G != 0) return GQA_ERR_INVALID_ARG;
  if (dt != GQA_F32 && dt != GQA_BF16) return GQA_ERR_INVALID_ARG;
  if (dt != GQA_BF16 || (d != 64 && d != 128) || A % kProjKT != 0) return GQA_ERR_UNSUPPORTED;
  if ((long long)A * 2 >= (1LL << 40) || H > 65535 || B > (1 << 24)) return GQA_ERR_UNSUPPORTED;
  for (const void *ptr : {x, wq, wk, wv, q, k, v})
    if (!aligned16(ptr)) return GQA_ERR_INVALID_ARG;
  return GQA_OK;
}

// P [heads, A, d] bf16 as a 3-D tensor (d, A, heads); a box is 64 outputs
// (128 bytes) by 64 inputs of one head, 128-byte swizzled.
bool encode_weight_map(CUtensorMap *map, const void *w, int heads, int A, int d) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)A, (cuuint64_t)heads};
  cuuint64_t strides[2] = {(cuuint64_t)(d * 2), (cuuint64_t)((size_t)A * d * 2)};
  cuuint32_t box[3] = {64, (cuuint32_t)kProjKT, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(w), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// x [B, A] bf16 as a 2-D tensor; a box is 64 inputs by `nb` rows (rows past
// B read as zeros), 128-byte swizzled: the K-major B operand.
bool encode_x_map(CUtensorMap *map, const void *x, int B, int A, int nb) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)A, (cuuint64_t)B};
  cuuint64_t strides[1] = {(cuuint64_t)A * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)nb};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(x), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NB>
int launch_proj(const CUtensorMap &mx, const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                const ProjParams &p, int P, cudaStream_t st) {
  using C = ProjCfg<NB, kProjKT>;
  static std::once_flag once[kMaxDevices];
  const int dev = current_device();
  if (dev < 0) return GQA_ERR_CUDA;
  bool attr_ok = true;
  std::call_once(once[dev], [&] {
    attr_ok = cudaFuncSetAttribute(gqa_qkv_proj_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   C::SMEM_BYTES) == cudaSuccess;
  });
  if (!attr_ok ||
      launch_pdl(gqa_qkv_proj_kernel<C>, dim3(P), dim3(C::THREADS), C::SMEM_BYTES, st, mx, mq, mk, mv, p) !=
          cudaSuccess) {
    cudaGetLastError();
    return GQA_ERR_CUDA;
  }
  return GQA_OK;
}

int run_projection(const void *x, const void *wq, const void *wk, const void *wv, void *q, void *k, void *v, int B,
                   int A, int H, int G, int d, void *ws, cudaStream_t st) {
  const ProjPlan pl = make_proj_plan(B, A, H, G, d);
  CUtensorMap mq, mk, mv;
  if (!encode_weight_map(&mq, wq, H, A, d) || !encode_weight_map(&mk, wk, G, A, d) ||
      !encode_weight_map(&mv, wv, G, A, d))
    return GQA_ERR_CUDA;
  char *w = reinterpret_cast<char *>(ws);
  for (int b0 = 0; b0 < B; b0 += kProjMaxBatch) {
    const int nbat = std::min(kProjMaxBatch, B - b0);
    const int nb = proj_nb(nbat);
    CUtensorMap mx;
    if (!encode_x_map(&mx, reinterpret_cast<const char *>(x) + (size_t)b0 * A * 2, nbat, A, nb)) return GQA_ERR_CUDA;
    ProjParams p;
    p.out[0] = reinterpret_cast<char *>(q) + (size_t)b0 * H * d * 2;
    p.out[1] = reinterpret_cast<char *>(k) + (size_t)b0 * G * d * 2;
    p.out[2] = reinterpret_cast<char *>(v) + (size_t)b0 * G * d * 2;
    p.heads[0] = H;
    p.heads[1] = G;
    p.heads[2] = G;
    p.item_start[0] = 0;
    p.item_start[1] = pl.items_q;
    p.item_start[2] = pl.items_q + pl.items_kv;
    p.item_start[3] = pl.items;
    p.ktiles = pl.ktiles;
    p.B = nbat;
    p.d = d;
    p.part = pl.P > 1 ? reinterpret_cast<float *>(w) : nullptr;
    p.item_cnt = pl.P > 1 ? reinterpret_cast<unsigned long long *>(w + proj_part_bytes(pl)) : nullptr;
    p.epoch = next_epoch();
    int rc;
    switch (nb) {
      case 16: rc = launch_proj<16>(mx, mq, mk, mv, p, pl.P, st); break;
      case 32: rc = launch_proj<32>(mx, mq, mk, mv, p, pl.P, st); break;
      case 64: rc = launch_proj<64>(mx, mq, mk, mv, p, pl.P, st); break;
      case 128: rc = launch_proj<128>(mx, mq, mk, mv, p, pl.P, st); break;
      default: rc = launch_proj<256>(mx, mq, mk, mv, p, pl.P, st); break;
    }
    if (rc) return rc;
  }
  return GQA_OK;
}
}  // namespace
}  // namespace gqa

using namespace gqa;

extern "C" {

int gqa_set_workspace_allocator(gqa_alloc_fn alloc, gqa_free_fn free_fn, void *ctx) {
  if ((alloc == nullptr) != (free_fn == nullptr)) return GQA_ERR_INVALID_ARG;
  g_alloc_ctx.store(ctx);
  g_free.store(free_fn);
  g_alloc.store(alloc);
  return GQA_OK;
}

int gqa_wait_timeout_selftest(int which, cudaStream_t stream) {
  if (which < 0 || which > 2) return GQA_ERR_INVALID_ARG;
  gqa_wait_selftest_kernel<<<1, 32, 0, stream>>>(which);
  if (cudaGetLastError() != cudaSuccess) return GQA_ERR_CUDA;
  return GQA_OK;
}

int gqa_stream_read(const void *buf, size_t bytes, int mode, uint32_t *sink, cudaStream_t stream) {
  if (!buf || !sink || !aligned16(buf) || bytes == 0) return GQA_ERR_INVALID_ARG;
  const int sms = device_sm_count();
  cudaError_t e;
  if (mode == 0) {
    if (bytes % 16) return GQA_ERR_INVALID_ARG;
    gqa_read_ldg_kernel<<<sms * 4, kProbeLdgThreads, 0, stream>>>(reinterpret_cast<const uint4 *>(buf), bytes / 16,
                                                                   sink);
    e = cudaGetLastError();
  } else if (mode == 1) {
    if (bytes % kProbeChunk) return GQA_ERR_INVALID_ARG;
    static std::once_flag once[kMaxDevices];
    const int dev = current_device();
    if (dev < 0) return GQA_ERR_CUDA;
    bool ok = true;
    std::call_once(once[dev], [&] {
      ok = cudaFuncSetAttribute(gqa_read_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kProbeBulkSmem) ==
           cudaSuccess;
    });
    if (!ok) {
      cudaGetLastError();
      return GQA_ERR_CUDA;
    }
    gqa_read_bulk_kernel<<<sms, kProbeBulkThreads, kProbeBulkSmem, stream>>>(reinterpret_cast<const uint8_t *>(buf),
                                                                              bytes / kProbeChunk, sink);
    e = cudaGetLastError();
  } else {
    return GQA_ERR_INVALID_ARG;
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GQA_ERR_CUDA;
  }
  return GQA_OK;
}

size_t gqa_decode_workspace_bytes_ex(int B, int H, int G, int d, int Nmax, gqa_dtype_t dtype, int split_tokens) {
  if (B <= 0 || H <= 0 || G <= 0 || Nmax <= 0 || H % G != 0 || (d != 64 && d != 128)) return 0;
  if (dtype != GQA_F32 && dtype != GQA_BF16) return 0;
  return workspace_for(make_plan(B, H, G, d, Nmax, dtype, split_tokens), B, H, d);
}

size_t gqa_decode_workspace_bytes(int B, int H, int G, int d, int Nmax, gqa_dtype_t dtype) {
  return gqa_decode_workspace_bytes_ex(B, H, G, d, Nmax, dtype, 0);
}

int gqa_decode_attention_ex(const void *q, const void *k_cache, const void *v_cache, const int32_t *seq_lens,
                            float scale, void *out, int B, int H, int G, int d, int Nmax, gqa_dtype_t dtype,
                            int split_tokens, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (int rc = check_attention_args(q, k_cache, v_cache, seq_lens, out, B, H, G, d, Nmax, dtype)) return rc;
  if (split_tokens < 0) return GQA_ERR_INVALID_ARG;
  const Plan pl = make_plan(B, H, G, d, Nmax, dtype, split_tokens);
  if (!plan_fits(pl, B, G)) return GQA_ERR_UNSUPPORTED;
  const size_t need = workspace_for(pl, B, H, d);
  if (need > 0 && (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
    return GQA_ERR_INVALID_ARG;
  return run_attention(q, k_cache, v_cache, seq_lens, scale, out, B, H, G, d, Nmax, dtype, pl, workspace, stream);
}

int gqa_decode_attention_ws(const void *q, const void *k_cache, const void *v_cache, const int32_t *seq_lens,
                            float scale, void *out, int B, int H, int G, int d, int Nmax, gqa_dtype_t dtype,
                            void *workspace, size_t workspace_bytes, cudaStream_t stream) {
  return gqa_decode_attention_ex(q, k_cache, v_cache, seq_lens, scale, out, B, H, G, d, Nmax, dtype, 0, workspace,
                                 workspace_bytes, stream);
}

int gqa_decode_attention(const void *q, const void *k_cache, const void *v_cache, const int32_t *seq_lens,
                         float scale, void *out, int B, int H, int G, int d, int Nmax, gqa_dtype_t dtype,
                         cudaStream_t stream) {
  if (int rc = check_attention_args(q, k_cache, v_cache, seq_lens, out, B, H, G, d, Nmax, dtype)) return rc;
  const Plan pl = make_plan(B, H, G, d, Nmax, dtype, 0);
  if (!plan_fits(pl, B, G)) return GQA_ERR_UNSUPPORTED;
  const size_t need = workspace_for(pl, B, H, d);
  void *ws = nullptr;
  if (need > 0) {
    if (!ws_alloc(&ws, need, stream)) return GQA_ERR_NO_MEMORY;
  }
  int rc = run_attention(q, k_cache, v_cache, seq_lens, scale, out, B, H, G, d, Nmax, dtype, pl, ws, stream);
  if (ws && !ws_free(ws, stream) && rc == GQA_OK) rc = GQA_ERR_CUDA;
  return rc;
}

namespace {
int decode_step(const void *q, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                int32_t *seq_lens, float scale, void *out, int B, int H, int G, int d, int Nmax, gqa_dtype_t dtype,
                void *workspace, size_t workspace_bytes, bool allocate, cudaStream_t stream) {
  if (int rc = check_attention_args(q, k_cache, v_cache, seq_lens, out, B, H, G, d, Nmax, dtype)) return rc;
  if (!k_new || !v_new) return GQA_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new)) return GQA_ERR_INVALID_ARG;
  const Plan pl = make_plan(B, H, G, d, Nmax, dtype, 0);
  if (!plan_fits(pl, B, G)) return GQA_ERR_UNSUPPORTED;
  const size_t need = workspace_for(pl, B, H, d);
  void *ws = workspace;
  if (allocate) {
    ws = nullptr;
    if (need > 0 && !ws_alloc(&ws, need, stream)) return GQA_ERR_NO_MEMORY;
  } else if (need > 0 && (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))) {
    return GQA_ERR_INVALID_ARG;
  }
  StepAppend app;
  app.k_new = k_new;
  app.v_new = v_new;
  app.k_cache = k_cache;
  app.v_cache = v_cache;
  app.seq_lens = seq_lens;
  int rc = run_attention(q, k_cache, v_cache, seq_lens, scale, out, B, H, G, d, Nmax, dtype, pl, ws, stream, app);
  if (allocate && ws && !ws_free(ws, stream) && rc == GQA_OK) rc = GQA_ERR_CUDA;
  return rc;
}
}  // namespace

int gqa_decode_step(const void *q, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                    int32_t *seq_lens, float scale, void *out, int B, int H, int G, int d, int Nmax,
                    gqa_dtype_t dtype, cudaStream_t stream) {
  return decode_step(q, k_new, v_new, k_cache, v_cache, seq_lens, scale, out, B, H, G, d, Nmax, dtype, nullptr, 0,
                     true, stream);
}

int gqa_decode_step_ws(const void *q, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                       int32_t *seq_lens, float scale, void *out, int B, int H, int G, int d, int Nmax,
                       gqa_dtype_t dtype, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
  return decode_step(q, k_new, v_new, k_cache, v_cache, seq_lens, scale, out, B, H, G, d, Nmax, dtype, workspace,
                     workspace_bytes, false, stream);
}

int gqa_decode_attention_noalloc(const void *q, const void *k_cache, const void *v_cache, const int32_t *seq_lens,
                                 float scale, void *out, int B, int H, int G, int d, int Nmax, gqa_dtype_t dtype,
                                 cudaStream_t stream) {
  if (int rc = check_attention_args(q, k_cache, v_cache, seq_lens, out, B, H, G, d, Nmax, dtype)) return rc;
  const Plan pl = make_plan(B, H, G, d, Nmax, dtype, 0);
  if (!plan_fits(pl, B, G)) return GQA_ERR_UNSUPPORTED;
  const size_t need = workspace_for(pl, B, H, d);
  if (need > GQA_NOALLOC_SCRATCH_BYTES) return GQA_ERR_SCRATCH_LIMIT;
  void *ws = nullptr;
  if (need > 0) {
    if (int rc = noalloc_scratch(&ws)) return rc;
  }
  return run_attention(q, k_cache, v_cache, seq_lens, scale, out, B, H, G, d, Nmax, dtype, pl, ws, stream);
}

namespace {
// Arguments of the several-token calls; the plan is the one for T * H query
// rows per sequence.
int check_multi_args(const void *q, const void *k, const void *v, const int32_t *sl, const void *out, int B, int T,
                     int H, int G, int d, int Nmax, gqa_dtype_t dt) {
  if (T <= 0) return GQA_ERR_INVALID_ARG;
  if (int rc = check_attention_args(q, k, v, sl, out, B, H, G, d, Nmax, dt)) return rc;
  if ((long long)T * H > (1 << 20)) return GQA_ERR_UNSUPPORTED;
  return GQA_OK;
}
}  // namespace

int gqa_decode_attention_multi_ex(const void *q, const void *k_cache, const void *v_cache, const int32_t *seq_lens,
                                  float scale, void *out, int B, int T, int H, int G, int d, int Nmax,
                                  gqa_dtype_t dtype, int split_tokens, void *workspace, size_t workspace_bytes,
                                  cudaStream_t stream) {
  if (int rc = check_multi_args(q, k_cache, v_cache, seq_lens, out, B, T, H, G, d, Nmax, dtype)) return rc;
  if (split_tokens < 0) return GQA_ERR_INVALID_ARG;
  const Plan pl = make_plan(B, T * H, G, d, Nmax, dtype, split_tokens, true);
  if (!plan_fits(pl, B, G)) return GQA_ERR_UNSUPPORTED;
  const size_t need = workspace_for(pl, B, T * H, d);
  if (need > 0 && (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
    return GQA_ERR_INVALID_ARG;
  return run_attention(q, k_cache, v_cache, seq_lens, scale, out, B, H, G, d, Nmax, dtype, pl, workspace, stream,
                       StepAppend(), T);
}

int gqa_decode_attention_multi(const void *q, const void *k_cache, const void *v_cache, const int32_t *seq_lens,
                               float scale, void *out, int B, int T, int H, int G, int d, int Nmax, gqa_dtype_t dtype,
                               cudaStream_t stream) {
  if (int rc = check_multi_args(q, k_cache, v_cache, seq_lens, out, B, T, H, G, d, Nmax, dtype)) return rc;
  const Plan pl = make_plan(B, T * H, G, d, Nmax, dtype, 0, true);
  if (!plan_fits(pl, B, G)) return GQA_ERR_UNSUPPORTED;
  const size_t need = workspace_for(pl, B, T * H, d);
  void *ws = nullptr;
  if (need > 0 && !ws_alloc(&ws, need, stream)) return GQA_ERR_NO_MEMORY;
  int rc = run_attention(q, k_cache, v_cache, seq_lens, scale, out, B, H, G, d, Nmax, dtype, pl, ws, stream,
                         StepAppend(), T);
  if (ws && !ws_free(ws, stream) && rc == GQA_OK) rc = GQA_ERR_CUDA;
  return rc;
}


size_t gqa_qkv_project_workspace_bytes(int B, int A, int H, int G, int d) {
  if (B <= 0 || A <= 0 || H <= 0 || G <= 0 || H % G != 0 || (d != 64 && d != 128) || A % kProjKT != 0) return 0;
  return proj_workspace(make_proj_plan(B, A, H, G, d));
}

int gqa_qkv_project_ws(const void *x, const void *w_q, const void *w_k, const void *w_v, void *q, void *k_new,
                       void *v_new, int B, int A, int H, int G, int d, gqa_dtype_t dtype, void *workspace,
                       size_t workspace_bytes, cudaStream_t stream) {
  if (int rc = check_proj_args(x, w_q, w_k, w_v, q, k_new, v_new, B, A, H, G, d, dtype)) return rc;
  const size_t need = proj_workspace(make_proj_plan(B, A, H, G, d));
  if (need > 0 && (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
    return GQA_ERR_INVALID_ARG;
  return run_projection(x, w_q, w_k, w_v, q, k_new, v_new, B, A, H, G, d, workspace, stream);
}

int gqa_qkv_project(const void *x, const void *w_q, const void *w_k, const void *w_v, void *q, void *k_new,
                    void *v_new, int B, int A, int H, int G, int d, gqa_dtype_t dtype, cudaStream_t stream) {
  if (int rc = check_proj_args(x, w_q, w_k, w_v, q, k_new, v_new, B, A, H, G, d, dtype)) return rc;
  const size_t need = proj_workspace(make_proj_plan(B, A, H, G, d));
  void *ws = nullptr;
  if (need > 0 && !ws_alloc(&ws, need, stream)) return GQA_ERR_NO_MEMORY;
  int rc = run_projection(x, w_q, w_k, w_v, q, k_new, v_new, B, A, H, G, d, ws, stream);
  if (ws && !ws_free(ws, stream) && rc == GQA_OK) rc = GQA_ERR_CUDA;
  return rc;
}

namespace {
int check_fp8_args(const void *q, const void *k, const void *v, const float *ks, const float *vs, const int32_t *sl,
                   const void *out, int B, int H, int G, int d, int Nmax) {
  if (!ks || !vs) return GQA_ERR_INVALID_ARG;
  if (int rc = check_attention_args(q, k, v, sl, out, B, H, G, d, Nmax, GQA_BF16)) return rc;
  if (d != 128) return GQA_ERR_UNSUPPORTED;
  return GQA_OK;
}
}  // namespace

size_t gqa_decode_workspace_bytes_fp8(int B, int H, int G, int d, int Nmax) {
  if (B <= 0 || H <= 0 || G <= 0 || Nmax <= 0 || H % G != 0 || d != 128) return 0;
  return workspace_for(make_plan(B, H, G, d, Nmax, GQA_FP8_E4M3, 0), B, H, d);
}

int gqa_decode_attention_fp8_ws(const void *q, const void *k_cache, const void *v_cache, const float *k_scale,
                                const float *v_scale, const int32_t *seq_lens, float scale, void *out, int B, int H,
                                int G, int d, int Nmax, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (int rc = check_fp8_args(q, k_cache, v_cache, k_scale, v_scale, seq_lens, out, B, H, G, d, Nmax)) return rc;
  const Plan pl = make_plan(B, H, G, d, Nmax, GQA_FP8_E4M3, 0);
  if (!plan_fits(pl, B, G)) return GQA_ERR_UNSUPPORTED;
  const size_t need = workspace_for(pl, B, H, d);
  if (need > 0 && (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
    return GQA_ERR_INVALID_ARG;
  return run_attention(q, k_cache, v_cache, seq_lens, scale, out, B, H, G, d, Nmax, GQA_FP8_E4M3, pl, workspace,
                       stream, StepAppend(), 1, k_scale, v_scale);
}

int gqa_decode_attention_fp8(const void *q, const void *k_cache, const void *v_cache, const float *k_scale,
                             const float *v_scale, const int32_t *seq_lens, float scale, void *out, int B, int H,
                             int G, int d, int Nmax, cudaStream_t stream) {
  if (int rc = check_fp8_args(q, k_cache, v_cache, k_scale, v_scale, seq_lens, out, B, H, G, d, Nmax)) return rc;
  const Plan pl = make_plan(B, H, G, d, Nmax, GQA_FP8_E4M3, 0);
  if (!plan_fits(pl, B, G)) return GQA_ERR_UNSUPPORTED;
  const size_t need = workspace_for(pl, B, H, d);
  void *ws = nullptr;
  if (need > 0 && !ws_alloc(&ws, need, stream)) return GQA_ERR_NO_MEMORY;
  int rc = run_attention(q, k_cache, v_cache, seq_lens, scale, out, B, H, G, d, Nmax, GQA_FP8_E4M3, pl, ws, stream,
                         StepAppend(), 1, k_scale, v_scale);
  if (ws && !ws_free(ws, stream) && rc == GQA_OK) rc = GQA_ERR_CUDA;
  return rc;
}

int kv_append_fp8(const void *k_new, const void *v_new, void *k_cache, void *v_cache, const float *k_scale,
                  const float *v_scale, int32_t *seq_lens, int B, int G, int d, int Nmax, cudaStream_t stream) {
  if (!k_new || !v_new || !k_cache || !v_cache || !k_scale || !v_scale || !seq_lens) return GQA_ERR_INVALID_ARG;
  if (B <= 0 || G <= 0 || d <= 0 || Nmax <= 0) return GQA_ERR_INVALID_ARG;
  if (d % 16 != 0) return GQA_ERR_UNSUPPORTED;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return GQA_ERR_INVALID_ARG;
  if (launch_pdl(gqa_kv_append_fp8_kernel, dim3(B), dim3(256), 0, stream,
                 reinterpret_cast<const __nv_bfloat16 *>(k_new), reinterpret_cast<const __nv_bfloat16 *>(v_new),
                 reinterpret_cast<uint8_t *>(k_cache), reinterpret_cast<uint8_t *>(v_cache), k_scale, v_scale,
                 seq_lens, G, Nmax, d) != cudaSuccess) {
    cudaGetLastError();
    return GQA_ERR_CUDA;
  }
  return GQA_OK;
}

int kv_append(const void *k_new, const void *v_new, void *k_cache, void *v_cache, int32_t *seq_lens, int B, int G,
              int d, int Nmax, gqa_dtype_t dtype, cudaStream_t stream) {
  if (!k_new || !v_new || !k_cache || !v_cache || !seq_lens) return GQA_ERR_INVALID_ARG;
  if (B <= 0 || G <= 0 || d <= 0 || Nmax <= 0) return GQA_ERR_INVALID_ARG;
  if (dtype != GQA_F32 && dtype != GQA_BF16) return GQA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return GQA_ERR_UNSUPPORTED;
  if (B > 2147483647) return GQA_ERR_UNSUPPORTED;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return GQA_ERR_INVALID_ARG;
  const int chunks = d * (dtype == GQA_BF16 ? 2 : 4) / 16;
  if (launch_pdl(gqa_kv_append_kernel, dim3(B), dim3(256), 0, stream, reinterpret_cast<const uint4 *>(k_new),
                 reinterpret_cast<const uint4 *>(v_new), reinterpret_cast<uint4 *>(k_cache),
                 reinterpret_cast<uint4 *>(v_cache), seq_lens, G, Nmax, chunks) != cudaSuccess) {
    cudaGetLastError();
    return GQA_ERR_CUDA;
  }
  return GQA_OK;
}

int mha_to_gqa_meanpool(const void *w, void *w_out, int H, int G, int d, int D, gqa_dtype_t dtype,
                        cudaStream_t stream) {
  if (!w || !w_out) return GQA_ERR_INVALID_ARG;
  if (H <= 0 || G <= 0 || d <= 0 || D <= 0 || H % G != 0) return GQA_ERR_INVALID_ARG;
  if (dtype != GQA_F32 && dtype != GQA_BF16) return GQA_ERR_INVALID_ARG;
  const long long per_head = (long long)d * D;
  const long long total = per_head * G;
  const int blocks = (int)std::min<long long>((total + 255) / 256, 148LL * 16);
  if (dtype == GQA_BF16)
    gqa_meanpool_kernel<__nv_bfloat16><<<blocks, 256, 0, stream>>>(
        reinterpret_cast<const __nv_bfloat16 *>(w), reinterpret_cast<__nv_bfloat16 *>(w_out), G, H / G, per_head);
  else
    gqa_meanpool_kernel<float><<<blocks, 256, 0, stream>>>(reinterpret_cast<const float *>(w),
                                                           reinterpret_cast<float *>(w_out), G, H / G, per_head);
  if (cudaPeekAtLastError() != cudaSuccess) {
    cudaGetLastError();
    return GQA_ERR_CUDA;
  }
  return GQA_OK;
}

int gqa_get_device_error(int32_t *host_err, cudaStream_t stream) {
  if (!host_err) return GQA_ERR_INVALID_ARG;
  int v = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_device_error, sizeof(int), 0, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return GQA_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbolAsync(g_device_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return GQA_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return GQA_ERR_CUDA;
  *host_err = v;
  return GQA_OK;
}

const char *gqa_status_string(int status) {
  switch (status) {
    case GQA_OK: return "ok";
    case GQA_ERR_INVALID_ARG: return "invalid argument";
    case GQA_ERR_UNSUPPORTED: return "unsupported shape";
    case GQA_ERR_CUDA: return "CUDA error";
    case GQA_ERR_NO_MEMORY: return "out of device memory";
    case GQA_ERR_SCRATCH_LIMIT: return "shape needs more split scratch than the fixed no-allocation buffer holds";
    default: return "unknown status";
  }
}

}  // extern "C"
