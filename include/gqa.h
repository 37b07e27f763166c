/*
 * gqa.h — C ABI of libgqa.so: grouped-query decode attention over a KV cache
 * on one NVIDIA B300 (sm_103a).
 *
 * The operation (GQA paper, Ainslie et al., section 2.2; 2kiu.com MHA/MQA/GQA
 * explainer, section 3): H query heads are split into G contiguous groups of
 * n_rep = H / G heads; every head of group g attends to the one K head and the
 * one V head of that group.  G = H is multi-head attention, G = 1 multi-query
 * attention.  One autoregressive decode step (fogdragon's CSDN blog on
 * MQA/GQA, section "KV Cache") first appends the new token's k and v to the
 * cache and then, per head, takes softmax(q.K^T * scale) over the cached
 * positions and the weighted sum of V.
 *
 * Conventions shared by every call:
 *  - Ownership: the caller owns every buffer.  All tensor pointers are DEVICE
 *    pointers to contiguous row-major data in the layouts stated per call;
 *    the library keeps no pointer after a call returns.
 *  - Element types: q, k_cache, v_cache, out (and k_new, v_new) share one
 *    gqa_dtype_t.  Lengths are int32.
 *  - Asynchrony: every call only enqueues work on `stream` and returns a host
 *    status without synchronising (except gqa_get_device_error).
 *  - Host-checked errors: bad arguments are rejected before any launch and
 *    return a negative gqa_status_t; nothing is enqueued then.
 *  - Device-detected errors: lengths outside their valid range are clamped
 *    (see each call), never trap, and set a bit in a per-device error word
 *    that gqa_get_device_error reads.  The kernels contain no unbounded wait:
 *    a pipeline wait that exceeds about one second sets GQA_DEVERR_TIMEOUT and
 *    the block returns.
 *  - No C++ exception crosses this interface.
 */
#ifndef GQA_DECODE_H_
#define GQA_DECODE_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GQA_F32 = 0,  /* IEEE binary32 */
    GQA_BF16 = 1, /* bfloat16, fp32 accumulation inside the kernels */
    GQA_FP8_E4M3 = 2 /* OCP FP8 E4M3 codes: the cache of the *_fp8 entry points only */
} gqa_dtype_t;

typedef enum {
    GQA_OK = 0,
    GQA_ERR_INVALID_ARG = -1, /* null pointer, non-positive size, H % G != 0, bad dtype,
                                 misaligned pointer, workspace too small */
    GQA_ERR_UNSUPPORTED = -2, /* head dimension d not in {64, 128} */
    GQA_ERR_CUDA = -3,        /* a CUDA runtime call or launch failed */
    GQA_ERR_NO_MEMORY = -4,   /* stream-ordered workspace allocation failed */
    GQA_ERR_SCRATCH_LIMIT = -5 /* gqa_decode_attention_noalloc: the shape needs more split
                                  scratch than GQA_NOALLOC_SCRATCH_BYTES */
} gqa_status_t;

/* Bits of the device error word. */
#define GQA_DEVERR_ATTN_LEN 1   /* attention saw seq_lens[b] <= 0 or > Nmax */
#define GQA_DEVERR_APPEND_LEN 2 /* kv_append saw seq_lens[b] < 0 or >= Nmax */
#define GQA_DEVERR_TIMEOUT 4    /* a pipeline wait gave up after its time limit */
#define GQA_DEVERR_RANGE 8      /* FP8 cache, groups of 33+ heads: a query value beyond the f16
                                   range (|q| > 65504) of that path's tensor-core operands
                                   (groups of 8..32 heads take any finite query) */
#define GQA_DEVERR_BOUNDS 16    /* only in the checking build (libgqa_debug.so, compiled with
                                   GQA_DEBUG): an index outside its buffer was computed; the
                                   access was skipped.  The release library never sets it. */

/*
 * gqa_decode_attention — attention of one decode token per sequence.
 *
 *   out[b,h,:] = sum_{n < L_b} softmax_n( scale * <q[b,h,:], K[b,g,n,:]> ) * V[b,g,n,:]
 *   with g = h / (H/G) and L_b = seq_lens[b].
 *
 * Source: fogdragon's CSDN blog on MQA/GQA, section "KV Cache" (logits =
 * einsum("bhd,bhnd->bhn"), softmax(logits / sqrt(d)), einsum("bhn,bhnd->bhd"))
 * with the KV head shared by a group as in the GQA paper, section 2.2.
 *
 *   q        [B, H, d]        query of the current token
 *   k_cache  [B, G, Nmax, d]  keys;   rows n >= L_b are never read
 *   v_cache  [B, G, Nmax, d]  values; rows n >= L_b are never read
 *   seq_lens [B] int32, DEVICE memory: cached length of each sequence
 *   scale    logit scale (1/sqrt(d) for the standard step)
 *   out      [B, H, d]        result, rounded to nearest even in `dtype`
 *   d in {64, 128}; H % G == 0; pointers 16-byte aligned.
 *
 * A length L_b > Nmax is treated as Nmax and L_b <= 0 gives out[b] = 0; both
 * set GQA_DEVERR_ATTN_LEN.  The cached positions of all sequences are divided
 * evenly among a persistent grid of thread blocks (one or two per SM); a
 * sequence's KV head that falls on several blocks leaves partial softmax
 * states that the last of those blocks to finish merges by log-sum-exp.  The
 * partials and a counter per (sequence, KV head) live in a workspace taken
 * from the stream-ordered allocator (cudaMallocAsync / cudaFreeAsync on
 * `stream`).  Results are deterministic: the merge order is fixed.
 */
int gqa_decode_attention(const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *seq_lens, float scale, void *out,
                         int B, int H, int G, int d, int Nmax, gqa_dtype_t dtype,
                         cudaStream_t stream);

/*
 * Bytes of workspace gqa_decode_attention_ws needs for this shape on the
 * current device (0 when no split is ever needed).  Host-only; enqueues
 * nothing.  Returns 0 for invalid shapes as well.
 */
size_t gqa_decode_workspace_bytes(int B, int H, int G, int d, int Nmax, gqa_dtype_t dtype);

/*
 * gqa_decode_attention_ws — as gqa_decode_attention, with the split partials
 * in a caller-provided device workspace of at least
 * gqa_decode_workspace_bytes(...) bytes (256-byte aligned; its contents need
 * no initialisation).  Allocates nothing, so it can be captured in a CUDA
 * graph.  Calls that share one workspace must not overlap on the device.
 */
int gqa_decode_attention_ws(const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *seq_lens, float scale, void *out,
                            int B, int H, int G, int d, int Nmax, gqa_dtype_t dtype,
                            void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * gqa_decode_attention_ex — as gqa_decode_attention_ws, with the grid sized
 * so that each thread block gets about `split_tokens` cached positions when
 * every sequence is full (rounded up to the kernel's tile of 32..128
 * positions; 0 = the automatic one-wave grid).  For tests of the split/merge
 * path and for tuning.  split_tokens < 0 is rejected.
 * gqa_decode_workspace_bytes_ex gives the workspace that choice needs.
 */
size_t gqa_decode_workspace_bytes_ex(int B, int H, int G, int d, int Nmax, gqa_dtype_t dtype,
                                     int split_tokens);
int gqa_decode_attention_ex(const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *seq_lens, float scale, void *out,
                            int B, int H, int G, int d, int Nmax, gqa_dtype_t dtype,
                            int split_tokens, void *workspace, size_t workspace_bytes,
                            cudaStream_t stream);

/*
 * gqa_decode_step — one whole autoregressive decode step in one launch: the
 * cache concatenation of kv_append followed by gqa_decode_attention over the
 * grown cache (fogdragon's CSDN blog on MQA/GQA, section "KV Cache": K =
 * cat([K_prev, k]), V = cat([V_prev, v]), then logits / softmax / weighted
 * sum over all positions including the new one).  Same result as
 *   kv_append(k_new, v_new, k_cache, v_cache, seq_lens, ...);
 *   gqa_decode_attention(q, k_cache, v_cache, seq_lens, scale, out, ...);
 * on the same stream (bit for bit), without the second launch: the thread
 * block that loads the tile holding row L_b writes k_new/v_new there first,
 * and the last block to stop reading seq_lens advances it.
 *
 *   q [B,H,d], k_new/v_new [B,G,d], k_cache/v_cache [B,G,Nmax,d] (updated),
 *   seq_lens [B] int32 DEVICE memory (read, then L_b + 1 where appended),
 *   out [B,H,d].  Pointers 16-byte aligned; d in {64, 128}; H % G == 0.
 * A row with L_b < 0 or L_b >= Nmax gets no append (GQA_DEVERR_APPEND_LEN)
 * and attention over its clamped stored length (GQA_DEVERR_ATTN_LEN when
 * that is <= 0 or > Nmax), exactly as the two separate calls would do.
 * gqa_decode_step takes its workspace from the stream-ordered allocator;
 * gqa_decode_step_ws from the caller: gqa_decode_workspace_bytes bytes,
 * 256-byte aligned, with any contents (it is never cleared).  The blocks
 * count their arrivals on a word at the start of the workspace that carries
 * the call's own tag; a word left by another call, of any shape or kind, or
 * never written, is re-tagged before the first count, so it cannot make a
 * block believe it is the last.  The same workspace also serves
 * gqa_decode_attention_ws and calls of other shapes (each needing at most
 * its size).  Calls sharing one workspace must not overlap on the device.
 */
int gqa_decode_step(const void *q, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                    int32_t *seq_lens, float scale, void *out, int B, int H, int G, int d, int Nmax,
                    gqa_dtype_t dtype, cudaStream_t stream);
int gqa_decode_step_ws(const void *q, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                       int32_t *seq_lens, float scale, void *out, int B, int H, int G, int d, int Nmax,
                       gqa_dtype_t dtype, void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * gqa_decode_attention_noalloc — gqa_decode_attention for callers that must
 * not allocate device memory during the call.  The paper has no counterpart:
 * this is an integration entry point, not part of the method.
 *
 * Who needs it: a serving engine that has already handed all free HBM to its
 * KV-cache pool (any further cudaMalloc would fail), a plugin whose host
 * framework owns the device allocator and forbids side allocations, or a
 * decode loop that cannot afford an allocator call on every step.
 *
 * Same arguments, result and error behaviour as gqa_decode_attention.  The
 * split partials go to one fixed buffer inside the library instead of a
 * per-call workspace: a static device array of GQA_NOALLOC_SCRATCH_BYTES that
 * every device which loads the library holds until the process exits.  The
 * call itself allocates nothing: no cudaMalloc/cudaMallocAsync/cudaFree and
 * no allocating library routine.
 *  - A shape whose partials need more than GQA_NOALLOC_SCRATCH_BYTES is
 *    rejected with GQA_ERR_SCRATCH_LIMIT before anything is enqueued
 *    (gqa_decode_workspace_bytes gives the need).
 *  - The first call on a device looks up that device's address of the
 *    buffer (cudaGetSymbolAddress, once per device, with the device
 *    current).  Make that first call before any stream capture begins.
 *  - Every call on a device shares the one buffer, which keeps the previous
 *    call's contents.  Nothing in it needs to start at zero: each call
 *    writes every partial it later reads.  Calls whose kernels overlap on
 *    the GPU (other streams, other host threads) race on the buffer:
 *    order them, e.g. on one stream.
 */
#define GQA_NOALLOC_SCRATCH_BYTES (32u << 20) /* 32 MiB per device */
int gqa_decode_attention_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                 const int32_t *seq_lens, float scale, void *out,
                                 int B, int H, int G, int d, int Nmax, gqa_dtype_t dtype,
                                 cudaStream_t stream);

/*
 * gqa_decode_attention_multi — attention of T new query tokens per sequence
 * in one pass, as when a large model scores a run of T tokens proposed by a
 * smaller one (speculative sampling: GQA paper, section 4, related work).
 * The T tokens' K/V rows are already in the cache: token t sits at cached
 * position L_b - T + t and attends to the positions up to and including its
 * own,
 *
 *   out[b,t,h,:] = sum_{n < L_b-T+1+t} softmax_n( scale * <q[b,t,h,:], K[b,g,n,:]> ) * V[b,g,n,:]
 *
 * with g = h / (H/G).  A token that sees no position (L_b - T + 1 + t <= 0)
 * gets out = 0.  T = 1 is gqa_decode_attention exactly (bit for bit).
 *
 *   q   [B, T, H, d]   queries of the T tokens
 *   out [B, T, H, d]   result, rounded to nearest even in `dtype`
 *   k_cache, v_cache, seq_lens, scale, d, dtype, alignment and the length
 *   errors as for gqa_decode_attention.  T >= 1 and T * H <= 2^20.
 *
 * Each K/V tile read from HBM serves all T * (H/G) query rows of its group,
 * so the call reads the same bytes as a one-token call.
 * gqa_decode_attention_multi takes its workspace from the stream-ordered
 * allocator.  gqa_decode_attention_multi_ex takes it from the caller, with
 * the grid choice of gqa_decode_attention_ex.  Its size is
 * gqa_decode_workspace_bytes_ex(B, T * H, G, d, Nmax, dtype, split_tokens),
 * 256-byte aligned, needing no initialisation.
 */
int gqa_decode_attention_multi(const void *q, const void *k_cache, const void *v_cache,
                               const int32_t *seq_lens, float scale, void *out,
                               int B, int T, int H, int G, int d, int Nmax, gqa_dtype_t dtype,
                               cudaStream_t stream);
int gqa_decode_attention_multi_ex(const void *q, const void *k_cache, const void *v_cache,
                                  const int32_t *seq_lens, float scale, void *out,
                                  int B, int T, int H, int G, int d, int Nmax, gqa_dtype_t dtype,
                                  int split_tokens, void *workspace, size_t workspace_bytes,
                                  cudaStream_t stream);

/*
 * FP8 KV cache (GQA paper, section 4: quantizing keys and values is the
 * lever that complements GQA; it halves the bytes a decode step reads
 * again).  The caches hold OCP FP8 E4M3 codes (1 sign bit, 4 exponent bits
 * with bias 7, 3 mantissa bits; no infinities; S.1111.111 is NaN; largest
 * finite 448), one byte per element, in the [B, G, Nmax, d] layout, with one
 * fp32 scale per KV head for K and one for V: element value = code * scale.
 *
 * kv_append_fp8 — kv_append onto such a cache: code = E4M3(x / scale[g]),
 * the division in fp32 (IEEE, round to nearest) and the conversion rounding
 * to nearest even, finite values beyond 448 saturating to +-448; then
 * seq_lens[b] += 1.  k_new, v_new [B, G, d] bf16; k_scale, v_scale [G] fp32,
 * device memory.  Rows with L_b < 0 or >= Nmax are left alone
 * (GQA_DEVERR_APPEND_LEN).  The codes are bit-exact to that definition.
 *
 * gqa_decode_attention_fp8[_ws] — gqa_decode_attention over such a cache:
 * K[b,g,n,:] = code * k_scale[g], V likewise; q and out [B, H, d] bf16,
 * fp32 accumulation.  d = 128.  Workspace as for gqa_decode_attention_ws,
 * of gqa_decode_workspace_bytes_fp8 bytes.  The kernel takes up to four
 * query heads of a group per pass over the group's K/V rows: groups of
 * more than four heads re-read them once per four heads.
 */
int kv_append_fp8(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                  const float *k_scale, const float *v_scale, int32_t *seq_lens,
                  int B, int G, int d, int Nmax, cudaStream_t stream);
size_t gqa_decode_workspace_bytes_fp8(int B, int H, int G, int d, int Nmax);
int gqa_decode_attention_fp8(const void *q, const void *k_cache, const void *v_cache,
                             const float *k_scale, const float *v_scale, const int32_t *seq_lens,
                             float scale, void *out, int B, int H, int G, int d, int Nmax,
                             cudaStream_t stream);
int gqa_decode_attention_fp8_ws(const void *q, const void *k_cache, const void *v_cache,
                                const float *k_scale, const float *v_scale,
                                const int32_t *seq_lens, float scale, void *out,
                                int B, int H, int G, int d, int Nmax, void *workspace,
                                size_t workspace_bytes, cudaStream_t stream);

/*
 * gqa_qkv_project — the Q, K and V projections of the decode token, the step
 * before kv_append: every query head computes its own query with its own
 * weights, every group one shared key and one shared value with the group's
 * weights (2kiu.com explainer, section 3.2, steps 2-3; CSDN blog on MQA/GQA,
 * section "MQA 的推导": q = einsum('ba,had->bhd', x, P_q), with the head axis
 * of P_k and P_v reduced to the G KV heads).
 *
 *   q[b,h,:]     = sum_a x[b,a] * w_q[h,a,:]
 *   k_new[b,g,:] = sum_a x[b,a] * w_k[g,a,:]
 *   v_new[b,g,:] = sum_a x[b,a] * w_v[g,a,:]
 *
 *   x   [B, A]     the token's hidden vector (A = model width)
 *   w_q [H, A, d], w_k and w_v [G, A, d]  (the blog's [h, a, d] layout)
 *   q [B, H, d], k_new and v_new [B, G, d]: the inputs of kv_append /
 *   gqa_decode_step.  Accumulated in fp32, rounded to nearest even.
 * bf16 only (GQA_ERR_UNSUPPORTED for fp32); d in {64, 128}; A % 64 == 0;
 * H % G == 0; pointers 16-byte aligned; any B (batches of more than 256 rows
 * run in chunks of 256).  The weights are read from HBM once per 256 rows:
 * the call is bound by those (H + 2G) * A * d * 2 bytes.  Results are
 * deterministic (a split projection head is summed in a fixed order).
 * gqa_qkv_project takes its workspace from the stream-ordered allocator;
 * gqa_qkv_project_ws from the caller: gqa_qkv_project_workspace_bytes
 * bytes (0 = none needed, or an invalid shape), 256-byte aligned, needing
 * no initialisation.  Calls sharing a workspace must not overlap.
 */
size_t gqa_qkv_project_workspace_bytes(int B, int A, int H, int G, int d);
int gqa_qkv_project(const void *x, const void *w_q, const void *w_k, const void *w_v,
                    void *q, void *k_new, void *v_new, int B, int A, int H, int G, int d,
                    gqa_dtype_t dtype, cudaStream_t stream);
int gqa_qkv_project_ws(const void *x, const void *w_q, const void *w_k, const void *w_v,
                       void *q, void *k_new, void *v_new, int B, int A, int H, int G, int d,
                       gqa_dtype_t dtype, void *workspace, size_t workspace_bytes,
                       cudaStream_t stream);

/*
 * kv_append — the cache concatenation of one decode step (fogdragon's CSDN
 * blog, section "KV Cache": K = cat([K_prev, k]), V = cat([V_prev, v])).
 *
 *   k_cache[b,g,L_b,:] = k_new[b,g,:];  v_cache[b,g,L_b,:] = v_new[b,g,:];  seq_lens[b] = L_b + 1
 *
 *   k_new, v_new [B, G, d]; k_cache, v_cache [B, G, Nmax, d];
 *   seq_lens [B] int32 DEVICE memory, read and updated in place.
 * Rows are copied bit-exactly.  A batch with L_b < 0 or L_b >= Nmax is left
 * untouched (no write, no increment) and sets GQA_DEVERR_APPEND_LEN.
 * Calling kv_append and then gqa_decode_attention with the same seq_lens on
 * the same stream is one decode step; the new token takes part in it.
 */
int kv_append(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
              int32_t *seq_lens, int B, int G, int d, int Nmax, gqa_dtype_t dtype,
              cudaStream_t stream);

/*
 * mha_to_gqa_meanpool — checkpoint conversion of the GQA paper, section 2.1
 * and 2.2 (2kiu.com explainer, section 4.3): the key (or value) projection of
 * KV head g is the mean of the projections of the n_rep = H/G heads of
 * group g.
 *
 *   w_out[g, :, :] = (1/n_rep) * sum_{j < n_rep} w[g*n_rep + j, :, :]
 *
 *   w [H, d, D] (heads leading; d = head dim, D = model width), w_out [G, d, D].
 * Any layout with the head axis leading works: only d*D, the element count
 * per head, matters.  A bias [H, d] is pooled the same way with D = 1.
 * Accumulates in fp32; the result is rounded to `dtype`.
 */
int mha_to_gqa_meanpool(const void *w, void *w_out, int H, int G, int d, int D,
                        gqa_dtype_t dtype, cudaStream_t stream);

/*
 * gqa_set_workspace_allocator — where the calls that get their own workspace
 * (gqa_decode_attention, gqa_decode_step, gqa_decode_attention_multi,
 * gqa_decode_attention_fp8, gqa_qkv_project) take it from.  An integration
 * hook with no counterpart in the pages: by default each such call takes its
 * split scratch from the stream-ordered allocator (cudaMallocAsync, released
 * with cudaFreeAsync after its kernels are enqueued); a serving engine that
 * manages device memory itself installs its pool here.
 *   alloc(ctx, &ptr, bytes, stream): returns 0 and a device pointer (256-byte
 *     aligned) valid for work ordered after it on `stream`; anything else is
 *     a failure, and the call then returns GQA_ERR_NO_MEMORY with nothing
 *     enqueued.
 *   free_fn(ctx, ptr, stream): releases ptr once the work enqueued on `stream`
 *     so far has finished (stream-ordered, as cudaFreeAsync).
 * Both NULL restores the default; exactly one NULL is GQA_ERR_INVALID_ARG.
 * Process-wide: set it while no call is running on another thread.  The
 * _ws / _ex calls, which take the caller's workspace, never use it.
 */
typedef int (*gqa_alloc_fn)(void *ctx, void **ptr, size_t bytes, cudaStream_t stream);
typedef void (*gqa_free_fn)(void *ctx, void *ptr, cudaStream_t stream);
int gqa_set_workspace_allocator(gqa_alloc_fn alloc, gqa_free_fn free_fn, void *ctx);

/*
 * gqa_stream_read — a measurement utility with no counterpart in the pages:
 * the read-only streaming ceiling that the decode kernels' HBM rates are
 * judged against (a decode call reads its K/V bytes once and writes almost
 * nothing, so a copy, which writes every byte too, is the wrong bound).
 * Reads `bytes` bytes at `buf` (DEVICE memory, 16-byte aligned) once and
 * XORs all its 32-bit words into *sink (DEVICE word, which the caller sets
 * beforehand; the result is a checksum).
 *   mode 0: 16-byte loads from every thread (bytes % 16 == 0);
 *   mode 1: bulk asynchronous copies of 32 KB chunks into shared memory, as
 *           the K/V pipeline streams (bytes % 32768 == 0).
 * Asynchronous on `stream`; a bad argument returns GQA_ERR_INVALID_ARG with
 * nothing enqueued.
 */
int gqa_stream_read(const void *buf, size_t bytes, int mode, uint32_t *sink, cudaStream_t stream);

/*
 * gqa_wait_timeout_selftest — a check of the error path, with no counterpart
 * in the pages: launches one warp that waits, through the same time-bounded
 * waits the split kernels use, on a condition that nothing will satisfy.
 * The wait gives up after about one second, sets GQA_DEVERR_TIMEOUT in the
 * error word and returns, and the kernel ends: no fault, no trap, and the
 * context stays usable.  Read (and clear) the word with gqa_get_device_error.
 *   which = 0: the single-thread mbarrier wait (TMA producers, CUDA-core and
 *              warp-MMA consumers);
 *           1: the whole-warp wait of the tcgen05 kernel's softmax and
 *              converter warps;
 *           2: a fused step's producer waiting for its warps' signals
 *              before it counts its block.
 * Asynchronous on `stream` (about one second of device time); `which`
 * outside 0..2 returns GQA_ERR_INVALID_ARG with nothing enqueued.
 */
int gqa_wait_timeout_selftest(int which, cudaStream_t stream);

/*
 * Reads the current device's error word into *host_err and clears it.  This
 * call synchronises `stream` (it copies the word to the host on it).
 */
int gqa_get_device_error(int32_t *host_err, cudaStream_t stream);

/* Static, human-readable text of a gqa_status_t value. */
const char *gqa_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* GQA_DECODE_H_ */
