/*
 * CPU fp64 oracle for grouped-query decode attention over a KV cache.
 *
 * TEST INFRASTRUCTURE.  This file is the checker, not the product: only the
 * test suite, the package entry point's smoke check and the bench's CPU
 * baseline may load or call it.  It shares no code, header or constant with
 * the CUDA library; it is written from the definitions on the source pages.
 *
 * Every value is read exactly from its stored type (bf16 or fp32) and all
 * arithmetic is in fp64.  Nothing is blocked, fused or reordered beyond the
 * definition: per (batch, query head) the logits over the cached positions,
 * the max-subtracted softmax, then the weighted sum of V.
 *
 * Sources (cited by page and section):
 *  - GQA paper (Ainslie et al., "GQA: Training Generalized Multi-Query
 *    Transformer Models from Multi-Head Checkpoints"), section 2.2: query heads
 *    split into G groups, each group sharing one key head and one value head;
 *    GQA-1 is MQA, GQA-H is MHA.  Section 2.1: K/V projection matrices of the
 *    heads of a group are mean-pooled into one.
 *  - 2kiu.com MHA/MQA/GQA explainer, section 3.1 (8 heads in 2 groups: heads
 *    1-4 share group 1, heads 5-8 share group 2, i.e. contiguous grouping) and
 *    section 4.3 (average the key and value weight matrices of each group).
 *  - fogdragon's CSDN blog on MQA/GQA, section "KV Cache": each decode step
 *    concatenates the new k, v onto the cache, then logits = q.K over the
 *    cached positions, weights = softmax(logits / sqrt(d)), out = weights.V;
 *    section "MQA 的推导" gives the shared-K/V (G = 1) form.
 *  - CSDN interview post on GQA, section 03: the key/value pair is repeated
 *    n_rep times, n_rep being the number of query heads sharing it.
 *  - GQA paper, section 4: quantization of keys and values (the FP8 cache
 *    functions; format and scale granularity are readings, stated there).
 *  - CSDN blog, section "MQA 的推导", and 2kiu.com explainer, section 3.2:
 *    the per-head Q and per-group K/V projections (oracle_qkv_project).
 *  - GQA paper, section 4: speculative sampling scores several proposed
 *    tokens in one pass (oracle_decode_attention_multi; the causal rule among
 *    the T new tokens is the plain reading of scoring a proposed run).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_F32 0
#define ORACLE_BF16 1

/* Exact widening of one stored element to fp64.  bf16 is the upper half of
 * an IEEE binary32, so shifting its 16 bits up gives the same float. */
static double load_value(const void *base, size_t idx, int dtype) {
    if (dtype == ORACLE_BF16) {
        uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return (double)((const float *)base)[idx];
}

static int clamp_len(int32_t L, int Nmax) {
    if (L < 0) return 0;
    if (L > Nmax) return Nmax;
    return (int)L;
}

/* repeat_kv: the head axis of the cache repeated n_rep = H / G times, each KV
 * head repeated in place (g0 g0 .. g0 g1 g1 ..), so that query head h reads
 * KV head h / n_rep.  Returned as the element offset of row 0 of the KV head
 * that each (b, h) reads; no cache data is copied. */
static size_t *repeat_kv_offsets(int B, int H, int G, int d, int Nmax) {
    int n_rep = H / G;
    size_t *off = (size_t *)malloc((size_t)B * H * sizeof(size_t));
    if (!off) return NULL;
    for (int b = 0; b < B; ++b)
        for (int g = 0; g < G; ++g)
            for (int r = 0; r < n_rep; ++r)
                off[(size_t)b * H + (size_t)g * n_rep + r] = ((size_t)b * G + g) * (size_t)Nmax * d;
    return off;
}

/* Softmax weights of one (b, h) over the L cached positions, in fp64. */
static void head_weights(const void *q, const void *k, size_t q_off, size_t kv_off,
                         int L, int d, double scale, int dtype, double *w) {
    double m = -INFINITY;
    for (int n = 0; n < L; ++n) {
        double dot = 0.0;
        for (int i = 0; i < d; ++i)
            dot += load_value(q, q_off + i, dtype) * load_value(k, kv_off + (size_t)n * d + i, dtype);
        w[n] = dot * scale; /* logits / sqrt(d) when scale = 1/sqrt(d) */
        if (w[n] > m) m = w[n];
    }
    double z = 0.0;
    for (int n = 0; n < L; ++n) {
        w[n] = exp(w[n] - m);
        z += w[n];
    }
    for (int n = 0; n < L; ++n) w[n] /= z;
}

/*
 * out[b,h,:] = sum_{n < L_b} softmax_n(scale * q[b,h,:].K[b,g,n,:]) * V[b,g,n,:]
 * with g = h / (H/G).  q [B,H,d], k/v [B,G,Nmax,d] in `dtype`, seq_lens [B],
 * out [B,H,d] fp64.  L_b is clamped to [0, Nmax]; L_b = 0 gives out = 0.
 * Returns 0, or -1 on bad arguments / no memory.
 */
int oracle_decode_attention(const void *q, const void *k, const void *v, const int32_t *seq_lens,
                            double scale, double *out, int B, int H, int G, int d, int Nmax,
                            int dtype, int nthreads) {
    if (B <= 0 || H <= 0 || G <= 0 || d <= 0 || Nmax <= 0 || H % G != 0) return -1;
    size_t *kv_off = repeat_kv_offsets(B, H, G, d, Nmax);
    if (!kv_off) return -1;
    int fail = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : fail)
#endif
    for (long bh = 0; bh < (long)B * H; ++bh) {
        int b = (int)(bh / H);
        int L = clamp_len(seq_lens[b], Nmax);
        double *o = out + (size_t)bh * d;
        for (int i = 0; i < d; ++i) o[i] = 0.0;
        if (L == 0) continue;
        double *w = (double *)malloc((size_t)L * sizeof(double));
        if (!w) { fail |= 1; continue; }
        head_weights(q, k, (size_t)bh * d, kv_off[bh], L, d, scale, dtype, w);
        for (int n = 0; n < L; ++n)
            for (int i = 0; i < d; ++i)
                o[i] += w[n] * load_value(v, kv_off[bh] + (size_t)n * d + i, dtype);
        free(w);
    }
    free(kv_off);
    return fail ? -1 : 0;
}

/*
 * Several new query tokens per sequence.  The GQA paper, section 4 (related
 * work), notes that speculative sampling eases the bandwidth bound by having
 * a small model propose several tokens that the large model then scores in
 * one parallel pass; that pass is this call.  q [B,T,H,d] holds the
 * queries of the last T cached positions, token t at position L_b - T + t,
 * and token t attends causally to the positions it may see,
 *   n < L_b - T + 1 + t   (clamped to [0, L_b]),
 * with the same grouped softmax as oracle_decode_attention.  A token that
 * sees no position gets out = 0.  out [B,T,H,d] fp64.
 */
int oracle_decode_attention_multi(const void *q, const void *k, const void *v, const int32_t *seq_lens,
                                  double scale, double *out, int B, int T, int H, int G, int d, int Nmax,
                                  int dtype, int nthreads) {
    if (B <= 0 || T <= 0 || H <= 0 || G <= 0 || d <= 0 || Nmax <= 0 || H % G != 0) return -1;
    size_t *kv_off = repeat_kv_offsets(B, H, G, d, Nmax);
    if (!kv_off) return -1;
    int fail = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : fail)
#endif
    for (long bth = 0; bth < (long)B * T * H; ++bth) {
        int b = (int)(bth / ((long)T * H));
        int t = (int)((bth / H) % T);
        int h = (int)(bth % H);
        int L = clamp_len(seq_lens[b], Nmax);
        int vis = L - T + 1 + t;
        if (vis < 0) vis = 0;
        if (vis > L) vis = L;
        double *o = out + (size_t)bth * d;
        for (int i = 0; i < d; ++i) o[i] = 0.0;
        if (vis == 0) continue;
        double *w = (double *)malloc((size_t)vis * sizeof(double));
        if (!w) { fail |= 1; continue; }
        size_t kvo = kv_off[(size_t)b * H + h];
        head_weights(q, k, (size_t)bth * d, kvo, vis, d, scale, dtype, w);
        for (int n = 0; n < vis; ++n)
            for (int i = 0; i < d; ++i)
                o[i] += w[n] * load_value(v, kvo + (size_t)n * d + i, dtype);
        free(w);
    }
    free(kv_off);
    return fail ? -1 : 0;
}

/* The softmax weights p_n (n < L_b) of one (b, h), written to w_out[0..L_b).
 * Returns L_b after clamping, or -1 on bad arguments. */
int oracle_softmax_weights(const void *q, const void *k, const int32_t *seq_lens, double scale,
                           int B, int H, int G, int d, int Nmax, int dtype, int b, int h,
                           double *w_out) {
    if (B <= 0 || H <= 0 || G <= 0 || H % G != 0 || b < 0 || b >= B || h < 0 || h >= H) return -1;
    size_t *kv_off = repeat_kv_offsets(B, H, G, d, Nmax);
    if (!kv_off) return -1;
    int L = clamp_len(seq_lens[b], Nmax);
    if (L > 0) head_weights(q, k, ((size_t)b * H + h) * d, kv_off[(size_t)b * H + h], L, d, scale, dtype, w_out);
    free(kv_off);
    return L;
}

/*
 * The cache concatenation of one decode step: row seq_lens[b] of every KV head
 * of batch b receives k_new[b,g,:] / v_new[b,g,:] (a byte copy), then
 * seq_lens[b] += 1.  A batch whose length is already outside [0, Nmax) is left
 * untouched.  Returns the number of such batches.
 */
int oracle_kv_append(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                     int32_t *seq_lens, int B, int G, int d, int Nmax, int elt_bytes) {
    int skipped = 0;
    size_t row = (size_t)d * elt_bytes;
    for (int b = 0; b < B; ++b) {
        int32_t L = seq_lens[b];
        if (L < 0 || L >= Nmax) { ++skipped; continue; }
        for (int g = 0; g < G; ++g) {
            size_t dst = (((size_t)b * G + g) * Nmax + (size_t)L) * row;
            size_t src = ((size_t)b * G + g) * row;
            memcpy((char *)k_cache + dst, (const char *)k_new + src, row);
            memcpy((char *)v_cache + dst, (const char *)v_new + src, row);
        }
        seq_lens[b] = L + 1;
    }
    return skipped;
}

/*
 * FP8 KV cache.  The GQA paper, section 4 (related work), names quantization
 * of keys and values as the lever complementary to GQA.  The cache then holds
 * OCP FP8 E4M3 codes ("e4m3fn": 1 sign bit, 4 exponent bits with bias 7, 3
 * mantissa bits; no infinities, S.1111.111 is NaN, the largest finite value
 * 448) and one fp32 scale per KV head for K and one for V: the stored value
 * of an element is code_value * scale[g].
 */
static double e4m3_value(uint8_t c) {
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);                 /* subnormal: m/8 * 2^(1-7) */
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* Round to nearest, ties to even, onto the E4M3 grid; finite values beyond
 * 448 saturate to +-448, NaN gives 0x7F.  A plain scan of the 127
 * non-negative finite codes (their values increase with the code). */
static uint8_t e4m3_encode(float r) {
    if (isnan(r)) return 0x7F;
    uint8_t sign = signbit(r) ? 0x80 : 0x00;
    double a = fabs((double)r);
    if (a >= 448.0) return sign | 0x7E;
    uint8_t best = 0;
    double best_err = a;
    for (int c = 1; c <= 0x7E; ++c) {
        double err = fabs(e4m3_value((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = (uint8_t)c;
            best_err = err;
        }
    }
    return sign | best;
}

void oracle_e4m3_decode_array(const uint8_t *c, double *out, long n) {
    for (long i = 0; i < n; ++i) out[i] = e4m3_value(c[i]);
}

void oracle_e4m3_encode_array(const float *r, uint8_t *out, long n) {
    for (long i = 0; i < n; ++i) out[i] = e4m3_encode(r[i]);
}

/*
 * kv_append onto an FP8 cache: code = e4m3(x / scale[g]) with the division
 * in fp32 (IEEE, round to nearest) from the stored new row x, then the same
 * placement and length rule as oracle_kv_append.  Returns rows skipped.
 */
int oracle_kv_append_fp8(const void *k_new, const void *v_new, uint8_t *k_cache, uint8_t *v_cache,
                         const float *k_scale, const float *v_scale, int32_t *seq_lens, int B, int G, int d,
                         int Nmax, int dtype) {
    int skipped = 0;
    for (int b = 0; b < B; ++b) {
        int32_t L = seq_lens[b];
        if (L < 0 || L >= Nmax) { ++skipped; continue; }
        for (int g = 0; g < G; ++g) {
            size_t src = ((size_t)b * G + g) * d;
            size_t dst = (((size_t)b * G + g) * Nmax + (size_t)L) * d;
            for (int i = 0; i < d; ++i) {
                float kx = (float)load_value(k_new, src + i, dtype);
                float vx = (float)load_value(v_new, src + i, dtype);
                k_cache[dst + i] = e4m3_encode(kx / k_scale[g]);
                v_cache[dst + i] = e4m3_encode(vx / v_scale[g]);
            }
        }
        seq_lens[b] += 1;
    }
    return skipped;
}

/*
 * Decode attention over an FP8 cache: the definition of
 * oracle_decode_attention with K[b,g,n,i] = e4m3_value(k8) * k_scale[g] and
 * V likewise (exact in fp64).  q and out as there.
 */
int oracle_decode_attention_fp8(const void *q, const uint8_t *k8, const uint8_t *v8, const float *k_scale,
                                const float *v_scale, const int32_t *seq_lens, double scale, double *out, int B,
                                int H, int G, int d, int Nmax, int dtype, int nthreads) {
    if (B <= 0 || H <= 0 || G <= 0 || d <= 0 || Nmax <= 0 || H % G != 0) return -1;
    int n_rep = H / G, fail = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : fail)
#endif
    for (long bh = 0; bh < (long)B * H; ++bh) {
        int b = (int)(bh / H), h = (int)(bh % H), g = h / n_rep;
        int L = clamp_len(seq_lens[b], Nmax);
        double *o = out + (size_t)bh * d;
        for (int i = 0; i < d; ++i) o[i] = 0.0;
        if (L == 0) continue;
        double *w = (double *)malloc((size_t)L * sizeof(double));
        if (!w) { fail |= 1; continue; }
        size_t kv = ((size_t)b * G + g) * Nmax * d;
        double wmax = -INFINITY;
        for (int n = 0; n < L; ++n) {
            double qk = 0.0;
            for (int i = 0; i < d; ++i)
                qk += load_value(q, (size_t)bh * d + i, dtype) * (e4m3_value(k8[kv + (size_t)n * d + i]) * k_scale[g]);
            w[n] = scale * qk;
            if (w[n] > wmax) wmax = w[n];
        }
        double z = 0.0;
        for (int n = 0; n < L; ++n) { w[n] = exp(w[n] - wmax); z += w[n]; }
        for (int n = 0; n < L; ++n) w[n] = w[n] / z;
        for (int n = 0; n < L; ++n)
            for (int i = 0; i < d; ++i)
                o[i] += w[n] * (e4m3_value(v8[kv + (size_t)n * d + i]) * v_scale[g]);
        free(w);
    }
    return fail ? -1 : 0;
}

/*
 * Q/K/V projections of the decode token.  CSDN blog on MQA/GQA, section
 * "MQA 的推导": q = einsum('ba,had->bhd', x, P_q) with P_q [h, a, d], and
 * the shared K/V projection loses the head axis for MQA; with G KV heads
 * (2kiu.com explainer, section 3.2, steps 2-3: every query head computes its
 * own Q with its own weights, every group one K and one V with the group's
 * weights) k = einsum('ba,gad->bgd', x, P_k), v likewise.
 * x [B, A] (A = model width), P_q [H, A, d], P_k and P_v [G, A, d];
 * q [B, H, d], k and v [B, G, d] in fp64.
 */
static void project_heads(const void *x, const void *p, double *out, int B, int A, int nh, int d, int dtype,
                          int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static)
#endif
    for (long bh = 0; bh < (long)B * nh; ++bh) {
        int b = (int)(bh / nh), h = (int)(bh % nh);
        for (int j = 0; j < d; ++j) {
            double s = 0.0;
            for (int a = 0; a < A; ++a)
                s += load_value(x, (size_t)b * A + a, dtype) *
                     load_value(p, ((size_t)h * A + a) * d + j, dtype);
            out[((size_t)b * nh + h) * d + j] = s;
        }
    }
}

int oracle_qkv_project(const void *x, const void *pq, const void *pk, const void *pv, double *q, double *k,
                       double *v, int B, int A, int H, int G, int d, int dtype, int nthreads) {
    if (B <= 0 || A <= 0 || H <= 0 || G <= 0 || d <= 0 || H % G != 0) return -1;
    project_heads(x, pq, q, B, A, H, d, dtype, nthreads);
    project_heads(x, pk, k, B, A, G, d, dtype, nthreads);
    project_heads(x, pv, v, B, A, G, d, dtype, nthreads);
    return 0;
}

/*
 * MHA -> GQA checkpoint conversion: the projection of KV head g is the mean of
 * the projections of the query heads of group g, w [H, per_head] ->
 * w_out [G, per_head] in fp64 (per_head = d * D for a [H, d, D] weight).
 */
int oracle_meanpool(const void *w, double *w_out, int H, int G, long per_head, int dtype) {
    if (H <= 0 || G <= 0 || H % G != 0 || per_head <= 0) return -1;
    int n_rep = H / G;
    for (int g = 0; g < G; ++g) {
        for (long e = 0; e < per_head; ++e) {
            double s = 0.0;
            for (int j = 0; j < n_rep; ++j)
                s += load_value(w, ((size_t)g * n_rep + j) * (size_t)per_head + (size_t)e, dtype);
            w_out[(size_t)g * per_head + e] = s / n_rep;
        }
    }
    return 0;
}
