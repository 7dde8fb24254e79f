/*
 * attn_oracle.c -- fp64 CPU oracle for masked attention and paged decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark load this file's library.  It shares no code
 * with the CUDA library and is written to be checked by eye, not to be fast:
 * every score row is materialised in full, exactly as the definition reads.
 *
 * Definitions followed (the pages' notation):
 *  - Masked scaled-dot-product attention, "MultiheadAttention fast path used
 *    18 GB of VRAM" (TL;DR and the SDPA replacement section): padding keys
 *    enter the softmax through an additive mask (0 for a real key, -inf for a
 *    padded one), and the SDPA route computes
 *        s_j   = scale * <q, k_j> + mask_j
 *        out   = sum_j softmax(s)_j * v_j.
 *  - Softmax log-sum-exp, "[sglang] ROCm aiter ring attention" (section 1,
 *    aiter.py, LSE return): lse = log(sum_j exp(s_j)), natural log, the only
 *    base under which the page's merge rule out = sum_i exp(lse_i - lse) out_i
 *    holds.
 *  - Paged KV, "LLM inference memory accounting" (section 15, paged KV cache):
 *    logical block n of a sequence lives in physical block block_table[n];
 *    token t sits in logical block t / block_size at slot t % block_size.
 *  - Decode, "KV cache in nanoVLM" (incremental computation): one query token
 *    per sequence attends over every cached key, the new one included.
 *  - Prefill, "KV cache in nanoVLM" (prefill and decode phases) and "LLM
 *    inference memory accounting" (section 20, chunked prefill): a prompt, or
 *    a chunk of it, is processed in one pass; its tokens' K/V join the cache
 *    and each of its queries attends over the cache.
 *
 * Readings where the pages are silent:
 *  - A row whose keys are all masked has no softmax; the oracle returns
 *    out = 0 and lse = -inf (never NaN), which makes such a partial carry
 *    zero weight in a merge.
 *  - The mask is added after scaling and is not scaled itself.
 *
 * Inputs are float32 or bfloat16 (raw 16-bit patterns); every element is
 * widened exactly to double before any arithmetic.  All arithmetic is fp64.
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

/* Exact widening of one stored element to double. */
static double widen(const void *base, int dtype, int64_t idx) {
    if (dtype == ORACLE_F32) {
        return (double)((const float *)base)[idx];
    } else {
        uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * One attention row over a materialised score vector.
 *   qrow(d)      = query element d
 *   key(j, d)    = key j element d;  val(j, d) likewise
 * The callers below supply those through index arithmetic on strided input.
 * s[] is caller scratch of length n_keys.
 */
static void attend_row(int64_t n_keys, int64_t D, double scale,
                       const double *q, /* [D] */
                       const void *k, const void *v, int kv_dtype,
                       const int64_t *key_index, /* element offset of key j row start */
                       const int64_t *val_index,
                       const float *mask, /* [n_keys] additive, or NULL */
                       double *s, double *out, double *lse) {
    for (int64_t j = 0; j < n_keys; ++j) {
        double dot = 0.0;
        for (int64_t d = 0; d < D; ++d)
            dot += q[d] * widen(k, kv_dtype, key_index[j] + d);
        s[j] = scale * dot + (mask ? (double)mask[j] : 0.0);
    }
    double m = -INFINITY;
    for (int64_t j = 0; j < n_keys; ++j)
        if (s[j] > m) m = s[j];
    for (int64_t d = 0; d < D; ++d) out[d] = 0.0;
    if (m == -INFINITY) { /* every key masked (or no keys at all) */
        *lse = -INFINITY;
        return;
    }
    double l = 0.0;
    for (int64_t j = 0; j < n_keys; ++j) {
        double e = (s[j] == -INFINITY) ? 0.0 : exp(s[j] - m);
        s[j] = e;
        l += e;
    }
    for (int64_t j = 0; j < n_keys; ++j) {
        if (s[j] == 0.0) continue;
        for (int64_t d = 0; d < D; ++d)
            out[d] += s[j] * widen(v, kv_dtype, val_index[j] + d);
    }
    for (int64_t d = 0; d < D; ++d) out[d] /= l;
    *lse = m + log(l);
}

/*
 * Masked attention over strided [B, H, P, D] tensors (element strides).
 * Query head h reads KV head h / (Hq / Hkv).
 * rows: flat query-row ids r = (b * Hq + h) * Pq + i to compute, or NULL for
 * all B*Hq*Pq rows in that order.  out: [n_rows, D] fp64, lse: [n_rows].
 * Returns 0, or -1 on bad arguments.
 */
int oracle_attn(int64_t B, int64_t Hq, int64_t Hkv, int64_t Pq, int64_t Pk, int64_t D,
                const void *q, int q_dtype, const int64_t *q_st,
                const void *k, int k_dtype, const int64_t *k_st,
                const void *v, int v_dtype, const int64_t *v_st,
                const float *mask, int64_t mask_stride_b, double scale,
                const int64_t *rows, int64_t n_rows, double *out, double *lse) {
    if (Hkv <= 0 || Hq % Hkv != 0 || k_dtype != v_dtype) return -1;
    if (rows == NULL) n_rows = B * Hq * Pq;
    const int64_t group = Hq / Hkv;
    int bad = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Pk > 0 ? Pk : 1));
        double *qv = (double *)malloc(sizeof(double) * (size_t)D);
        int64_t *ki = (int64_t *)malloc(sizeof(int64_t) * (size_t)(Pk > 0 ? Pk : 1));
        int64_t *vi = (int64_t *)malloc(sizeof(int64_t) * (size_t)(Pk > 0 ? Pk : 1));
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < n_rows; ++r) {
            int64_t flat = rows ? rows[r] : r;
            if (flat < 0 || flat >= B * Hq * Pq) { bad = 1; continue; }
            int64_t i = flat % Pq, h = (flat / Pq) % Hq, b = flat / (Pq * Hq);
            int64_t g = h / group;
            for (int64_t d = 0; d < D; ++d)
                qv[d] = widen(q, q_dtype, b * q_st[0] + h * q_st[1] + i * q_st[2] + d * q_st[3]);
            for (int64_t j = 0; j < Pk; ++j) {
                ki[j] = b * k_st[0] + g * k_st[1] + j * k_st[2];
                vi[j] = b * v_st[0] + g * v_st[1] + j * v_st[2];
            }
            /* keys and values walk d with unit step: their last dim is contiguous */
            attend_row(Pk, D, scale, qv, k, v, k_dtype, ki, vi,
                       mask ? mask + b * mask_stride_b : NULL, s, out + r * D, lse + r);
        }
        free(s); free(qv); free(ki); free(vi);
    }
    return bad ? -1 : 0;
}

/*
 * Paged GQA decode: for every sequence b and query head h, attend q[b, h]
 * over the first ctx_lens[b] tokens of KV head h / (Hq / Hkv), where token t
 * is read from physical block block_table[b * bt_stride + t / block_size],
 * slot t % block_size of a cache laid out [num_blocks, Hkv, block_size, D]
 * (contiguous).  q: [B, Hq, D] contiguous.  out: [B, Hq, D], lse: [B, Hq].
 * Returns 0, or -1 if a table entry points outside the cache or a context
 * needs more blocks than max_blocks.
 */
int oracle_paged_decode(int64_t B, int64_t Hq, int64_t Hkv, int64_t D, int64_t block_size,
                        int64_t num_blocks, const void *q, int q_dtype,
                        const void *k_cache, const void *v_cache, int kv_dtype,
                        const int32_t *block_table, int64_t bt_stride, int64_t max_blocks,
                        const int32_t *ctx_lens, double scale, double *out, double *lse) {
    if (Hkv <= 0 || Hq % Hkv != 0) return -1;
    const int64_t group = Hq / Hkv;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < B * Hq; ++bh) {
        int64_t b = bh / Hq, h = bh % Hq, g = h / group;
        int64_t L = ctx_lens[b];
        if (L < 0 || (L + block_size - 1) / block_size > max_blocks) { bad = 1; continue; }
        double *s = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        double *qv = (double *)malloc(sizeof(double) * (size_t)D);
        int64_t *ki = (int64_t *)malloc(sizeof(int64_t) * (size_t)(L > 0 ? L : 1));
        int ok = 1;
        /* the contiguous K/V of this (sequence, KV head), found by walking the table */
        for (int64_t t = 0; t < L; ++t) {
            int64_t blk = block_table[b * bt_stride + t / block_size];
            if (blk < 0 || blk >= num_blocks) { ok = 0; break; }
            ki[t] = ((blk * Hkv + g) * block_size + t % block_size) * D;
        }
        if (!ok) {
            bad = 1;
        } else {
            for (int64_t d = 0; d < D; ++d) qv[d] = widen(q, q_dtype, (b * Hq + h) * D + d);
            attend_row(L, D, scale, qv, k_cache, v_cache, kv_dtype, ki, ki, NULL, s,
                       out + bh * D, lse + bh);
        }
        free(s); free(qv); free(ki);
    }
    return bad ? -1 : 0;
}

/*
 * Paged prefill of a chunk of T new tokens per sequence.  Sequence b already
 * held start_pos[b] tokens; token i of its chunk sits at position
 * start_pos[b] + i, and the caches passed here already contain the chunk.
 * Query i of (b, h) attends over the tokens [0, n) of KV head h / (Hq / Hkv),
 * each read through the block table like the decode above, with
 *   n = start_pos[b] + i + 1   when causal (no token after its own position)
 *   n = start_pos[b] + T       otherwise (every token of the chunk).
 * q: [B, Hq, T, D] contiguous.  out: [B, Hq, T, D], lse: [B, Hq, T].
 * Returns 0, or -1 if a table entry points outside the cache or a sequence
 * needs more blocks than max_blocks.
 */
int oracle_paged_prefill(int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t D, int64_t block_size,
                         int64_t num_blocks, const void *q, int q_dtype,
                         const void *k_cache, const void *v_cache, int kv_dtype,
                         const int32_t *block_table, int64_t bt_stride, int64_t max_blocks,
                         const int32_t *start_pos, int causal, double scale, double *out, double *lse) {
    if (Hkv <= 0 || Hq % Hkv != 0) return -1;
    const int64_t group = Hq / Hkv;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < B * Hq * T; ++r) {
        int64_t i = r % T, h = (r / T) % Hq, b = r / (T * Hq);
        int64_t g = h / group;
        int64_t start = start_pos[b];
        int64_t total = start + T;
        if (start < 0 || (total + block_size - 1) / block_size > max_blocks) { bad = 1; continue; }
        int64_t n = causal ? start + i + 1 : total;
        double *s = (double *)malloc(sizeof(double) * (size_t)n);
        double *qv = (double *)malloc(sizeof(double) * (size_t)D);
        int64_t *ki = (int64_t *)malloc(sizeof(int64_t) * (size_t)n);
        int ok = 1;
        for (int64_t t = 0; t < n; ++t) {
            int64_t blk = block_table[b * bt_stride + t / block_size];
            if (blk < 0 || blk >= num_blocks) { ok = 0; break; }
            ki[t] = ((blk * Hkv + g) * block_size + t % block_size) * D;
        }
        if (!ok) {
            bad = 1;
        } else {
            for (int64_t d = 0; d < D; ++d) qv[d] = widen(q, q_dtype, r * D + d);
            attend_row(n, D, scale, qv, k_cache, v_cache, kv_dtype, ki, ki, NULL, s, out + r * D, lse + r);
        }
        free(s); free(qv); free(ki);
    }
    return bad ? -1 : 0;
}
