/*
 * pkv_oracle.c -- plain, slow CPU definition of paged-KV attention.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline arm use it. It shares no code with the CUDA kernels.
 *
 * What it computes (one pass, no blocking, no fusion, fp64 arithmetic):
 *
 *  1. store_kvcache  -- "vLLM 学习笔记 02：nano-vllm 源码逐段精读",
 *     layers/attention.py listing (store_kvcache_kernel and its wrapper);
 *     restated in "Nano-vLLM代码手撕笔记", section "请求执行 – run model":
 *     for every new token i whose slot s = slot_mapping[i] is not -1, the
 *     D = num_kv_heads*head_dim elements of k[i] and v[i] are copied to
 *     row s of k_cache / v_cache (row length D).
 *
 *  2. gather         -- the key/value rows of sequence b at logical position t
 *     live at physical slot block_tables[b][t / block_size] * block_size
 *     + t % block_size (same listing: flash_attn_* receive block_table and the
 *     paged k_cache/v_cache; the slot formula is the one
 *     engine/model_runner.py prepare_prefill uses to write them).
 *     In contiguous mode (no block table) they are k[cu_seqlens_k[b] + t].
 *
 *  3. attention      -- causal softmax attention. Query row i of sequence b
 *     sits at absolute position p = Lk_b - Lq_b + i (prepare_prefill sets
 *     positions = range(num_cached_tokens, end) and seqlen_k = end), and
 *     attends to keys t = 0..p. Query head h reads kv head h / (Hq/Hkv).
 *     s_t = scale * sum_j q_j k_tj;  m = max_t s_t;  w_t = exp(s_t - m);
 *     o = sum_t w_t v_t / sum_t w_t.  A row with no keys gives zeros.
 *     Decode (flash_attn_with_kvcache) is the same with one query per
 *     sequence at position context_lens[b] - 1, i.e. keys 0..ctx-1.
 *
 * Element storage: q, k, v and the caches hold 16-bit values passed as raw
 * bit patterns and widened exactly to double. Two element types are read:
 * bf16 (the pages' default model dtype) and IEEE fp16 (the experiment code in
 * "Nano-vLLM代码手撕笔记", section "目录结构概览", builds the engine with
 * dtype=torch.float16). The store copies bit patterns and has no type.
 * Results are written as double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum {
    ORACLE_OK = 0,
    ORACLE_ERR_SLOT_RANGE = -1,
    ORACLE_ERR_SLOT_DUPLICATE = -2,
    ORACLE_ERR_BLOCK_RANGE = -3,
    ORACLE_ERR_SHAPE = -4,
    ORACLE_ERR_NOMEM = -5,
};

enum { ORACLE_ELEM_BF16 = 0, ORACLE_ELEM_F16 = 1 };

/* bf16 bit pattern -> double, exact (bf16 is the top half of an fp32). */
static double bf16_to_double(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE 754 binary16 bit pattern -> double, exact. Fields: sign (bit 15),
 * exponent (bits 10-14, bias 15), fraction (bits 0-9). Exponent 0 encodes
 * zero and subnormals, fraction * 2^-24; exponent 31 encodes infinity
 * (fraction 0) or NaN; otherwise the value is (1024 + fraction) * 2^(e-25). */
static double f16_to_double(uint16_t bits) {
    int sign = (bits >> 15) & 1;
    int e = (bits >> 10) & 0x1f;
    int f = bits & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return sign ? -v : v;
}

static double elem_to_double(uint16_t bits, int elem) {
    return elem == ORACLE_ELEM_F16 ? f16_to_double(bits) : bf16_to_double(bits);
}

/* Exported for the pins: widen n bit patterns of the given element type. */
int oracle_elements_to_double(const uint16_t *bits, int64_t n, int elem, double *out) {
    if (elem != ORACLE_ELEM_BF16 && elem != ORACLE_ELEM_F16) return -4;
    for (int64_t i = 0; i < n; i++) out[i] = elem_to_double(bits[i], elem);
    return 0;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- 1. store ---------------------------------------------------------- */

int oracle_store_kvcache(const uint16_t *k, int64_t k_row_stride,
                         const uint16_t *v, int64_t v_row_stride,
                         uint16_t *k_cache, uint16_t *v_cache,
                         const int32_t *slot_mapping, int64_t num_tokens,
                         int64_t D, int64_t num_slots) {
    /* Reject what the pages never produce: a slot outside the pool, or two
     * tokens writing the same slot (the result would depend on order). */
    for (int64_t i = 0; i < num_tokens; i++) {
        int64_t s = slot_mapping[i];
        if (s == -1) continue;
        if (s < 0 || s >= num_slots) return ORACLE_ERR_SLOT_RANGE;
        for (int64_t j = 0; j < i; j++)
            if (slot_mapping[j] == s) return ORACLE_ERR_SLOT_DUPLICATE;
    }
    for (int64_t i = 0; i < num_tokens; i++) {
        int64_t slot = slot_mapping[i];
        if (slot == -1) continue;
        for (int64_t e = 0; e < D; e++) {
            k_cache[slot * D + e] = k[i * k_row_stride + e];
            v_cache[slot * D + e] = v[i * v_row_stride + e];
        }
    }
    return ORACLE_OK;
}

/* ---- 3. one query row against n_keys gathered key/value rows ------------ */

/* krows[t] / vrows[t] point at the head_dim elements of key/value t. */
static int attend_one_row(const double *q, const uint16_t *const *krows,
                          const uint16_t *const *vrows, int64_t n_keys,
                          int64_t head_dim, double scale, int elem, double *out) {
    for (int64_t j = 0; j < head_dim; j++) out[j] = 0.0;
    if (n_keys <= 0) return ORACLE_OK;
    double *s = (double *)malloc(sizeof(double) * (size_t)n_keys);
    if (!s) return ORACLE_ERR_NOMEM;
    for (int64_t t = 0; t < n_keys; t++) {
        double dot = 0.0;
        for (int64_t j = 0; j < head_dim; j++) dot += q[j] * elem_to_double(krows[t][j], elem);
        s[t] = scale * dot;
    }
    double m = s[0];
    for (int64_t t = 1; t < n_keys; t++)
        if (s[t] > m) m = s[t];
    double denom = 0.0;
    for (int64_t t = 0; t < n_keys; t++) {
        double w = exp(s[t] - m);
        denom += w;
        for (int64_t j = 0; j < head_dim; j++) out[j] += w * elem_to_double(vrows[t][j], elem);
    }
    for (int64_t j = 0; j < head_dim; j++) out[j] = out[j] / denom;
    free(s);
    return ORACLE_OK;
}

/* ---- 2. gather the key/value rows of one sequence ----------------------- */

/* Fills krows/vrows[0..n_keys) for sequence b and kv head hk. Paged mode when
 * block_tables != NULL, contiguous mode otherwise. */
static int gather_rows(int64_t b, int64_t hk, int64_t n_keys,
                       const uint16_t *k, const uint16_t *v, int64_t kv_row_stride,
                       const int32_t *cu_seqlens_k,
                       const uint16_t *k_cache, const uint16_t *v_cache, int64_t num_blocks,
                       const int32_t *block_tables, int64_t bt_stride,
                       int64_t Hkv, int64_t head_dim, int64_t block_size,
                       const uint16_t **krows, const uint16_t **vrows) {
    int64_t D = Hkv * head_dim;
    for (int64_t t = 0; t < n_keys; t++) {
        if (block_tables) {
            int64_t block = block_tables[b * bt_stride + t / block_size];
            if (block < 0 || block >= num_blocks) return ORACLE_ERR_BLOCK_RANGE;
            int64_t slot = block * block_size + t % block_size;
            krows[t] = k_cache + slot * D + hk * head_dim;
            vrows[t] = v_cache + slot * D + hk * head_dim;
        } else {
            int64_t row = (int64_t)cu_seqlens_k[b] + t;
            krows[t] = k + row * kv_row_stride + hk * head_dim;
            vrows[t] = v + row * kv_row_stride + hk * head_dim;
        }
    }
    return ORACLE_OK;
}

/* ---- prefill: flash_attn_varlen_func(q, k, v, cu_seqlens_q/k, causal,
 *      block_table) as called in layers/attention.py ------------------------
 *
 * q: [total_q, Hq, head_dim] with row stride q_row_stride (elements).
 * Paged mode: block_tables != NULL, keys from k_cache/v_cache
 *             [num_blocks, block_size, Hkv, head_dim].
 * Contiguous mode: block_tables == NULL, keys from k/v [total_k, Hkv, head_dim]
 *             with row stride kv_row_stride.
 * rows: optional list of n_rows (token, head) pairs to compute; when NULL,
 *       every (token, head) is computed and out is [total_q, Hq, head_dim].
 *       Otherwise out is [n_rows, head_dim].
 * elem: ORACLE_ELEM_BF16 or ORACLE_ELEM_F16, the type of q, k, v and caches.
 */
int oracle_prefill_varlen(const uint16_t *q, int64_t q_row_stride,
                          const uint16_t *k, const uint16_t *v, int64_t kv_row_stride,
                          const uint16_t *k_cache, const uint16_t *v_cache, int64_t num_blocks,
                          const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                          const int32_t *block_tables, int64_t bt_stride,
                          int64_t num_seqs, int64_t Hq, int64_t Hkv, int64_t head_dim,
                          int64_t block_size, double scale,
                          const int64_t *rows, int64_t n_rows, int elem, double *out) {
    if (elem != ORACLE_ELEM_BF16 && elem != ORACLE_ELEM_F16) return ORACLE_ERR_SHAPE;
    if (Hkv <= 0 || Hq % Hkv != 0 || head_dim <= 0 || block_size <= 0) return ORACLE_ERR_SHAPE;
    int64_t group = Hq / Hkv;
    int64_t total_q = cu_seqlens_q[num_seqs];
    int64_t n_items = rows ? n_rows : total_q * Hq;
    int status = ORACLE_OK;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t it = 0; it < n_items; it++) {
        int64_t token = rows ? rows[2 * it] : it / Hq;
        int64_t h = rows ? rows[2 * it + 1] : it % Hq;
        double *o = out + it * head_dim;
        if (token < 0 || token >= total_q || h < 0 || h >= Hq) {
#pragma omp atomic write
            status = ORACLE_ERR_SHAPE;
            continue;
        }
        /* which sequence owns this packed query row */
        int64_t b = 0;
        while (!(cu_seqlens_q[b] <= token && token < cu_seqlens_q[b + 1])) b++;
        int64_t Lq = cu_seqlens_q[b + 1] - cu_seqlens_q[b];
        int64_t Lk = cu_seqlens_k[b + 1] - cu_seqlens_k[b];
        int64_t i = token - cu_seqlens_q[b];
        int64_t p = Lk - Lq + i;           /* absolute position of this query */
        int64_t n_keys = p + 1;            /* causal: keys 0..p */
        if (n_keys > Lk) n_keys = Lk;
        if (n_keys < 0) n_keys = 0;
        int64_t hk = h / group;

        double *qd = (double *)malloc(sizeof(double) * (size_t)head_dim);
        const uint16_t **krows = (const uint16_t **)malloc(sizeof(void *) * (size_t)(n_keys + 1));
        const uint16_t **vrows = (const uint16_t **)malloc(sizeof(void *) * (size_t)(n_keys + 1));
        int st = ORACLE_OK;
        if (!qd || !krows || !vrows) st = ORACLE_ERR_NOMEM;
        if (st == ORACLE_OK) {
            for (int64_t j = 0; j < head_dim; j++)
                qd[j] = elem_to_double(q[token * q_row_stride + h * head_dim + j], elem);
            st = gather_rows(b, hk, n_keys, k, v, kv_row_stride, cu_seqlens_k,
                             k_cache, v_cache, num_blocks, block_tables, bt_stride,
                             Hkv, head_dim, block_size, krows, vrows);
        }
        if (st == ORACLE_OK) st = attend_one_row(qd, krows, vrows, n_keys, head_dim, scale, elem, o);
        free(qd);
        free(krows);
        free(vrows);
        if (st != ORACLE_OK) {
#pragma omp atomic write
            status = st;
        }
    }
    return status;
}

/* ---- decode: flash_attn_with_kvcache(q.unsqueeze(1), k_cache, v_cache,
 *      cache_seqlens=context_lens, block_table, causal) ----------------------
 *
 * q: [num_seqs, Hq, head_dim] contiguous. One query per sequence; it attends
 * to keys 0..context_lens[b]-1 (context_lens counts the token just stored,
 * engine/model_runner.py prepare_decode appends len(seq)).
 * seqs: optional subset of n_seqs sequence indices; out is
 * [n_seqs or num_seqs, Hq, head_dim]. elem as for prefill.
 */
int oracle_decode(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                  int64_t num_blocks, const int32_t *block_tables, int64_t bt_stride,
                  const int32_t *context_lens, int64_t num_seqs, int64_t Hq, int64_t Hkv,
                  int64_t head_dim, int64_t block_size, double scale,
                  const int64_t *seqs, int64_t n_seqs, int elem, double *out) {
    if (elem != ORACLE_ELEM_BF16 && elem != ORACLE_ELEM_F16) return ORACLE_ERR_SHAPE;
    if (Hkv <= 0 || Hq % Hkv != 0 || head_dim <= 0 || block_size <= 0) return ORACLE_ERR_SHAPE;
    if (!block_tables) return ORACLE_ERR_SHAPE;
    int64_t group = Hq / Hkv;
    int64_t n_b = seqs ? n_seqs : num_seqs;
    int64_t n_items = n_b * Hq;
    int status = ORACLE_OK;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t it = 0; it < n_items; it++) {
        int64_t b = seqs ? seqs[it / Hq] : it / Hq;
        int64_t h = it % Hq;
        double *o = out + it * head_dim;
        if (b < 0 || b >= num_seqs) {
#pragma omp atomic write
            status = ORACLE_ERR_SHAPE;
            continue;
        }
        int64_t n_keys = context_lens[b];
        if (n_keys < 0) n_keys = 0;
        int64_t hk = h / group;
        double *qd = (double *)malloc(sizeof(double) * (size_t)head_dim);
        const uint16_t **krows = (const uint16_t **)malloc(sizeof(void *) * (size_t)(n_keys + 1));
        const uint16_t **vrows = (const uint16_t **)malloc(sizeof(void *) * (size_t)(n_keys + 1));
        int st = ORACLE_OK;
        if (!qd || !krows || !vrows) st = ORACLE_ERR_NOMEM;
        if (st == ORACLE_OK) {
            for (int64_t j = 0; j < head_dim; j++)
                qd[j] = elem_to_double(q[(b * Hq + h) * head_dim + j], elem);
            st = gather_rows(b, hk, n_keys, NULL, NULL, 0, NULL, k_cache, v_cache, num_blocks,
                             block_tables, bt_stride, Hkv, head_dim, block_size, krows, vrows);
        }
        if (st == ORACLE_OK) st = attend_one_row(qd, krows, vrows, n_keys, head_dim, scale, elem, o);
        free(qd);
        free(krows);
        free(vrows);
        if (st != ORACLE_OK) {
#pragma omp atomic write
            status = st;
        }
    }
    return status;
}
