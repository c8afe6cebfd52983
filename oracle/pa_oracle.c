/*
 * pa_oracle.c -- plain, slow, fp64 CPU oracle for grouped-query attention over a
 * block-paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and its
 * Python binding) may call, link or load this file; it exists so that the tests,
 * the smoke check and the benchmark's CPU baseline can check the CUDA results
 * against the plain definition.  It shares no code, header, table or helper with
 * the CUDA library.
 *
 * What it computes, from the pages "Qwen3-4B / 8B / 32B" (section "Architecture
 * Notes": full attention with grouped-query attention, 32 query heads over 8 KV
 * heads, head dim 128; Qwen3-32B 64 query heads, group 8; the KV cache is paged)
 * and section "Qwen3-32B Serving Load" (the KV budget of 21.4 GB = 5360 blocks,
 * which fixes 16-token blocks):
 *
 *   For query head h of sequence s at absolute position p, with group size
 *   g = num_heads / num_kv_heads and kv head kvh = h / g,
 *
 *     o = sum_{t <= p, t < L_s} softmax_t( scale * <q, K_t> ) * V_t
 *
 *   where K_t and V_t are read at pool[block_tables[s][t / bs], kvh, t % bs, :].
 *   Decode: one query per sequence at p = L_s - 1.  Chunked prefill: the chunk of
 *   C_s queries sits at positions L_s - C_s + i (i = 0..C_s-1), seq_lens counting
 *   the chunk.  The softmax is taken in two passes (maximum, then the sum of
 *   exponentials), in double precision, from the bf16 bits of the inputs.
 *
 *   Split-KV partitions: partition j of P covers logical blocks
 *   [j*ceil(nb/P), (j+1)*ceil(nb/P)) of the nb = ceil(L/bs) blocks; it yields its
 *   own normalised output O_j and log-sum-exp lse_j = m_j + ln(l_j); an empty
 *   partition has O_j = 0 and lse_j = -inf.  The merge weights partition j by
 *   exp(lse_j - max_j lse_j) and divides by the weights' sum.
 *
 * Conventions (readings where the pages are silent): kvh = h / g (consecutive
 * query heads share a kv head); inputs are post-RoPE; a sequence of length 0
 * gives o = 0; slot_mapping entries < 0 are skipped by the append.
 *
 * Every function returns 0 on success and a negative value on an invalid argument
 * (null pointer, bad shape, block id or slot outside the pool).
 *
 * Threads.  Every output row (one query head of one query token) is computed on its own,
 * start to finish, by one thread; compiled with OpenMP, the loops over rows may hand rows to
 * several threads (pa_oracle_set_threads), which changes neither the arithmetic nor its
 * order within a row, so the results are the same bits for any thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARG (-1)
#define ORACLE_ERR_RANGE (-2)
#define ORACLE_ERR_NOMEM (-3)

static int g_threads = 1;

/* Threads the row loops may use (1 without OpenMP); returns the count now in effect. */
int pa_oracle_set_threads(int32_t n) {
#ifdef _OPENMP
    g_threads = n > 0 ? n : 1;
#else
    (void)n;
    g_threads = 1;
#endif
    return g_threads;
}

/* bf16 is the upper half of an IEEE binary32: widen the bits, then the value. */
static double bf16_to_double(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

typedef struct {
    const uint16_t *k, *v;
    int32_t num_blocks, block_size, num_kv_heads, head_dim;
} pool_t;

/* Row t of kv head kvh of one sequence, translated through its block table. */
static int kv_rows(const pool_t *pool, const int32_t *bt_row, int32_t max_blocks, int32_t t, int32_t kvh,
                   const uint16_t **k_row, const uint16_t **v_row) {
    int32_t logical = t / pool->block_size;
    if (logical >= max_blocks) return ORACLE_ERR_RANGE;
    int32_t blk = bt_row[logical];
    if (blk < 0 || blk >= pool->num_blocks) return ORACLE_ERR_RANGE;
    int32_t off = t % pool->block_size;
    size_t row = ((size_t)blk * pool->num_kv_heads + kvh) * pool->block_size + off;
    *k_row = pool->k + row * pool->head_dim;
    *v_row = pool->v + row * pool->head_dim;
    return ORACLE_OK;
}

/*
 * Attention of one query row over the keys [t_begin, t_end) of one sequence.
 * Writes the normalised output (head_dim doubles) and the log-sum-exp of the
 * scaled scores.  An empty range gives o = 0 and lse = -inf.
 */
static int attend(const pool_t *pool, const int32_t *bt_row, int32_t max_blocks, int32_t kvh,
                  const uint16_t *q_row, double scale, int32_t t_begin, int32_t t_end,
                  double *o, double *lse) {
    const int32_t d = pool->head_dim;
    for (int32_t e = 0; e < d; ++e) o[e] = 0.0;
    if (t_end <= t_begin) {
        *lse = -INFINITY;
        return ORACLE_OK;
    }
    double *s = (double *)malloc(sizeof(double) * (size_t)(t_end - t_begin));
    if (!s) return ORACLE_ERR_NOMEM;

    /* pass 1: scores and their maximum */
    double m = -INFINITY;
    for (int32_t t = t_begin; t < t_end; ++t) {
        const uint16_t *k_row, *v_row;
        int rc = kv_rows(pool, bt_row, max_blocks, t, kvh, &k_row, &v_row);
        if (rc) { free(s); return rc; }
        double dot = 0.0;
        for (int32_t e = 0; e < d; ++e) dot += bf16_to_double(q_row[e]) * bf16_to_double(k_row[e]);
        s[t - t_begin] = scale * dot;
        if (s[t - t_begin] > m) m = s[t - t_begin];
    }
    /* pass 2: exponentials relative to the maximum, their sum, and the weighted V */
    double l = 0.0;
    for (int32_t t = t_begin; t < t_end; ++t) {
        const uint16_t *k_row, *v_row;
        kv_rows(pool, bt_row, max_blocks, t, kvh, &k_row, &v_row);
        double w = exp(s[t - t_begin] - m);
        l += w;
        for (int32_t e = 0; e < d; ++e) o[e] += w * bf16_to_double(v_row[e]);
    }
    for (int32_t e = 0; e < d; ++e) o[e] /= l;
    *lse = m + log(l);
    free(s);
    return ORACLE_OK;
}

static int check_pool(const pool_t *p) {
    if (!p->k || !p->v) return ORACLE_ERR_ARG;
    if (p->num_blocks < 0 || p->block_size <= 0 || p->num_kv_heads <= 0 || p->head_dim <= 0) return ORACLE_ERR_ARG;
    return ORACLE_OK;
}

/* The scatter: k_cache[slot / bs, h, slot % bs, :] = k_new[t, h, :] (and V), slot < 0 skipped. */
int pa_oracle_kv_append(uint16_t *k_cache, uint16_t *v_cache, int32_t num_blocks, int32_t block_size,
                        int32_t num_kv_heads, int32_t head_dim, const uint16_t *k_new, const uint16_t *v_new,
                        const int64_t *slot_mapping, int32_t num_tokens) {
    if (!k_cache || !v_cache || num_tokens < 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
        return ORACLE_ERR_ARG;
    if (num_tokens > 0 && (!k_new || !v_new || !slot_mapping)) return ORACLE_ERR_ARG;
    for (int32_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= (int64_t)num_blocks * block_size) return ORACLE_ERR_RANGE;
        int64_t blk = slot / block_size, off = slot % block_size;
        for (int32_t h = 0; h < num_kv_heads; ++h) {
            size_t dst = (((size_t)blk * num_kv_heads + h) * block_size + off) * head_dim;
            size_t src = ((size_t)t * num_kv_heads + h) * head_dim;
            for (int32_t e = 0; e < head_dim; ++e) {
                k_cache[dst + e] = k_new[src + e];
                v_cache[dst + e] = v_new[src + e];
            }
        }
    }
    return ORACLE_OK;
}

/* Decode: out[b, h, :] (doubles) for one query per sequence, q = [B, Hq, D]. */
int pa_oracle_decode(const uint16_t *k_cache, const uint16_t *v_cache, int32_t num_blocks, int32_t block_size,
                     int32_t num_kv_heads, int32_t head_dim, const uint16_t *q, const int32_t *block_tables,
                     int32_t max_blocks, const int32_t *seq_lens, int32_t batch, int32_t num_heads, double scale,
                     double *out) {
    pool_t pool = {k_cache, v_cache, num_blocks, block_size, num_kv_heads, head_dim};
    if (check_pool(&pool) || !q || !block_tables || !seq_lens || !out || batch < 0 || num_heads <= 0 ||
        num_heads % num_kv_heads)
        return ORACLE_ERR_ARG;
    const int32_t g = num_heads / num_kv_heads;
    for (int32_t b = 0; b < batch; ++b)
        if (seq_lens[b] < 0 || seq_lens[b] > max_blocks * block_size) return ORACLE_ERR_ARG;
    const long long rows = (long long)batch * num_heads;
    int err = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1) num_threads(g_threads) reduction(min : err)
    for (long long row = 0; row < rows; ++row) {
        const int32_t b = (int32_t)(row / num_heads), h = (int32_t)(row % num_heads);
        double lse;
        int rc = attend(&pool, block_tables + (size_t)b * max_blocks, max_blocks, h / g,
                        q + (size_t)row * head_dim, scale, 0, seq_lens[b], out + (size_t)row * head_dim, &lse);
        if (rc < err) err = rc;
    }
    return err;
}

/* Split-KV partitions: o_part [B, Hq, P, D] normalised per partition, lse_part [B, Hq, P]. */
int pa_oracle_decode_partitions(const uint16_t *k_cache, const uint16_t *v_cache, int32_t num_blocks,
                                int32_t block_size, int32_t num_kv_heads, int32_t head_dim, const uint16_t *q,
                                const int32_t *block_tables, int32_t max_blocks, const int32_t *seq_lens,
                                int32_t batch, int32_t num_heads, double scale, int32_t num_partitions,
                                double *o_part, double *lse_part) {
    pool_t pool = {k_cache, v_cache, num_blocks, block_size, num_kv_heads, head_dim};
    if (check_pool(&pool) || !q || !block_tables || !seq_lens || !o_part || !lse_part || batch < 0 ||
        num_heads <= 0 || num_heads % num_kv_heads || num_partitions < 1)
        return ORACLE_ERR_ARG;
    const int32_t g = num_heads / num_kv_heads;
    for (int32_t b = 0; b < batch; ++b)
        if (seq_lens[b] < 0 || seq_lens[b] > max_blocks * block_size) return ORACLE_ERR_ARG;
    const long long rows = (long long)batch * num_heads;
    int err = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1) num_threads(g_threads) reduction(min : err)
    for (long long row = 0; row < rows; ++row) {
        const int32_t b = (int32_t)(row / num_heads), h = (int32_t)(row % num_heads);
        const int32_t L = seq_lens[b];
        const int32_t nb = (L + block_size - 1) / block_size;
        const int32_t per = (nb + num_partitions - 1) / num_partitions;
        for (int32_t j = 0; j < num_partitions; ++j) {
            int32_t t0 = j * per * block_size;
            int32_t t1 = (j + 1) * per * block_size;
            if (t1 > L) t1 = L;
            size_t pr = (size_t)row * num_partitions + j;
            int rc = attend(&pool, block_tables + (size_t)b * max_blocks, max_blocks, h / g,
                            q + (size_t)row * head_dim, scale, t0, t1, o_part + pr * head_dim, lse_part + pr);
            if (rc < err) err = rc;
        }
    }
    return err;
}

/* Log-sum-exp merge of P partitions into out [B, Hq, D]. */
int pa_oracle_combine(const double *o_part, const double *lse_part, int32_t batch, int32_t num_heads,
                      int32_t head_dim, int32_t num_partitions, double *out) {
    if (!o_part || !lse_part || !out || batch < 0 || num_heads <= 0 || head_dim <= 0 || num_partitions < 1)
        return ORACLE_ERR_ARG;
    for (int32_t r = 0; r < batch * num_heads; ++r) {
        const double *lse = lse_part + (size_t)r * num_partitions;
        const double *op = o_part + (size_t)r * num_partitions * head_dim;
        double *o = out + (size_t)r * head_dim;
        double mx = -INFINITY;
        for (int32_t j = 0; j < num_partitions; ++j)
            if (lse[j] > mx) mx = lse[j];
        for (int32_t e = 0; e < head_dim; ++e) o[e] = 0.0;
        if (mx == -INFINITY) continue; /* every partition empty: zero output */
        double wsum = 0.0;
        for (int32_t j = 0; j < num_partitions; ++j) {
            double w = exp(lse[j] - mx);
            wsum += w;
            for (int32_t e = 0; e < head_dim; ++e) o[e] += w * op[(size_t)j * head_dim + e];
        }
        for (int32_t e = 0; e < head_dim; ++e) o[e] /= wsum;
    }
    return ORACLE_OK;
}

/*
 * Chunked prefill, one (token, head) row at a time.  q = [sum C, Hq, D] packed by
 * cu_q_lens [B+1]; seq_lens counts each chunk.  Query token i of sequence s sits at
 * position L_s - C_s + i and attends causally to keys 0 .. that position.
 * rows == NULL computes every row into out [sum C, Hq, D]; otherwise only the
 * nrows listed (row_tokens[r], row_heads[r]) pairs, into out [nrows, D].
 */
int pa_oracle_prefill_rows(const uint16_t *k_cache, const uint16_t *v_cache, int32_t num_blocks,
                           int32_t block_size, int32_t num_kv_heads, int32_t head_dim, const uint16_t *q,
                           const int32_t *cu_q_lens, const int32_t *block_tables, int32_t max_blocks,
                           const int32_t *seq_lens, int32_t batch, int32_t num_heads, double scale,
                           const int32_t *row_tokens, const int32_t *row_heads, int32_t nrows, double *out) {
    pool_t pool = {k_cache, v_cache, num_blocks, block_size, num_kv_heads, head_dim};
    if (check_pool(&pool) || !q || !cu_q_lens || !block_tables || !seq_lens || !out || batch < 0 ||
        num_heads <= 0 || num_heads % num_kv_heads || (row_tokens && (!row_heads || nrows < 0)))
        return ORACLE_ERR_ARG;
    const int32_t g = num_heads / num_kv_heads;
    const int32_t total = cu_q_lens[batch];
    const int32_t n = row_tokens ? nrows : total * num_heads;
    int err = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1) num_threads(g_threads) reduction(min : err)
    for (int32_t r = 0; r < n; ++r) {
        int32_t tok = row_tokens ? row_tokens[r] : r / num_heads;
        int32_t h = row_tokens ? row_heads[r] : r % num_heads;
        if (tok < 0 || tok >= total || h < 0 || h >= num_heads) {
            err = ORACLE_ERR_ARG;
            continue;
        }
        int32_t s = 0;
        while (!(cu_q_lens[s] <= tok && tok < cu_q_lens[s + 1])) ++s;
        const int32_t L = seq_lens[s];
        const int32_t C = cu_q_lens[s + 1] - cu_q_lens[s];
        if (L < C || L > max_blocks * block_size) {
            err = ORACLE_ERR_ARG;
            continue;
        }
        const int32_t pos = L - C + (tok - cu_q_lens[s]);
        double lse;
        int rc = attend(&pool, block_tables + (size_t)s * max_blocks, max_blocks, h / g,
                        q + ((size_t)tok * num_heads + h) * head_dim, scale, 0, pos + 1,
                        out + (size_t)r * head_dim, &lse);
        if (rc < err) err = rc;
    }
    return err;
}

int pa_oracle_prefill(const uint16_t *k_cache, const uint16_t *v_cache, int32_t num_blocks, int32_t block_size,
                      int32_t num_kv_heads, int32_t head_dim, const uint16_t *q, const int32_t *cu_q_lens,
                      const int32_t *block_tables, int32_t max_blocks, const int32_t *seq_lens, int32_t batch,
                      int32_t num_heads, double scale, double *out) {
    return pa_oracle_prefill_rows(k_cache, v_cache, num_blocks, block_size, num_kv_heads, head_dim, q, cu_q_lens,
                                  block_tables, max_blocks, seq_lens, batch, num_heads, scale, NULL, NULL, 0,
                                  out);
}
