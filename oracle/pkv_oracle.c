/*
 * pkv_oracle.c -- plain, slow, obviously correct CPU oracle for the paged
 * KV-cache hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the test-suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code, header, table or constant with
 * the CUDA path.
 *
 * Precision: every attention quantity is computed in IEEE binary64 from the
 * exact widening of the bf16 (or int8 code x fp32 scale) inputs.  The int8
 * quantiser works in IEEE binary32, because the pages fix the scale as an fp32
 * value rounded to nearest-even, and a quantised code is an integer decided by
 * floating point: both sides take that decision in binary32.
 *
 * Build: gcc -O2 -fPIC -shared -ffp-contract=off -pthread (no -ffast-math, no
 * FMA contraction, so results are identical on x86-64 and aarch64).
 *
 * Layouts (all row-major, innermost last):
 *   pool      [n_blocks + 1][block_size][n_kv_heads][head_dim]   (token-major)
 *   scales    [n_blocks + 1][block_size][n_kv_heads]             (fp32)
 *   tables    [n_seqs][max_blocks] int32; physical id n_blocks = scratch block
 *   new rows  [n_seqs][n_new][n_kv_heads][head_dim]
 *   q decode  [n_seqs][n_q_heads][head_dim]
 *   q prefill [n_seqs][chunk][n_q_heads][head_dim]
 *   gather    [n_seqs][n_kv_heads][out_tokens][head_dim]
 *
 * Parity pins: every function here is checked by the CPU test-suite against
 * identity-table layouts, library routines (torch indexing, torch SDPA in
 * float64, numpy) and closed forms; none is "parity unpinned".
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define PKVO_OK 0
#define PKVO_BAD_ARG (-1)
#define PKVO_BAD_INDEX (-2)

static float bf16_to_float(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static double bf16_to_double(uint16_t bits) { return (double)bf16_to_float(bits); }

/*
 * Token -> slot map.  tiny-llm paged_kv.py, module docstring: token t of a
 * sequence lives at (table[t // block_size], t % block_size).  Returns the pool
 * row (physical block * block_size + offset) or -1 when the logical block is
 * outside the table or the table names an id outside [0, n_blocks].
 */
static int64_t slot_of(const int32_t *table_row, int32_t max_blocks, int32_t n_blocks,
                       int32_t block_size, int64_t t)
{
    if (t < 0) return -1;
    int64_t logical_block = t / block_size;
    if (logical_block >= max_blocks) return -1;
    int32_t physical = table_row[logical_block];
    if (physical < 0 || physical > n_blocks) return -1;
    return (int64_t)physical * block_size + (t % block_size);
}

/*
 * Native page write (tiny-llm paged_kv.py, PagedLayerKV.update; AstrAI
 * cache.py, PagedCache.write; libmir-metal paged/mod.rs, write::native).
 * For each sequence s and new token j the position is t = start_pos[s] + j and
 * the whole [n_kv_heads][head_dim] row of K and of V is copied, as raw 16-bit
 * patterns, to pool row slot_of(t).  Rows whose slot is invalid are skipped and
 * the call returns PKVO_BAD_INDEX.
 */
int pkvo_write_bf16(const uint16_t *k_new, const uint16_t *v_new, uint16_t *k_pool,
                    uint16_t *v_pool, int32_t n_blocks, int32_t block_size, int32_t n_kv_heads,
                    int32_t head_dim, const int32_t *tables, int32_t max_blocks,
                    const int32_t *start_pos, int32_t n_seqs, int32_t n_new)
{
    if (n_blocks < 0 || block_size <= 0 || n_kv_heads <= 0 || head_dim <= 0 || max_blocks <= 0 ||
        n_seqs < 0 || n_new < 0)
        return PKVO_BAD_ARG;
    int status = PKVO_OK;
    int64_t row = (int64_t)n_kv_heads * head_dim;
    for (int32_t s = 0; s < n_seqs; ++s) {
        for (int32_t j = 0; j < n_new; ++j) {
            int64_t t = (int64_t)start_pos[s] + j;
            int64_t slot = slot_of(tables + (int64_t)s * max_blocks, max_blocks, n_blocks,
                                   block_size, t);
            if (slot < 0) {
                status = PKVO_BAD_INDEX;
                continue;
            }
            const uint16_t *src_k = k_new + ((int64_t)s * n_new + j) * row;
            const uint16_t *src_v = v_new + ((int64_t)s * n_new + j) * row;
            for (int64_t e = 0; e < row; ++e) {
                k_pool[slot * row + e] = src_k[e];
                v_pool[slot * row + e] = src_v[e];
            }
        }
    }
    return status;
}

/*
 * Symmetric int8 quantisation of one [head_dim] row (libmir-metal paged/mod.rs,
 * KvPageFormat::Int8PerTokenHead and write::quantized; the scale rule is
 * absmax / 127 with round-to-nearest-even).  In binary32:
 *   amax = max_d |x_d|            (exact)
 *   scale = amax / 127            (one IEEE division, RNE)
 *   code_d = clamp(rint(x_d / scale), -127, 127)   (IEEE division, RNE)
 * A row of zeros stores scale 0 and codes 0.
 */
static void quantize_row(const uint16_t *x_bits, int32_t head_dim, int8_t *codes, float *scale)
{
    float amax = 0.0f;
    for (int32_t d = 0; d < head_dim; ++d) {
        float a = fabsf(bf16_to_float(x_bits[d]));
        if (a > amax) amax = a;
    }
    float s = amax / 127.0f;
    *scale = s;
    for (int32_t d = 0; d < head_dim; ++d) {
        int8_t c = 0;
        if (amax != 0.0f) {
            float quotient = bf16_to_float(x_bits[d]) / s;
            float r = nearbyintf(quotient); /* default rounding mode: ties to even */
            if (r > 127.0f) r = 127.0f;
            if (r < -127.0f) r = -127.0f;
            c = (int8_t)r;
        }
        codes[d] = c;
    }
}

/*
 * Quantised page write: the same token -> slot map as pkvo_write_bf16, with
 * every (token, kv_head) row of K and of V quantised by quantize_row and its
 * scale stored at scales[slot][kv_head].
 */
int pkvo_write_int8(const uint16_t *k_new, const uint16_t *v_new, int8_t *k_pool, int8_t *v_pool,
                    float *k_scales, float *v_scales, int32_t n_blocks, int32_t block_size,
                    int32_t n_kv_heads, int32_t head_dim, const int32_t *tables,
                    int32_t max_blocks, const int32_t *start_pos, int32_t n_seqs, int32_t n_new)
{
    if (n_blocks < 0 || block_size <= 0 || n_kv_heads <= 0 || head_dim <= 0 || max_blocks <= 0 ||
        n_seqs < 0 || n_new < 0)
        return PKVO_BAD_ARG;
    int status = PKVO_OK;
    for (int32_t s = 0; s < n_seqs; ++s) {
        for (int32_t j = 0; j < n_new; ++j) {
            int64_t t = (int64_t)start_pos[s] + j;
            int64_t slot = slot_of(tables + (int64_t)s * max_blocks, max_blocks, n_blocks,
                                   block_size, t);
            if (slot < 0) {
                status = PKVO_BAD_INDEX;
                continue;
            }
            for (int32_t h = 0; h < n_kv_heads; ++h) {
                int64_t src = (((int64_t)s * n_new + j) * n_kv_heads + h) * head_dim;
                int64_t dst = (slot * n_kv_heads + h) * head_dim;
                quantize_row(k_new + src, head_dim, k_pool + dst, &k_scales[slot * n_kv_heads + h]);
                quantize_row(v_new + src, head_dim, v_pool + dst, &v_scales[slot * n_kv_heads + h]);
            }
        }
    }
    return status;
}

/*
 * Explicit gather into a contiguous view (tiny-llm paged_kv.py,
 * PagedLayerKV.update -> gather; AstrAI cache.py, PagedCache.gather and
 * CacheView.gather; libmir-metal paged/mod.rs, context).  For t < lens[s]:
 *   out[s][h][t][:] = pool[slot_of(t)][h][:]
 * and columns lens[s] <= t < out_tokens are zero-filled (the cut at the
 * sequence length that AstrAI and libmir-metal make, written out as zeros so
 * the view is deterministic).
 */
int pkvo_gather(const uint16_t *k_pool, const uint16_t *v_pool, int32_t n_blocks,
                int32_t block_size, int32_t n_kv_heads, int32_t head_dim, const int32_t *tables,
                int32_t max_blocks, const int32_t *lens, int32_t n_seqs, int32_t out_tokens,
                uint16_t *k_out, uint16_t *v_out)
{
    if (n_blocks < 0 || block_size <= 0 || n_kv_heads <= 0 || head_dim <= 0 || max_blocks <= 0 ||
        n_seqs < 0 || out_tokens < 0)
        return PKVO_BAD_ARG;
    int status = PKVO_OK;
    for (int32_t s = 0; s < n_seqs; ++s) {
        int32_t len = lens[s];
        if (len < 0 || len > out_tokens) {
            status = PKVO_BAD_INDEX;
            len = len < 0 ? 0 : out_tokens;
        }
        for (int32_t h = 0; h < n_kv_heads; ++h) {
            for (int32_t t = 0; t < out_tokens; ++t) {
                int64_t dst = (((int64_t)s * n_kv_heads + h) * out_tokens + t) * head_dim;
                int64_t slot = -1;
                if (t < len) {
                    slot = slot_of(tables + (int64_t)s * max_blocks, max_blocks, n_blocks,
                                   block_size, t);
                    if (slot < 0) status = PKVO_BAD_INDEX;
                }
                for (int32_t d = 0; d < head_dim; ++d) {
                    if (slot >= 0) {
                        int64_t src = (slot * n_kv_heads + h) * head_dim + d;
                        k_out[dst + d] = k_pool[src];
                        v_out[dst + d] = v_pool[src];
                    } else {
                        k_out[dst + d] = 0;
                        v_out[dst + d] = 0;
                    }
                }
            }
        }
    }
    return status;
}

/* ------------------------------------------------------------------------ */
/* Attention                                                                  */
/* ------------------------------------------------------------------------ */

typedef struct {
    const void *k_pool, *v_pool;
    const float *k_scales, *v_scales;
    int32_t kv_dtype; /* 0 = bf16 pages, 1 = int8 pages + fp32 scales */
    int32_t n_blocks, block_size, n_kv_heads, head_dim;
    const int32_t *tables;
    int32_t max_blocks;
} pool_view;

/*
 * The value of element d of the K (which=0) or V (which=1) row of kv head h at
 * pool row `slot`, widened exactly to binary64.  Int8 pages dequantise as
 * (double)code * (double)scale (libmir-metal paged/mod.rs: quantised pages are
 * consumed by the attention itself).
 */
static double pool_value(const pool_view *pv, int which, int64_t slot, int32_t h, int32_t d)
{
    int64_t idx = (slot * pv->n_kv_heads + h) * pv->head_dim + d;
    if (pv->kv_dtype == 0) {
        const uint16_t *p = (const uint16_t *)(which ? pv->v_pool : pv->k_pool);
        return bf16_to_double(p[idx]);
    }
    const int8_t *p = (const int8_t *)(which ? pv->v_pool : pv->k_pool);
    const float *sc = which ? pv->v_scales : pv->k_scales;
    return (double)p[idx] * (double)sc[slot * pv->n_kv_heads + h];
}

/*
 * Softmax attention of one query row over logical tokens [t0, t1) of sequence
 * s, reading every key in place through the block table (tiny-llm paged_kv.py
 * module docstring: attention over the blocks in place instead of a gathered
 * copy).  Plain two passes in binary64:
 *   sc_t = softmax_scale * sum_d q_d k_{t,d}
 *   m = max_t sc_t,  w_t = exp(sc_t - m),  l = sum_t w_t,  acc_d = sum_t w_t v_{t,d}
 * Writes m, l and acc (unnormalised).  Returns -1 on an invalid slot, 0 when
 * the range is empty (m = -inf, l = 0, acc = 0), 1 otherwise.
 */
static int attend_range(const pool_view *pv, const int32_t *table_row, const uint16_t *q_row,
                        int32_t kv_head, double softmax_scale, int64_t t0, int64_t t1, double *m_out,
                        double *l_out, double *acc)
{
    int32_t D = pv->head_dim;
    for (int32_t d = 0; d < D; ++d) acc[d] = 0.0;
    *m_out = -INFINITY;
    *l_out = 0.0;
    if (t1 <= t0) return 0;
    int64_t n = t1 - t0;
    double *sc = (double *)malloc((size_t)n * sizeof(double));
    int64_t *slots = (int64_t *)malloc((size_t)n * sizeof(int64_t));
    if (!sc || !slots) {
        free(sc);
        free(slots);
        return -1;
    }
    int ok = 1;
    double m = -INFINITY;
    for (int64_t i = 0; i < n; ++i) {
        int64_t slot = slot_of(table_row, pv->max_blocks, pv->n_blocks, pv->block_size, t0 + i);
        if (slot < 0) {
            ok = 0;
            break;
        }
        slots[i] = slot;
        double dot = 0.0;
        for (int32_t d = 0; d < D; ++d)
            dot += bf16_to_double(q_row[d]) * pool_value(pv, 0, slot, kv_head, d);
        sc[i] = softmax_scale * dot;
        if (sc[i] > m) m = sc[i];
    }
    if (ok) {
        double l = 0.0;
        for (int64_t i = 0; i < n; ++i) {
            double w = exp(sc[i] - m);
            l += w;
            for (int32_t d = 0; d < D; ++d) acc[d] += w * pool_value(pv, 1, slots[i], kv_head, d);
        }
        *m_out = m;
        *l_out = l;
    }
    free(sc);
    free(slots);
    return ok ? 1 : -1;
}

/* ---- a tiny fixed-size thread fan-out over an index range ---------------- */

typedef void (*range_fn)(void *ctx, int64_t begin, int64_t end);

typedef struct {
    range_fn fn;
    void *ctx;
    int64_t begin, end;
} range_job;

static void *range_job_main(void *arg)
{
    range_job *job = (range_job *)arg;
    job->fn(job->ctx, job->begin, job->end);
    return NULL;
}

/* Runs fn over [0, n) split into n_threads contiguous pieces (n_threads <= 1:
 * in the calling thread). */
static void run_parallel(range_fn fn, void *ctx, int64_t n, int n_threads)
{
    if (n_threads <= 1 || n <= 1) {
        fn(ctx, 0, n);
        return;
    }
    if (n_threads > n) n_threads = (int)n;
    pthread_t *tids = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
    range_job *jobs = (range_job *)malloc(sizeof(range_job) * (size_t)n_threads);
    int *started = (int *)calloc((size_t)n_threads, sizeof(int));
    for (int i = 0; i < n_threads; ++i) {
        jobs[i].fn = fn;
        jobs[i].ctx = ctx;
        jobs[i].begin = n * i / n_threads;
        jobs[i].end = n * (i + 1) / n_threads;
        started[i] = pthread_create(&tids[i], NULL, range_job_main, &jobs[i]) == 0;
        if (!started[i]) fn(ctx, jobs[i].begin, jobs[i].end);
    }
    for (int i = 0; i < n_threads; ++i)
        if (started[i]) pthread_join(tids[i], NULL);
    free(tids);
    free(jobs);
    free(started);
}

/* ---- decode --------------------------------------------------------------- */

typedef struct {
    pool_view pv;
    const uint16_t *q;
    int32_t n_q_heads;
    const int32_t *ctx_lens;
    double softmax_scale;
    int32_t split_tokens; /* 0: one pass over the whole context */
    double *out;
    double *lse;
    int status;
    pthread_mutex_t lock;
} decode_job;

static void decode_fail(decode_job *job)
{
    pthread_mutex_lock(&job->lock);
    job->status = PKVO_BAD_INDEX;
    pthread_mutex_unlock(&job->lock);
}

/*
 * One (sequence, query head) of decode.  GQA: query head h reads kv head
 * h / (n_q_heads / n_kv_heads) (contiguous groups).  With split_tokens > 0 the
 * context is cut into logical ranges [k*S, (k+1)*S), each range keeps its own
 * (m_k, l_k, acc_k) and the ranges are combined by their log-sum-exp
 * lse_k = m_k + ln l_k (metrale high_speed_swap impl_more.rs,
 * attend_layer_on_stream_with_q_pos: per-tile steps joined by one finalize):
 *   M = max_k lse_k,  o = sum_k e^{lse_k - M} acc_k / l_k  /  sum_k e^{lse_k - M}
 * Without splits o = acc / l and lse = m + ln l.  An empty context gives o = 0
 * and lse = -inf.
 */
static void decode_one(decode_job *job, int64_t index)
{
    const pool_view *pv = &job->pv;
    int32_t D = pv->head_dim;
    int32_t s = (int32_t)(index / job->n_q_heads);
    int32_t h = (int32_t)(index % job->n_q_heads);
    int32_t group = job->n_q_heads / pv->n_kv_heads;
    int32_t kv_head = h / group;
    const int32_t *table_row = pv->tables + (int64_t)s * pv->max_blocks;
    const uint16_t *q_row = job->q + index * D;
    double *o = job->out + index * D;
    int64_t L = job->ctx_lens[s];
    double *acc = (double *)malloc(sizeof(double) * (size_t)D);
    for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
    if (job->lse) job->lse[index] = -INFINITY;
    if (L < 0 || L > (int64_t)pv->max_blocks * pv->block_size) {
        decode_fail(job);
        free(acc);
        return;
    }
    if (job->split_tokens <= 0) {
        double m, l;
        int r = attend_range(pv, table_row, q_row, kv_head, job->softmax_scale, 0, L, &m, &l, acc);
        if (r < 0) decode_fail(job);
        if (r == 1) {
            for (int32_t d = 0; d < D; ++d) o[d] = acc[d] / l;
            if (job->lse) job->lse[index] = m + log(l);
        }
        free(acc);
        return;
    }
    int64_t S = job->split_tokens;
    int64_t n_splits = (L + S - 1) / S;
    double *lse_k = (double *)malloc(sizeof(double) * (size_t)(n_splits > 0 ? n_splits : 1));
    double *o_k = (double *)malloc(sizeof(double) * (size_t)D * (size_t)(n_splits > 0 ? n_splits : 1));
    int bad = 0;
    for (int64_t k = 0; k < n_splits; ++k) {
        int64_t t0 = k * S, t1 = (k + 1) * S < L ? (k + 1) * S : L;
        double m, l;
        int r = attend_range(pv, table_row, q_row, kv_head, job->softmax_scale, t0, t1, &m, &l, acc);
        if (r < 0) {
            bad = 1;
            break;
        }
        lse_k[k] = m + log(l);
        for (int32_t d = 0; d < D; ++d) o_k[k * D + d] = acc[d] / l;
    }
    if (bad) {
        decode_fail(job);
    } else if (n_splits > 0) {
        double M = -INFINITY;
        for (int64_t k = 0; k < n_splits; ++k)
            if (lse_k[k] > M) M = lse_k[k];
        double denom = 0.0;
        for (int64_t k = 0; k < n_splits; ++k) denom += exp(lse_k[k] - M);
        for (int32_t d = 0; d < D; ++d) {
            double num = 0.0;
            for (int64_t k = 0; k < n_splits; ++k) num += exp(lse_k[k] - M) * o_k[k * D + d];
            o[d] = num / denom;
        }
        if (job->lse) job->lse[index] = M + log(denom);
    }
    free(lse_k);
    free(o_k);
    free(acc);
}

static void decode_range(void *ctx, int64_t begin, int64_t end)
{
    for (int64_t i = begin; i < end; ++i) decode_one((decode_job *)ctx, i);
}

/*
 * Paged decode attention: for every sequence s and query head h, softmax
 * attention of q[s][h] over the ctx_lens[s] tokens of sequence s, read in place
 * through its block table.  out [n_seqs][n_q_heads][head_dim] and lse
 * [n_seqs][n_q_heads] (nullable) are binary64.  split_tokens > 0 computes the
 * same result through per-range partials and the log-sum-exp merge.
 */
int pkvo_decode(const uint16_t *q, int32_t n_q_heads, const void *k_pool, const void *v_pool,
                const float *k_scales, const float *v_scales, int32_t kv_dtype, int32_t n_blocks,
                int32_t block_size, int32_t n_kv_heads, int32_t head_dim, const int32_t *tables,
                int32_t max_blocks, const int32_t *ctx_lens, int32_t n_seqs, float softmax_scale,
                int32_t split_tokens, double *out, double *lse, int32_t n_threads)
{
    if (n_blocks < 0 || block_size <= 0 || n_kv_heads <= 0 || head_dim <= 0 || max_blocks <= 0 ||
        n_seqs < 0 || n_q_heads <= 0 || n_q_heads % n_kv_heads != 0 ||
        (kv_dtype != 0 && kv_dtype != 1) || (kv_dtype == 1 && (!k_scales || !v_scales)))
        return PKVO_BAD_ARG;
    decode_job job;
    job.pv = (pool_view){k_pool,    v_pool,     k_scales,   v_scales, kv_dtype,  n_blocks,
                         block_size, n_kv_heads, head_dim, tables,   max_blocks};
    job.q = q;
    job.n_q_heads = n_q_heads;
    job.ctx_lens = ctx_lens;
    job.softmax_scale = (double)softmax_scale;
    job.split_tokens = split_tokens;
    job.out = out;
    job.lse = lse;
    job.status = PKVO_OK;
    pthread_mutex_init(&job.lock, NULL);
    run_parallel(decode_range, &job, (int64_t)n_seqs * n_q_heads, n_threads);
    pthread_mutex_destroy(&job.lock);
    return job.status;
}

/* ---- chunked prefill --------------------------------------------------------- */

typedef struct {
    pool_view pv;
    const uint16_t *q;
    int32_t n_q_heads, chunk;
    const int32_t *prefix_lens;
    const uint8_t *row_select; /* [n_seqs][chunk], nullable = all rows */
    double softmax_scale;
    double *out;
    double *lse;
    int status;
    pthread_mutex_t lock;
} prefill_job;

/*
 * One (sequence, chunk row i, query head h) of chunked prefill.  The chunk's
 * K/V rows were already written at positions P .. P+chunk-1 (P = prefix_lens[s],
 * AstrAI cache.py, PagedCache.write with seq_len > 1), and query i sits at
 * absolute position P + i.  It attends keys 0 .. P+i: the whole resident prefix
 * and, causally, the chunk up to itself (metrale impl_more.rs: a query at q_pos
 * sees only the first (q_pos % block_size) + 1 slots of its own last block).
 */
static void prefill_one(prefill_job *job, int64_t index)
{
    const pool_view *pv = &job->pv;
    int32_t D = pv->head_dim;
    int32_t h = (int32_t)(index % job->n_q_heads);
    int64_t si = index / job->n_q_heads;
    int32_t s = (int32_t)(si / job->chunk);
    int32_t i = (int32_t)(si % job->chunk);
    if (job->row_select && !job->row_select[si]) return;
    int32_t group = job->n_q_heads / pv->n_kv_heads;
    double *o = job->out + index * D;
    double *acc = (double *)malloc(sizeof(double) * (size_t)D);
    double m, l;
    int64_t t1 = (int64_t)job->prefix_lens[s] + i + 1;
    int r = attend_range(pv, pv->tables + (int64_t)s * pv->max_blocks, job->q + index * D,
                         h / group, job->softmax_scale, 0, t1, &m, &l, acc);
    if (r == 1) {
        for (int32_t d = 0; d < D; ++d) o[d] = acc[d] / l;
        if (job->lse) job->lse[index] = m + log(l);
    } else {
        for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
        if (job->lse) job->lse[index] = -INFINITY;
        pthread_mutex_lock(&job->lock);
        job->status = PKVO_BAD_INDEX;
        pthread_mutex_unlock(&job->lock);
    }
    free(acc);
}

static void prefill_range(void *ctx, int64_t begin, int64_t end)
{
    for (int64_t i = begin; i < end; ++i) prefill_one((prefill_job *)ctx, i);
}

/*
 * Chunked paged prefill.  q and out are [n_seqs][chunk][n_q_heads][head_dim]
 * (out in binary64), lse [n_seqs][chunk][n_q_heads] (nullable).  row_select
 * (nullable, [n_seqs][chunk]) restricts the work to the selected chunk rows;
 * unselected rows of out/lse are left untouched.
 */
int pkvo_prefill(const uint16_t *q, int32_t n_q_heads, const uint16_t *k_pool,
                 const uint16_t *v_pool, int32_t n_blocks, int32_t block_size, int32_t n_kv_heads,
                 int32_t head_dim, const int32_t *tables, int32_t max_blocks,
                 const int32_t *prefix_lens, int32_t n_seqs, int32_t chunk, float softmax_scale,
                 const uint8_t *row_select, double *out, double *lse, int32_t n_threads)
{
    if (n_blocks < 0 || block_size <= 0 || n_kv_heads <= 0 || head_dim <= 0 || max_blocks <= 0 ||
        n_seqs < 0 || chunk < 0 || n_q_heads <= 0 || n_q_heads % n_kv_heads != 0)
        return PKVO_BAD_ARG;
    prefill_job job;
    job.pv = (pool_view){k_pool,    v_pool,     NULL,     NULL,   0,         n_blocks,
                         block_size, n_kv_heads, head_dim, tables, max_blocks};
    job.q = q;
    job.n_q_heads = n_q_heads;
    job.chunk = chunk;
    job.prefix_lens = prefix_lens;
    job.row_select = row_select;
    job.softmax_scale = (double)softmax_scale;
    job.out = out;
    job.lse = lse;
    job.status = PKVO_OK;
    pthread_mutex_init(&job.lock, NULL);
    run_parallel(prefill_range, &job, (int64_t)n_seqs * chunk * n_q_heads, n_threads);
    pthread_mutex_destroy(&job.lock);
    return job.status;
}
