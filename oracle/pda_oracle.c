/*
 * pda_oracle.c -- TEST INFRASTRUCTURE ONLY (see pda_oracle.h).
 *
 * The plain definition of paged grouped-query decode attention, in fp64, with
 * no blocking, splitting or online rescaling: for each (b, h)
 *
 *   kvh   = h / (Hq / Hkv)
 *   K_t   = k_pool row (block_table[b][t / bs], t % bs, kvh),  t < seq_len
 *   V_t   = v_pool row (same address)
 *   s_t   = scale * sum_d q[b][h][d] * K_t[d]
 *   w_t   = exp(s_t - max_u s_u)
 *   out   = (sum_t w_t V_t) / (sum_t w_t)
 *
 * The online-softmax state (m, l, o) of tiled_attention.rs (module comment,
 * TiledAttention::begin_step / finalize) reaches exactly this value: m is the
 * running max, l the running sum of w_t and o the running sum of w_t V_t, and
 * the finalize step returns o / l.  Subtracting the maximum changes nothing
 * mathematically; it keeps exp() finite for large scores.
 */
#include "pda_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

double pdo_bf16_to_double(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

typedef struct {
    const uint16_t* q;
    const uint16_t* k_pool;
    const uint16_t* v_pool;
    const int32_t* block_table;
    const int32_t* seq_lens;
    int32_t B, Hq, Hkv, D, bs;
    int64_t num_blocks;
    int32_t max_blocks;
    int64_t blk_stride, tok_stride, kvh_stride;
    double scale;
} problem;

static int check_problem(const problem* P) {
    if (!P->q || !P->k_pool || !P->v_pool || !P->block_table || !P->seq_lens) return PDO_ERR_ARG;
    if (P->B < 0 || P->Hq <= 0 || P->Hkv <= 0 || P->D <= 0 || P->bs <= 0) return PDO_ERR_ARG;
    if (P->Hq % P->Hkv != 0) return PDO_ERR_ARG;
    if (P->num_blocks < 0 || P->max_blocks < 0) return PDO_ERR_ARG;
    if (P->blk_stride < 0 || P->tok_stride < 0 || P->kvh_stride < 0) return PDO_ERR_ARG;
    return PDO_OK;
}

/* Element offset of K/V row (blk, slot, kvh) in the pool. */
static int64_t row_offset(const problem* P, int64_t blk, int32_t slot, int32_t kvh) {
    return blk * P->blk_stride + (int64_t)slot * P->tok_stride + (int64_t)kvh * P->kvh_stride;
}

/* Resolves token t of sequence b to its pool block; -1 if the id is bad. */
static int64_t token_block(const problem* P, int32_t b, int32_t t) {
    int64_t blk = P->block_table[(int64_t)b * P->max_blocks + t / P->bs];
    if (blk < 0 || blk >= P->num_blocks) return -1;
    return blk;
}

/* Attention of query row qrow (q head h) over tokens 0..n-1 of sequence b. */
static int attend_prefix(const problem* P, int32_t b, int32_t h, int32_t n,
                         const uint16_t* qrow, double* out) {
    const int32_t D = P->D;
    const int32_t G = P->Hq / P->Hkv;
    const int32_t kvh = h / G;
    if (n < 0 || (int64_t)n > (int64_t)P->max_blocks * P->bs) return PDO_ERR_SEQLEN;
    for (int32_t d = 0; d < D; ++d) out[d] = 0.0;
    if (n == 0) return PDO_OK;

    double* s = (double*)malloc(sizeof(double) * (size_t)n);
    if (!s) return PDO_ERR_NOMEM;

    /* scores */
    for (int32_t t = 0; t < n; ++t) {
        int64_t blk = token_block(P, b, t);
        if (blk < 0) { free(s); return PDO_ERR_TABLE; }
        const uint16_t* krow = P->k_pool + row_offset(P, blk, t % P->bs, kvh);
        double dot = 0.0;
        for (int32_t d = 0; d < D; ++d)
            dot += pdo_bf16_to_double(qrow[d]) * pdo_bf16_to_double(krow[d]);
        s[t] = P->scale * dot;
    }
    /* softmax weights */
    double mx = s[0];
    for (int32_t t = 1; t < n; ++t) if (s[t] > mx) mx = s[t];
    double z = 0.0;
    for (int32_t t = 0; t < n; ++t) { s[t] = exp(s[t] - mx); z += s[t]; }
    /* weighted sum of value rows */
    for (int32_t t = 0; t < n; ++t) {
        int64_t blk = token_block(P, b, t);
        const uint16_t* vrow = P->v_pool + row_offset(P, blk, t % P->bs, kvh);
        for (int32_t d = 0; d < D; ++d) out[d] += s[t] * pdo_bf16_to_double(vrow[d]);
    }
    for (int32_t d = 0; d < D; ++d) out[d] /= z;
    free(s);
    return PDO_OK;
}

static int attend_one(const problem* P, int32_t b, int32_t h, double* out) {
    const uint16_t* qrow = P->q + ((int64_t)b * P->Hq + h) * P->D;
    return attend_prefix(P, b, h, P->seq_lens[b], qrow, out);
}

typedef struct {
    const problem* P;
    const int32_t* pairs;
    int64_t begin, end;
    double* out;
    int status;
    int32_t q_len;  /* > 0: multi-query job over (b, i, h) rows */
} job;

static void* run_job(void* arg) {
    job* j = (job*)arg;
    j->status = PDO_OK;
    if (j->q_len > 0) {  /* row i = (b, qi, h) of the [B, q_len, Hq] output */
        const problem* P = j->P;
        for (int64_t i = j->begin; i < j->end; ++i) {
            const int32_t h = (int32_t)(i % P->Hq);
            const int32_t qi = (int32_t)((i / P->Hq) % j->q_len);
            const int32_t b = (int32_t)(i / ((int64_t)P->Hq * j->q_len));
            int32_t n = P->seq_lens[b] - j->q_len + 1 + qi;
            if (n < 0) n = 0;
            const uint16_t* qrow = P->q + i * P->D;
            int st = attend_prefix(P, b, h, n, qrow, j->out + i * P->D);
            if (st != PDO_OK) { j->status = st; return NULL; }
        }
        return NULL;
    }
    for (int64_t i = j->begin; i < j->end; ++i) {
        int32_t b, h;
        if (j->pairs) { b = j->pairs[2 * i]; h = j->pairs[2 * i + 1]; }
        else { b = (int32_t)(i / j->P->Hq); h = (int32_t)(i % j->P->Hq); }
        if (b < 0 || b >= j->P->B || h < 0 || h >= j->P->Hq) { j->status = PDO_ERR_ARG; return NULL; }
        int st = attend_one(j->P, b, h, j->out + i * j->P->D);
        if (st != PDO_OK) { j->status = st; return NULL; }
    }
    return NULL;
}

static int run_jobs(const problem* P, const int32_t* pairs, int64_t total, int32_t q_len,
                    int32_t n_threads, double* out);

int pdo_decode(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
               const int32_t* block_table, const int32_t* seq_lens,
               int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t block_size,
               int64_t num_blocks, int32_t max_blocks,
               int64_t blk_stride, int64_t tok_stride, int64_t kvh_stride,
               double scale, const int32_t* pairs, int64_t n_pairs,
               int32_t n_threads, double* out) {
    problem P = {q, k_pool, v_pool, block_table, seq_lens, B, Hq, Hkv, D, block_size,
                 num_blocks, max_blocks, blk_stride, tok_stride, kvh_stride, scale};
    int st = check_problem(&P);
    if (st != PDO_OK) return st;
    if (!out) return PDO_ERR_ARG;
    int64_t total = pairs ? n_pairs : (int64_t)B * Hq;
    if (total < 0) return PDO_ERR_ARG;
    if (total == 0) return PDO_OK;

    return run_jobs(&P, pairs, total, 0, n_threads, out);
}

/* Runs `total` output rows on n_threads threads (the calling thread included). */
static int run_jobs(const problem* P, const int32_t* pairs, int64_t total, int32_t q_len,
                    int32_t n_threads, double* out) {
    if (n_threads < 1) n_threads = 1;
    if ((int64_t)n_threads > total) n_threads = (int32_t)total;
    job* jobs = (job*)calloc((size_t)n_threads, sizeof(job));
    pthread_t* tids = (pthread_t*)calloc((size_t)n_threads, sizeof(pthread_t));
    if (!jobs || !tids) { free(jobs); free(tids); return PDO_ERR_NOMEM; }
    for (int32_t i = 0; i < n_threads; ++i) {
        jobs[i].P = P;
        jobs[i].pairs = pairs;
        jobs[i].begin = total * i / n_threads;
        jobs[i].end = total * (i + 1) / n_threads;
        jobs[i].out = out;
        jobs[i].q_len = q_len;
    }
    int started = 0;
    for (int32_t i = 1; i < n_threads; ++i) {
        if (pthread_create(&tids[i], NULL, run_job, &jobs[i]) != 0) break;
        started = i;
    }
    run_job(&jobs[0]);
    /* jobs that could not get a thread run here */
    for (int32_t i = started + 1; i < n_threads; ++i) run_job(&jobs[i]);
    for (int32_t i = 1; i <= started; ++i) pthread_join(tids[i], NULL);
    int st = PDO_OK;
    for (int32_t i = 0; i < n_threads; ++i) if (jobs[i].status != PDO_OK) { st = jobs[i].status; break; }
    free(jobs);
    free(tids);
    return st;
}

int pdo_decode_multi(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                     const int32_t* block_table, const int32_t* seq_lens,
                     int32_t B, int32_t q_len, int32_t Hq, int32_t Hkv, int32_t D,
                     int32_t block_size, int64_t num_blocks, int32_t max_blocks,
                     int64_t blk_stride, int64_t tok_stride, int64_t kvh_stride,
                     double scale, int32_t n_threads, double* out) {
    problem P = {q, k_pool, v_pool, block_table, seq_lens, B, Hq, Hkv, D, block_size,
                 num_blocks, max_blocks, blk_stride, tok_stride, kvh_stride, scale};
    int st = check_problem(&P);
    if (st != PDO_OK) return st;
    if (!out || q_len < 1) return PDO_ERR_ARG;
    const int64_t total = (int64_t)B * q_len * Hq;
    if (total == 0) return PDO_OK;
    return run_jobs(&P, NULL, total, q_len, n_threads, out);
}

int pdo_gather(const uint16_t* k_pool, const uint16_t* v_pool,
               const int32_t* block_table, const int32_t* seq_lens,
               int32_t B, int32_t Hkv, int32_t D, int32_t block_size,
               int64_t num_blocks, int32_t max_blocks,
               int64_t blk_stride, int64_t tok_stride, int64_t kvh_stride,
               int32_t b, int32_t kvh, uint16_t* k_rows, uint16_t* v_rows) {
    /* q is unused by the gather; any non-null pointer passes the check */
    problem P = {k_pool, k_pool, v_pool, block_table, seq_lens, B, Hkv, Hkv, D, block_size,
                 num_blocks, max_blocks, blk_stride, tok_stride, kvh_stride, 1.0};
    int st = check_problem(&P);
    if (st != PDO_OK) return st;
    if (b < 0 || b >= B || kvh < 0 || kvh >= Hkv || !k_rows || !v_rows) return PDO_ERR_ARG;
    int32_t n = seq_lens[b];
    if (n < 0 || (int64_t)n > (int64_t)max_blocks * block_size) return PDO_ERR_SEQLEN;
    for (int32_t t = 0; t < n; ++t) {
        int64_t blk = token_block(&P, b, t);
        if (blk < 0) return PDO_ERR_TABLE;
        int64_t off = row_offset(&P, blk, t % block_size, kvh);
        memcpy(k_rows + (int64_t)t * D, k_pool + off, sizeof(uint16_t) * (size_t)D);
        memcpy(v_rows + (int64_t)t * D, v_pool + off, sizeof(uint16_t) * (size_t)D);
    }
    return PDO_OK;
}
