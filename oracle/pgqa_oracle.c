/*
 * CPU oracle for paged GQA decode attention, in f64.  TEST INFRASTRUCTURE
 * ONLY: the library under paged_gqa_decode_attn_gb300/ never links, loads or
 * calls this file, and this file shares no code or header with it.
 *
 * What it computes follows the f64 `reference` function of span-02
 * `engine/crates/kernels/tests/gpu.rs` (the kernels crate's GPU test file):
 * for every query row t and head h, with kv head kh = h / (nh / nkv),
 *
 *   lo   = window > 0 ? max(0, qpos[t] + 1 - window) : 0
 *   s_p  = sum_d q[t,h,d] * K[p,kh,d]              p in [lo, qpos[t]]
 *   m    = max_p s_p
 *   e_p  = exp(s_p - m),   z = sum_p e_p
 *   o_d  = sum_p (e_p / z) * V[p,kh,d]
 *   out  = bf16 of (f32 of o), bf16 taken by truncation (the page's `bf`).
 *
 * Scaling is 1.0.  K/V position p of row t lives in physical page
 * phys = block_table[off[t] + p/16] (then page_map[phys] when a page map is
 * given), at element ((phys*nkv + kh)*16 + p%16)*hd + d of the
 * [page][nkv][16][hd] pool, as the same test file indexes it.
 *
 * Readings where the page is silent:
 *  - `kvpos` (the second position array the page passes, always equal to
 *    qpos there) is the last KV position written for the row.  The `reference`
 *    range ends at the query's own position (`lo..=qp`: the attention is
 *    causal), so the second array can only shorten it: the row attends over
 *    [lo, min(qpos[t], kvpos[t])], lo still taken from qpos.  NULL means
 *    kvpos = qpos.
 *  - The page map composes after the block table: page_map[block_table[.]].
 *  - A row with no visible position (kvpos < lo) yields zeros.
 *
 * Plain loops, no blocking, no reordering: threads only split the
 * (row, head) pairs, each pair is computed start to end by one thread.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
    const uint16_t *q, *k_pool, *v_pool;
    const int32_t *block_table, *off, *qpos, *kvpos, *page_map;
    int rows, nh, nkv, hd, window;
    const int32_t *pairs; /* npairs x (row, head), or NULL for all pairs */
    int npairs;
    double *out_f64;      /* [npairs][hd] or NULL */
    uint16_t *out_bf16;   /* [npairs][hd] or NULL */
    int next;             /* shared work counter */
    int status;
} job_t;

/* bf16 bits -> value (the page's `f`, widened to f64, which is exact). */
static double bf16_value(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* f64 -> f32 (round to nearest even) -> bf16 by dropping the low 16 bits. */
static uint16_t bf16_truncate(double x)
{
    float f = (float)x;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* Element offset of (row t, position p, kv head kh, dim 0) in the pool. */
static int64_t kv_offset(const job_t *j, int t, int p, int kh)
{
    int64_t phys = j->block_table[(int64_t)j->off[t] + p / 16];
    if (j->page_map)
        phys = j->page_map[phys];
    return ((phys * j->nkv + kh) * 16 + p % 16) * (int64_t)j->hd;
}

static void row_head(const job_t *j, int t, int h, double *o, double *s)
{
    int hd = j->hd;
    int qp = j->qpos[t];
    int hi = qp;                      /* causal: no position past the query's own */
    if (j->kvpos && j->kvpos[t] < hi)
        hi = j->kvpos[t];             /* the second position array only shortens the range */
    int lo = 0;
    if (j->window > 0) {
        lo = qp + 1 - j->window;
        if (lo < 0)
            lo = 0;
    }
    for (int d = 0; d < hd; d++)
        o[d] = 0.0;
    if (hi < lo)
        return;
    int n = hi - lo + 1;
    int kh = h / (j->nh / j->nkv);
    const uint16_t *qv = j->q + ((int64_t)t * j->nh + h) * hd;

    /* scores */
    for (int i = 0; i < n; i++) {
        const uint16_t *kv = j->k_pool + kv_offset(j, t, lo + i, kh);
        double acc = 0.0;
        for (int d = 0; d < hd; d++)
            acc += bf16_value(qv[d]) * bf16_value(kv[d]);
        s[i] = acc;
    }
    /* max, exponentials, normaliser */
    double m = -INFINITY;
    for (int i = 0; i < n; i++)
        if (s[i] > m)
            m = s[i];
    double z = 0.0;
    for (int i = 0; i < n; i++) {
        s[i] = exp(s[i] - m);
        z += s[i];
    }
    /* weighted sum of V */
    for (int i = 0; i < n; i++) {
        const uint16_t *vv = j->v_pool + kv_offset(j, t, lo + i, kh);
        double w = s[i] / z;
        for (int d = 0; d < hd; d++)
            o[d] += w * bf16_value(vv[d]);
    }
}

static int max_len(const job_t *j)
{
    int best = 1;
    for (int t = 0; t < j->rows; t++) {
        int qp = j->qpos[t];
        int hi = j->kvpos && j->kvpos[t] < qp ? j->kvpos[t] : qp;
        int lo = j->window > 0 ? qp + 1 - j->window : 0;
        if (lo < 0)
            lo = 0;
        if (hi - lo + 1 > best)
            best = hi - lo + 1;
    }
    return best;
}

static void *worker(void *arg)
{
    job_t *j = (job_t *)arg;
    int hd = j->hd;
    double *o = (double *)malloc(sizeof(double) * (size_t)hd);
    double *s = (double *)malloc(sizeof(double) * (size_t)max_len(j));
    if (!o || !s) {
        __atomic_store_n(&j->status, -2, __ATOMIC_SEQ_CST);
        free(o);
        free(s);
        return NULL;
    }
    for (;;) {
        int i = __atomic_fetch_add(&j->next, 1, __ATOMIC_RELAXED);
        if (i >= j->npairs)
            break;
        int t = j->pairs ? j->pairs[2 * i] : i / j->nh;
        int h = j->pairs ? j->pairs[2 * i + 1] : i % j->nh;
        row_head(j, t, h, o, s);
        for (int d = 0; d < hd; d++) {
            if (j->out_f64)
                j->out_f64[(int64_t)i * hd + d] = o[d];
            if (j->out_bf16)
                j->out_bf16[(int64_t)i * hd + d] = bf16_truncate(o[d]);
        }
    }
    free(o);
    free(s);
    return NULL;
}

/*
 * Decode attention for `npairs` (row, head) pairs listed in `pairs`
 * (2 int32 each), or for all rows*nh pairs in row-major order when `pairs`
 * is NULL.  Outputs are [pair][hd].  `nthreads <= 0` uses every online core.
 * Returns 0, or -1 on bad arguments, -2 when memory runs out.
 */
int pgqa_oracle_decode(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                       const int32_t *block_table, const int32_t *off, const int32_t *qpos,
                       const int32_t *kvpos, const int32_t *page_map, int rows, int nh, int nkv,
                       int hd, int window, const int32_t *pairs, int npairs, double *out_f64,
                       uint16_t *out_bf16, int nthreads)
{
    if (!q || !k_pool || !v_pool || !block_table || !off || !qpos || rows < 0 || nh <= 0 ||
        nkv <= 0 || nh % nkv != 0 || hd <= 0 || window < 0)
        return -1;
    job_t j;
    memset(&j, 0, sizeof j);
    j.q = q;
    j.k_pool = k_pool;
    j.v_pool = v_pool;
    j.block_table = block_table;
    j.off = off;
    j.qpos = qpos;
    j.kvpos = kvpos;
    j.page_map = page_map;
    j.rows = rows;
    j.nh = nh;
    j.nkv = nkv;
    j.hd = hd;
    j.window = window;
    j.pairs = pairs;
    j.npairs = pairs ? npairs : rows * nh;
    j.out_f64 = out_f64;
    j.out_bf16 = out_bf16;
    if (nthreads <= 0)
        nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > j.npairs)
        nthreads = j.npairs > 0 ? j.npairs : 1;
    if (nthreads == 1) {
        worker(&j);
        return j.status;
    }
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!tid)
        return -2;
    int started = 0;
    for (int i = 0; i < nthreads; i++) {
        if (pthread_create(&tid[i], NULL, worker, &j) != 0)
            break;
        started++;
    }
    if (started == 0)
        worker(&j);
    for (int i = 0; i < started; i++)
        pthread_join(tid[i], NULL);
    free(tid);
    return j.status;
}

/* Number of threads the oracle would use for `nthreads <= 0`. */
int pgqa_oracle_default_threads(void)
{
    int n = (int)sysconf(_SC_NPROCESSORS_ONLN);
    return n < 1 ? 1 : n;
}
