/*
 * fd_oracle.c -- plain fp64 CPU oracle for split-KV decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: only tests/, the smoke check and the benchmark's CPU-baseline leg
 * use it.  It shares no code, header, table or helper with the CUDA library.
 *
 * Source of the method: "FlashDecoding++: sequence-dimension KV split
 * parallelism for LLM serving" (techknowgenie.com), §3 "Partial softmax and
 * two-stage global reduction".  Three functions:
 *
 *   fdo_decode          the plain definition the two-stage method reaches
 *                       exactly (the article's §3 closing paragraph: the
 *                       two-stage result equals single-pass attention up to
 *                       rounding).  For each request b and query head hq:
 *                         s_j  = scale * sum_d q[b,hq,d] * K[j,kvh,d]
 *                         M    = max_j s_j
 *                         Z    = sum_j exp(s_j - M)
 *                         O    = sum_j exp(s_j - M) * V[j,kvh,:] / Z
 *                         LSE  = M + ln Z
 *                       over the request's rows j, with kvh = hq / (Hq/Hkv)
 *                       (contiguous query-head groups share one KV head).
 *                       An empty request gives O = 0, LSE = -inf.
 *
 *   fdo_split_partials  stage 1 of §3: for one chunk of one request's keys,
 *                       the local logits, local max m, local sum l of
 *                       exp(logit - m), and the local partial output
 *                       acc = sum exp(logit - m) * V  (un-normalised), i.e.
 *                       the three quantities the article stores per chunk.
 *
 *   fdo_merge           stage 2 of §3: global max M = max_i m_i, rescaling
 *                       factors f_i = exp(m_i - M), global denominator
 *                       sum_i f_i l_i, output sum_i f_i acc_i / denominator,
 *                       and LSE = M + ln(denominator).  No epsilon is added to
 *                       the denominator (it is >= 1 whenever a chunk is
 *                       non-empty).  A segment with no non-empty chunk gives
 *                       O = 0, LSE = -inf.
 *
 * Element types of q, K, V: 0 = bf16 (raw 16-bit patterns, widened exactly to
 * fp32 then fp64), 1 = fp32, 2 = fp64.  All arithmetic is fp64.
 * Every function returns 0 on success, -1 on a bad argument.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { FDO_BF16 = 0, FDO_F32 = 1, FDO_F64 = 2 };

static double elem(int dtype, const void *base, int64_t idx)
{
    if (dtype == FDO_BF16) {
        uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    if (dtype == FDO_F32)
        return (double)((const float *)base)[idx];
    return ((const double *)base)[idx];
}

typedef struct {
    int dtype;
    const void *q, *k, *v;
    const int64_t *kv_indptr;
    int64_t batch, hq_n, hkv_n, d_n;
    double scale;
} inputs_t;

/* scale * <q[b,hq,:], K[j,kvh,:]> */
static double logit(const inputs_t *in, int64_t b, int64_t hq, int64_t kvh, int64_t j)
{
    double dot = 0.0;
    for (int64_t d = 0; d < in->d_n; ++d)
        dot += elem(in->dtype, in->q, (b * in->hq_n + hq) * in->d_n + d) *
               elem(in->dtype, in->k, (j * in->hkv_n + kvh) * in->d_n + d);
    return in->scale * dot;
}

/* ---------------------------------------------------------------- decode */

static void decode_row(const inputs_t *in, int64_t row, double *o, double *lse)
{
    const int64_t b = row / in->hq_n, hq = row % in->hq_n;
    const int64_t group = in->hq_n / in->hkv_n, kvh = hq / group;
    const int64_t j0 = in->kv_indptr[b], j1 = in->kv_indptr[b + 1], n = j1 - j0;
    for (int64_t d = 0; d < in->d_n; ++d)
        o[d] = 0.0;
    if (n <= 0) {
        *lse = -INFINITY;
        return;
    }
    double *s = (double *)malloc((size_t)n * sizeof(double));
    for (int64_t j = 0; j < n; ++j)
        s[j] = logit(in, b, hq, kvh, j0 + j);
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j)
        if (s[j] > m)
            m = s[j];
    double z = 0.0;
    for (int64_t j = 0; j < n; ++j)
        z += exp(s[j] - m);
    for (int64_t j = 0; j < n; ++j) {
        const double p = exp(s[j] - m);
        for (int64_t d = 0; d < in->d_n; ++d)
            o[d] += p * elem(in->dtype, in->v, ((j0 + j) * in->hkv_n + kvh) * in->d_n + d);
    }
    for (int64_t d = 0; d < in->d_n; ++d)
        o[d] /= z;
    *lse = m + log(z);
    free(s);
}

typedef struct {
    const inputs_t *in;
    const int64_t *rows;
    int64_t nrows;
    double *o, *lse;
    int64_t next;
    pthread_mutex_t lock;
} decode_job_t;

static void *decode_worker(void *arg)
{
    decode_job_t *job = (decode_job_t *)arg;
    for (;;) {
        pthread_mutex_lock(&job->lock);
        const int64_t i = job->next++;
        pthread_mutex_unlock(&job->lock);
        if (i >= job->nrows)
            return NULL;
        const int64_t row = job->rows ? job->rows[i] : i;
        decode_row(job->in, row, job->o + i * job->in->d_n, job->lse + i);
    }
}

/*
 * q [batch, hq_n, d_n], k/v [T, hkv_n, d_n], kv_indptr int64 [batch+1].
 * rows: flat (b * hq_n + hq) indices to compute (NULL = all batch*hq_n rows).
 * o [nrows, d_n], lse [nrows] (fp64, caller-owned).
 */
int fdo_decode(int dtype, const void *q, const void *k, const void *v,
               const int64_t *kv_indptr, int64_t batch, int64_t hq_n, int64_t hkv_n,
               int64_t d_n, double scale, const int64_t *rows, int64_t nrows,
               double *o, double *lse, int nthreads)
{
    if (!q || !kv_indptr || !o || !lse || batch < 0 || hq_n <= 0 || hkv_n <= 0 ||
        d_n <= 0 || hq_n % hkv_n != 0 || nrows < 0 || dtype < 0 || dtype > 2)
        return -1;
    if (!rows && nrows != batch * hq_n)
        return -1;
    for (int64_t i = 0; rows && i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= batch * hq_n)
            return -1;
    inputs_t in = {dtype, q, k, v, kv_indptr, batch, hq_n, hkv_n, d_n, scale};
    decode_job_t job = {&in, rows, nrows, o, lse, 0, PTHREAD_MUTEX_INITIALIZER};
    if (nthreads < 1)
        nthreads = 1;
    pthread_t *tid = (pthread_t *)malloc((size_t)nthreads * sizeof(pthread_t));
    for (int t = 0; t < nthreads; ++t)
        pthread_create(&tid[t], NULL, decode_worker, &job);
    for (int t = 0; t < nthreads; ++t)
        pthread_join(tid[t], NULL);
    free(tid);
    return 0;
}

/* ------------------------------------------------------ stage 1 (chunks) */

/*
 * items [n_items][4] = (b, kvh, tok_begin, tok_end): absolute key rows
 * [tok_begin, tok_end) of request b, which must lie inside the request.
 * Outputs per item and per query head g of the group (hq = kvh*G + g):
 *   acc [n_items, G, d_n]   sum_j exp(s_j - m) V[j]  (un-normalised)
 *   m   [n_items, G]        local max of the logits
 *   l   [n_items, G]        local sum of exp(s_j - m)
 */
int fdo_split_partials(int dtype, const void *q, const void *k, const void *v,
                       const int64_t *kv_indptr, int64_t batch, int64_t hq_n,
                       int64_t hkv_n, int64_t d_n, double scale,
                       const int64_t *items, int64_t n_items,
                       double *acc, double *m, double *l)
{
    if (!q || !k || !v || !kv_indptr || !items || !acc || !m || !l || hq_n <= 0 ||
        hkv_n <= 0 || d_n <= 0 || hq_n % hkv_n != 0 || dtype < 0 || dtype > 2)
        return -1;
    inputs_t in = {dtype, q, k, v, kv_indptr, batch, hq_n, hkv_n, d_n, scale};
    const int64_t group = hq_n / hkv_n;
    for (int64_t it = 0; it < n_items; ++it) {
        const int64_t b = items[4 * it], kvh = items[4 * it + 1];
        const int64_t t0 = items[4 * it + 2], t1 = items[4 * it + 3];
        if (b < 0 || b >= batch || kvh < 0 || kvh >= hkv_n || t0 >= t1 ||
            t0 < kv_indptr[b] || t1 > kv_indptr[b + 1])
            return -1;
        double *s = (double *)malloc((size_t)(t1 - t0) * sizeof(double));
        for (int64_t g = 0; g < group; ++g) {
            const int64_t hq = kvh * group + g;
            double *acc_row = acc + (it * group + g) * d_n;
            for (int64_t j = t0; j < t1; ++j)
                s[j - t0] = logit(&in, b, hq, kvh, j);
            double mx = -INFINITY;
            for (int64_t j = 0; j < t1 - t0; ++j)
                if (s[j] > mx)
                    mx = s[j];
            double sum = 0.0;
            for (int64_t d = 0; d < d_n; ++d)
                acc_row[d] = 0.0;
            for (int64_t j = t0; j < t1; ++j) {
                const double e = exp(s[j - t0] - mx);
                sum += e;
                for (int64_t d = 0; d < d_n; ++d)
                    acc_row[d] += e * elem(dtype, v, (j * hkv_n + kvh) * d_n + d);
            }
            m[it * group + g] = mx;
            l[it * group + g] = sum;
        }
        free(s);
    }
    return 0;
}

/* ----------------------------------------------- stage 2 (global reduce) */

/*
 * Partials i = seg_indptr[r] .. seg_indptr[r+1]-1 belong to output row r.
 * acc [n, d_n], m [n], l [n]  ->  o [n_rows, d_n], lse [n_rows].
 * A partial with l = 0 (an empty chunk, m = -inf) carries no weight.
 */
int fdo_merge(const double *acc, const double *m, const double *l,
              const int64_t *seg_indptr, int64_t n_rows, int64_t d_n,
              double *o, double *lse)
{
    if (!seg_indptr || !o || !lse || n_rows < 0 || d_n <= 0)
        return -1;
    for (int64_t r = 0; r < n_rows; ++r) {
        const int64_t i0 = seg_indptr[r], i1 = seg_indptr[r + 1];
        if (i1 < i0)
            return -1;
        double *orow = o + r * d_n;
        for (int64_t d = 0; d < d_n; ++d)
            orow[d] = 0.0;
        double gmax = -INFINITY;
        for (int64_t i = i0; i < i1; ++i)
            if (m[i] > gmax)
                gmax = m[i];
        if (gmax == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double denom = 0.0;
        for (int64_t i = i0; i < i1; ++i) {
            if (m[i] == -INFINITY)
                continue;
            const double f = exp(m[i] - gmax);
            denom += f * l[i];
            for (int64_t d = 0; d < d_n; ++d)
                orow[d] += f * acc[i * d_n + d];
        }
        for (int64_t d = 0; d < d_n; ++d)
            orow[d] /= denom;
        lse[r] = gmax + log(denom);
    }
    return 0;
}
