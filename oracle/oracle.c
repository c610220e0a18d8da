/*
 * Reference oracle for paged-KV decode attention -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, fp64.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg load this file's library; the product path
 * never does.  It shares no code, header or constant with the CUDA library.
 *
 * What it computes (each function cites the passage it follows):
 *
 *   oracle_lengths   -- request length from the page table,
 *                       l = P (n - 1) + r with 1 <= r <= P
 *                       ("FlashInfer 完全拆解", section 页表就是一张块稀疏矩阵;
 *                        "FlashInfer, in depth", section "The block-sparse
 *                        page table").
 *   oracle_attend    -- for one query row (request i, query head h) and a
 *                       token range [t0, t1) of that request:
 *                       s_t = q . k_t / sqrt(d), P = softmax(s), O = P V,
 *                       plus the natural-log log-sum-exp of the scaled
 *                       scores ("FlashInfer 完全拆解", section 从推理形状出发,
 *                       the definitions S = QK^T/sqrt(d), P = softmax(S),
 *                       O = PV; section 在线 Softmax 为什么允许任意切块, the
 *                       attention state (O_I, L_I)).  The full range gives
 *                       decode attention; a sub-range gives the partial state
 *                       of that chunk.
 *   oracle_merge     -- the exact combination of two attention states over
 *                       disjoint key sets: M = max(L_a, L_b),
 *                       Z = exp(L_a - M) + exp(L_b - M), L = M + log Z,
 *                       O = (exp(L_a - M) O_a + exp(L_b - M) O_b) / Z
 *                       ("FlashInfer 完全拆解", section 在线 Softmax 为什么
 *                       允许任意切块; "FlashInfer, in depth", section "Load
 *                       balancing with split-KV").
 *
 * Page gather: token t of request i lives in page indices[indptr[i] + t / P]
 * at slot t % P; the cache is NHD, [pages][2][P][Hkv][D] with K at index 0
 * and V at index 1 of the second dimension ("FlashInfer, in depth", section
 * "The block-sparse page table").  Query head h reads KV head h / g with
 * g = Hq / Hkv: consecutive query heads form a group (a reading; the pages
 * say a group of g query heads shares one KV head but not which ones).
 * The HND layout (layout 1 of oracle_attend_ex) swaps the last three
 * dimensions' first two: [pages][2][Hkv][P][D] ("FlashInfer 完全拆解",
 * section 接口层最容易踩的四个坑: NHD and HND differ in the order of the last
 * three dimensions); the same token, head and element are read.
 *
 * Inputs are the same bf16 bit patterns the GPU consumes, widened exactly to
 * double.  An FP8 cache (oracle_attend_ex, kv_type 1) holds E4M3 bytes --
 * 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, subnormals at
 * exponent 0, the all-ones pattern (S.1111.111) NaN, no infinities -- each
 * decoded exactly and multiplied by its tensor's scale: the attended key is
 * k_scale * K and the value v_scale * V ("FlashInfer 完全拆解", performance
 * section: E4M3 KV cache; applicability table: low-precision KV needs a
 * scale contract).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_E_ARG -1
#define ORACLE_E_TABLE -2
#define ORACLE_E_SELFCHECK -3

static double bf16_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* E4M3 byte -> double, from the format definition. */
double oracle_e4m3_to_double(uint8_t b) {
    int sign = b >> 7, e = (b >> 3) & 0xF, m = b & 7;
    double v;
    if (e == 0xF && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, 1 - 7);        /* subnormal */
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* Table check and lengths.  Returns ORACLE_OK or ORACLE_E_TABLE. */
int oracle_lengths(const int32_t *indptr, const int32_t *indices,
                   const int32_t *last, int batch, int page_size,
                   int num_pages, int64_t *lens_out) {
    if (batch < 0 || page_size < 1) return ORACLE_E_ARG;
    if (batch > 0 && indptr[0] != 0) return ORACLE_E_TABLE;
    for (int i = 0; i < batch; ++i) {
        int n = indptr[i + 1] - indptr[i];
        int r = last[i];
        if (n < 1) return ORACLE_E_TABLE;          /* l = 0 is not expressible */
        if (r < 1 || r > page_size) return ORACLE_E_TABLE;
        for (int k = indptr[i]; k < indptr[i + 1]; ++k)
            if (indices[k] < 0 || indices[k] >= num_pages) return ORACLE_E_TABLE;
        lens_out[i] = (int64_t)page_size * (n - 1) + r;
    }
    return ORACLE_OK;
}

typedef struct {
    const uint16_t *q;     /* [B][Hq][D] bf16 bits */
    const void *kv;        /* [pages][2][P][Hkv][D] bf16 bits or E4M3 bytes */
    int kv_type;           /* 0 bf16, 1 E4M3 */
    int layout;            /* 0 NHD [pages][2][P][Hkv][D], 1 HND [pages][2][Hkv][P][D] */
    double k_scale, v_scale;
    const int32_t *indptr, *indices, *last;
    int batch, hq, hkv, d, p, num_pages;
    const int32_t *rows;   /* n_rows x 4: req, head, t0, t1 (t1 < 0: to end) */
    int n_rows;
    double *out;           /* n_rows x D */
    double *lse;           /* n_rows */
    int next;              /* work counter (guarded by mu) */
    int status;
    pthread_mutex_t mu;
} job_t;

/* Element c of the K (kv = 0) or V (kv = 1) row of a page slot, decoded and
 * scaled. */
static double kv_elem(const job_t *j, int page, int kv, int slot, int kvh, int c) {
    size_t off = j->layout == 0
        ? ((((size_t)page * 2 + kv) * j->p + slot) * j->hkv + kvh) * (size_t)j->d + (size_t)c
        : ((((size_t)page * 2 + kv) * j->hkv + kvh) * j->p + slot) * (size_t)j->d + (size_t)c;
    if (j->kv_type == 1) {
        double s = kv ? j->v_scale : j->k_scale;
        return s * oracle_e4m3_to_double(((const uint8_t *)j->kv)[off]);
    }
    return (kv ? j->v_scale : j->k_scale) * bf16_to_double(((const uint16_t *)j->kv)[off]);
}

/* One query row over tokens [t0, t1).  Two passes over the keys (max, then
 * weights) so the definition is followed literally: s, m = max s,
 * Z = sum exp(s - m), O = sum exp(s - m) v / Z, L = m + log Z. */
static int attend_row(const job_t *j, int r, double *scores) {
    const int32_t *row = j->rows + 4 * (size_t)r;
    int i = row[0], h = row[1], t0 = row[2], t1 = row[3];
    int g = j->hq / j->hkv;
    int kvh = h / g;
    int n = j->indptr[i + 1] - j->indptr[i];
    int64_t len = (int64_t)j->p * (n - 1) + j->last[i];
    if (t1 < 0) t1 = (int)len;
    if (t0 < 0 || t1 > len || t0 >= t1) return ORACLE_E_ARG;
    const uint16_t *q = j->q + ((size_t)i * j->hq + h) * j->d;
    double inv_sqrt_d = 1.0 / sqrt((double)j->d);
    double m = -INFINITY;
    for (int t = t0; t < t1; ++t) {
        int page = j->indices[j->indptr[i] + t / j->p];
        double s = 0.0;
        for (int c = 0; c < j->d; ++c)
            s += bf16_to_double(q[c]) * kv_elem(j, page, 0, t % j->p, kvh, c);
        s *= inv_sqrt_d;
        scores[t - t0] = s;
        if (s > m) m = s;
    }
    double z = 0.0;
    for (int t = t0; t < t1; ++t) z += exp(scores[t - t0] - m);
    double *o = j->out + (size_t)r * j->d;
    for (int c = 0; c < j->d; ++c) o[c] = 0.0;
    double psum = 0.0;
    for (int t = t0; t < t1; ++t) {
        double w = exp(scores[t - t0] - m) / z;   /* softmax weight */
        psum += w;
        int page = j->indices[j->indptr[i] + t / j->p];
        for (int c = 0; c < j->d; ++c) o[c] += w * kv_elem(j, page, 1, t % j->p, kvh, c);
    }
    /* self-check: the softmax weights of a row sum to one */
    if (fabs(psum - 1.0) > 1e-12 * (double)(t1 - t0)) return ORACLE_E_SELFCHECK;
    j->lse[r] = m + log(z);
    return ORACLE_OK;
}

static void *worker(void *arg) {
    job_t *j = (job_t *)arg;
    int max_len = 0;
    for (int i = 0; i < j->batch; ++i) {
        int n = j->indptr[i + 1] - j->indptr[i];
        int len = j->p * (n - 1) + j->last[i];
        if (len > max_len) max_len = len;
    }
    double *scores = (double *)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
    if (!scores) {
        pthread_mutex_lock(&j->mu);
        j->status = ORACLE_E_ARG;
        pthread_mutex_unlock(&j->mu);
        return NULL;
    }
    for (;;) {
        pthread_mutex_lock(&j->mu);
        int r = j->next++;
        pthread_mutex_unlock(&j->mu);
        if (r >= j->n_rows) break;
        int st = attend_row(j, r, scores);
        if (st != ORACLE_OK) {
            pthread_mutex_lock(&j->mu);
            j->status = st;
            pthread_mutex_unlock(&j->mu);
        }
    }
    free(scores);
    return NULL;
}

/* Attention for a list of query rows (req, head, t0, t1).
 * q: [batch][hq][d] bf16 bits; kv: [num_pages][2][p][hkv][d] bf16 bits.
 * out: n_rows x d doubles; lse: n_rows doubles (natural log). */
int oracle_attend_ex(const uint16_t *q, const void *kv, int kv_type, int layout,
                     double k_scale, double v_scale, const int32_t *indptr,
                     const int32_t *indices, const int32_t *last, int batch, int hq, int hkv,
                     int d, int p, int num_pages, const int32_t *rows, int n_rows, double *out,
                     double *lse, int nthreads);

int oracle_attend(const uint16_t *q, const uint16_t *kv, const int32_t *indptr,
                  const int32_t *indices, const int32_t *last, int batch,
                  int hq, int hkv, int d, int p, int num_pages,
                  const int32_t *rows, int n_rows, double *out, double *lse,
                  int nthreads) {
    return oracle_attend_ex(q, kv, 0, 0, 1.0, 1.0, indptr, indices, last, batch, hq, hkv, d, p,
                            num_pages, rows, n_rows, out, lse, nthreads);
}

/* As oracle_attend, for a cache of kv_type (0 bf16, 1 E4M3) with scales, in
 * layout 0 (NHD) or 1 (HND). */
int oracle_attend_ex(const uint16_t *q, const void *kv, int kv_type, int layout,
                     double k_scale, double v_scale, const int32_t *indptr,
                     const int32_t *indices, const int32_t *last, int batch, int hq, int hkv,
                     int d, int p, int num_pages, const int32_t *rows, int n_rows, double *out,
                     double *lse, int nthreads) {
    if (kv_type != 0 && kv_type != 1) return ORACLE_E_ARG;
    if (layout != 0 && layout != 1) return ORACLE_E_ARG;
    if (hq < 1 || hkv < 1 || hq % hkv != 0 || d < 1 || p < 1) return ORACLE_E_ARG;
    int64_t *lens = (int64_t *)malloc(sizeof(int64_t) * (size_t)(batch > 0 ? batch : 1));
    if (!lens) return ORACLE_E_ARG;
    int st = oracle_lengths(indptr, indices, last, batch, p, num_pages, lens);
    free(lens);
    if (st != ORACLE_OK) return st;
    for (int r = 0; r < n_rows; ++r) {
        if (rows[4 * r] < 0 || rows[4 * r] >= batch) return ORACLE_E_ARG;
        if (rows[4 * r + 1] < 0 || rows[4 * r + 1] >= hq) return ORACLE_E_ARG;
    }
    job_t j;
    memset(&j, 0, sizeof j);
    j.q = q; j.kv = kv; j.kv_type = kv_type; j.layout = layout;
    j.k_scale = k_scale; j.v_scale = v_scale;
    j.indptr = indptr; j.indices = indices; j.last = last;
    j.batch = batch; j.hq = hq; j.hkv = hkv; j.d = d; j.p = p;
    j.num_pages = num_pages; j.rows = rows; j.n_rows = n_rows;
    j.out = out; j.lse = lse; j.next = 0; j.status = ORACLE_OK;
    pthread_mutex_init(&j.mu, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (nthreads > n_rows) nthreads = n_rows > 0 ? n_rows : 1;
    pthread_t th[256];
    int started = 0;
    for (int t = 1; t < nthreads; ++t)
        if (pthread_create(&th[started], NULL, worker, &j) == 0) ++started;
    worker(&j);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    pthread_mutex_destroy(&j.mu);
    return j.status;
}

/* Merge of two attention states, elementwise over n rows of width d.
 * A state with lse = -inf is empty; merging two empty states gives an empty
 * state with a zero output. */
int oracle_merge(const double *o_a, const double *l_a, const double *o_b,
                 const double *l_b, int n, int d, double *o_out, double *l_out) {
    for (int r = 0; r < n; ++r) {
        double la = l_a[r], lb = l_b[r];
        double *o = o_out + (size_t)r * d;
        if (isinf(la) && la < 0 && isinf(lb) && lb < 0) {
            for (int c = 0; c < d; ++c) o[c] = 0.0;
            l_out[r] = -INFINITY;
            continue;
        }
        double m = la > lb ? la : lb;
        double wa = exp(la - m), wb = exp(lb - m);
        double z = wa + wb;
        for (int c = 0; c < d; ++c)
            o[c] = (wa * o_a[(size_t)r * d + c] + wb * o_b[(size_t)r * d + c]) / z;
        l_out[r] = m + log(z);
    }
    return ORACLE_OK;
}
