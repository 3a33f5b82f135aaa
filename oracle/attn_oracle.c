/*
 * attn_oracle.c -- plain CPU oracle for the attention forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: it is used by the tests, by the smoke check and by the
 * bench's CPU-baseline leg, and it shares no code with the CUDA library.
 *
 * What it computes (the definition, not the tiled algorithm):
 *   for every (b, h) and query row i, over the visible keys j
 *     s_ij  = scale * sum_d q_id * k_jd                       (step 1)
 *     m_i   = max_j s_ij,  p_ij = exp(s_ij - m_i) / l_i,
 *     l_i   = sum_j exp(s_ij - m_i)                           (step 2)
 *     O_i   = sum_j p_ij * v_j,   LSE_i = m_i + ln(l_i)       (step 3)
 *   This is the naive three-step attention (full score row, max-subtracted
 *   softmax, then P.V) that "The FA5090 Optimization Journey" starts from in
 *   section 2.2 (v0: the score matrix materialised, online softmax only for
 *   overflow safety) and that every FlashAttention variant on the pages reaches
 *   through the online-softmax identity.  The pages never write the formula or
 *   LSE down; LSE is read here as the natural-log log-sum-exp of the scaled
 *   scores, m_i + ln l_i.
 *
 * Causal masking is bottom-right aligned: key j is visible from query i iff
 * j <= i + (Skv - Sq).  A row with no visible key gets O = 0 and LSE = -inf.
 *
 * Two references live here:
 *   oracle_attention_rows : fp64 throughout (the oracle proper);
 *   floor_attention_rows  : the same three steps in fp32 on the 16-bit inputs,
 *                           with the normalised P and the output rounded to the
 *                           input format (round to nearest even).  It measures
 *                           the error that any correct same-precision
 *                           implementation is entitled to; the tolerance
 *                           rule of section 2.1 of the FA5090 page scales
 *                           its bound from this per-configuration error.
 *
 * Layout: Q [B,H,Sq,D], K and V [B,H,Skv,D], row-major, contiguous.
 * Rows are addressed by their flat index r = (b*H + h)*Sq + i.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Last key index visible from query row i (inclusive); negative if none. */
static long last_visible_key(long i, long Sq, long Skv, int causal)
{
    long last = Skv - 1;
    if (causal) {
        long diag = i + (Skv - Sq);
        if (diag < last) last = diag;
    }
    return last;
}

/* ------------------------------------------------------------------ fp64 */

/* Steps 1 and 2 for one row: writes the normalised probabilities p[0..n) for
 * the n visible keys and returns m and l through the pointers. */
static void row_probs_f64(const double *q, const double *K, long n, long D,
                          double scale, double *p, double *m_out, double *l_out)
{
    /* step 1: scaled scores */
    for (long j = 0; j < n; ++j) {
        double dot = 0.0;
        for (long d = 0; d < D; ++d) dot += q[d] * K[j * D + d];
        p[j] = scale * dot;
    }
    /* step 2: softmax with the row maximum subtracted */
    double m = p[0];
    for (long j = 1; j < n; ++j)
        if (p[j] > m) m = p[j];
    double l = 0.0;
    for (long j = 0; j < n; ++j) {
        p[j] = exp(p[j] - m);
        l += p[j];
    }
    for (long j = 0; j < n; ++j) p[j] /= l;
    *m_out = m;
    *l_out = l;
}

static void attend_row_f64(const double *q, const double *K, const double *V,
                           long n, long D, double scale, double *o,
                           double *lse, double *scratch)
{
    if (n <= 0) {
        for (long d = 0; d < D; ++d) o[d] = 0.0;
        *lse = -INFINITY;
        return;
    }
    double m, l;
    row_probs_f64(q, K, n, D, scale, scratch, &m, &l);
    /* step 3: O = P V */
    for (long d = 0; d < D; ++d) o[d] = 0.0;
    for (long j = 0; j < n; ++j) {
        const double pj = scratch[j];
        for (long d = 0; d < D; ++d) o[d] += pj * V[j * D + d];
    }
    *lse = m + log(l);
}

/* -------------------------------------------------------- 16-bit rounding */

/* Round x to the nearest value of a binary format with `mant` explicit
 * mantissa bits and minimum normal exponent `emin` (ties to even, gradual
 * underflow).  fp16: mant 10, emin -14.  bf16: mant 7, emin -126.  Values are
 * far from either format's overflow threshold here, so overflow is not
 * handled. */
static double round_to_format(double x, int mant, int emin)
{
    if (x == 0.0 || !isfinite(x)) return x;
    int e;
    frexp(x, &e);                 /* |x| in [2^(e-1), 2^e) */
    int E = e - 1;
    if (E < emin) E = emin;       /* subnormal range: fixed spacing */
    const double ulp = ldexp(1.0, E - mant);
    return nearbyint(x / ulp) * ulp;   /* default rounding mode: ties to even */
}

/* fmt: 0 = fp16, 1 = bf16 */
static float round_f32_to_fmt(float x, int fmt)
{
    return fmt == 1 ? (float)round_to_format((double)x, 7, -126)
                    : (float)round_to_format((double)x, 10, -14);
}

/* The floor reference for one row, in fp32 arithmetic. */
static void attend_row_floor(const float *q, const float *K, const float *V,
                             long n, long D, float scale, int fmt, float *o,
                             float *lse, float *p)
{
    if (n <= 0) {
        for (long d = 0; d < D; ++d) o[d] = 0.0f;
        *lse = -INFINITY;
        return;
    }
    for (long j = 0; j < n; ++j) {
        float dot = 0.0f;
        for (long d = 0; d < D; ++d) dot += q[d] * K[j * D + d];
        p[j] = scale * dot;
    }
    float m = p[0];
    for (long j = 1; j < n; ++j)
        if (p[j] > m) m = p[j];
    float l = 0.0f;
    for (long j = 0; j < n; ++j) {
        p[j] = expf(p[j] - m);
        l += p[j];
    }
    for (long j = 0; j < n; ++j) p[j] = round_f32_to_fmt(p[j] / l, fmt);
    for (long d = 0; d < D; ++d) o[d] = 0.0f;
    for (long j = 0; j < n; ++j)
        for (long d = 0; d < D; ++d) o[d] += p[j] * V[j * D + d];
    for (long d = 0; d < D; ++d) o[d] = round_f32_to_fmt(o[d], fmt);
    *lse = m + logf(l);
}

/* ----------------------------------------------------------- row workers */

typedef struct {
    const void *q, *k, *v;
    long B, H, Sq, Skv, D;
    double scale;
    int causal;
    int fmt;                 /* floor only */
    const int64_t *rows;     /* NULL: all rows in order */
    long nrows;
    void *o, *lse;
    long begin, end;         /* slice of [0, nrows) for this worker */
    int is_floor;
    int status;
} job_t;

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    const long D = J->D;
    void *scratch = malloc((size_t)(J->Skv > 0 ? J->Skv : 1) *
                           (J->is_floor ? sizeof(float) : sizeof(double)));
    if (!scratch) {
        J->status = -1;
        return NULL;
    }
    for (long t = J->begin; t < J->end; ++t) {
        const long r = J->rows ? (long)J->rows[t] : t;
        const long bh = r / J->Sq, i = r % J->Sq;
        const long n = last_visible_key(i, J->Sq, J->Skv, J->causal) + 1;
        const long qoff = r * D, kvoff = bh * J->Skv * D;
        if (J->is_floor) {
            attend_row_floor((const float *)J->q + qoff,
                             (const float *)J->k + kvoff,
                             (const float *)J->v + kvoff, n, D,
                             (float)J->scale, J->fmt,
                             (float *)J->o + t * D, (float *)J->lse + t,
                             (float *)scratch);
        } else {
            attend_row_f64((const double *)J->q + qoff,
                           (const double *)J->k + kvoff,
                           (const double *)J->v + kvoff, n, D, J->scale,
                           (double *)J->o + t * D, (double *)J->lse + t,
                           (double *)scratch);
        }
    }
    free(scratch);
    J->status = 0;
    return NULL;
}

static int run_rows(job_t proto, int nthreads)
{
    if (proto.B <= 0 || proto.H <= 0 || proto.Sq <= 0 || proto.Skv < 0 ||
        proto.D <= 0)
        return -2;
    if (!proto.rows) proto.nrows = proto.B * proto.H * proto.Sq;
    if (proto.rows) {
        const long total = proto.B * proto.H * proto.Sq;
        for (long t = 0; t < proto.nrows; ++t)
            if (proto.rows[t] < 0 || proto.rows[t] >= total) return -3;
    }
    if (nthreads < 1) nthreads = 1;
    if (nthreads > proto.nrows) nthreads = proto.nrows > 0 ? (int)proto.nrows : 1;
    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) {
        free(jobs);
        free(tids);
        return -1;
    }
    int rc = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = proto;
        jobs[t].begin = proto.nrows * t / nthreads;
        jobs[t].end = proto.nrows * (t + 1) / nthreads;
        jobs[t].status = -1;
        if (pthread_create(&tids[t], NULL, worker, &jobs[t]) != 0) {
            worker(&jobs[t]);   /* run inline if a thread cannot start */
            tids[t] = 0;
        }
    }
    for (int t = 0; t < nthreads; ++t) {
        if (tids[t]) pthread_join(tids[t], NULL);
        if (jobs[t].status != 0) rc = -1;
    }
    free(jobs);
    free(tids);
    return rc;
}

/* ------------------------------------------------------------ public API */

/* fp64 oracle over the rows listed in `rows` (flat indices into [B,H,Sq]), or
 * over every row in order when rows == NULL.  o: [nrows, D], lse: [nrows].
 * Returns 0 on success, negative on bad arguments or allocation failure. */
int oracle_attention_rows(const double *q, const double *k, const double *v,
                          long B, long H, long Sq, long Skv, long D,
                          double scale, int causal, const int64_t *rows,
                          long nrows, double *o, double *lse, int nthreads)
{
    job_t J;
    memset(&J, 0, sizeof J);
    J.q = q; J.k = k; J.v = v;
    J.B = B; J.H = H; J.Sq = Sq; J.Skv = Skv; J.D = D;
    J.scale = scale; J.causal = causal;
    J.rows = rows; J.nrows = nrows; J.o = o; J.lse = lse;
    J.is_floor = 0;
    return run_rows(J, nthreads);
}

/* fp32 floor reference, same conventions; fmt 0 = fp16, 1 = bf16.  Inputs are
 * the 16-bit values widened to fp32 (exact). */
int floor_attention_rows(const float *q, const float *k, const float *v,
                         long B, long H, long Sq, long Skv, long D,
                         float scale, int causal, int fmt, const int64_t *rows,
                         long nrows, float *o, float *lse, int nthreads)
{
    if (fmt != 0 && fmt != 1) return -2;
    job_t J;
    memset(&J, 0, sizeof J);
    J.q = q; J.k = k; J.v = v;
    J.B = B; J.H = H; J.Sq = Sq; J.Skv = Skv; J.D = D;
    J.scale = scale; J.causal = causal; J.fmt = fmt;
    J.rows = rows; J.nrows = nrows; J.o = o; J.lse = lse;
    J.is_floor = 1;
    return run_rows(J, nthreads);
}

/* The normalised probability matrix P [Sq, Skv] of one head (zeros at masked
 * positions), from steps 1 and 2 of the fp64 oracle.  For small checks. */
int oracle_probs(const double *q, const double *k, long Sq, long Skv, long D,
                 double scale, int causal, double *P)
{
    if (Sq <= 0 || Skv <= 0 || D <= 0) return -2;
    double *row = (double *)malloc((size_t)Skv * sizeof(double));
    if (!row) return -1;
    for (long i = 0; i < Sq; ++i) {
        const long n = last_visible_key(i, Sq, Skv, causal) + 1;
        for (long j = 0; j < Skv; ++j) P[i * Skv + j] = 0.0;
        if (n <= 0) continue;
        double m, l;
        row_probs_f64(q + i * D, k, n, D, scale, row, &m, &l);
        for (long j = 0; j < n; ++j) P[i * Skv + j] = row[j];
    }
    free(row);
    return 0;
}

/* Round each of n fp32 values to fp16 (fmt 0) or bf16 (fmt 1), in place. */
void oracle_round_fmt(float *x, long n, int fmt)
{
    for (long t = 0; t < n; ++t) x[t] = round_f32_to_fmt(x[t], fmt);
}
