/*
 * Continuous Softmax Attention: CPU oracle, double precision.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark load this file's library.  The CUDA
 * library never calls it, and it shares no code with the CUDA library.
 *
 * Source: Jianlin Su, "Continuous Softmax Attention" (Scientific Spaces
 * #11980, English translation), sections "Problem Statement",
 * "Preliminaries", "Assembly and Simplification", "Analysis of the Result",
 * equations (1)-(13).  Standard causal attention follows the same page's
 * eq. (12) and S. K. Sahu, "Attention, from the softmax up", section
 * "The one line".
 *
 * Conventions used by every entry point:
 *   q, k, v      float32, contiguous [B, H, T, d].  Values are widened to
 *                double before any arithmetic (bf16 inputs arrive here as
 *                their exactly representable float32 values).
 *   k0, v0       float32 [H, d], read only when k0_mode == 2 (given).
 *   out          double [B, H, T, d];  lse  double [B, H, T] (may be NULL).
 *   Array row r is the page's token t = r + 1; array key j is the page's
 *   key i = j + 1; the page's k_0, v_0 are the separate sink vectors.
 *   Logits are a_{t,i} = scale * q_t . k_i.
 *   k0_mode: 0 = zero vectors, 1 = copy of the first token (k_0 = k_1,
 *   v_0 = v_1), 2 = given per-head vectors (the three choices listed at the
 *   end of "Analysis of the Result").
 * Return value: 0 on success, -1 on a bad argument.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_ZERO 0
#define ORACLE_COPY_FIRST 1
#define ORACLE_GIVEN 2

/* ------------------------------------------------------------------------
 * phi_1, phi_2 of eq. (6):  phi1(x) = int_0^1 e^{sx} ds = (e^x - 1)/x,
 * phi2(x) = int_0^1 e^{sx}(1-s) ds = (e^x - 1 - x)/x^2, with the limits
 * phi1(0) = 1 and phi2(0) = 1/2 stated right after eq. (6).
 * Near 0 the closed forms cancel, so |x| < 0.1 uses the power series that
 * follows from expanding e^{sx} under the integral:
 *   phi1(x) = sum_n x^n/(n+1)!,   phi2(x) = sum_n x^n/(n+2)!.
 * Fourteen terms leave a truncation error below 1e-28 at |x| = 0.1.
 * ---------------------------------------------------------------------- */
static double series_phi(double x, int shift)
{
    /* sum_{n=0}^{13} x^n / (n+shift)!  evaluated by Horner's rule */
    double c[14];
    double f = 1.0;
    for (int i = 1; i <= shift; ++i) f *= (double)i;
    for (int n = 0; n < 14; ++n) {
        if (n > 0) f *= (double)(n + shift);
        c[n] = 1.0 / f;
    }
    double acc = c[13];
    for (int n = 12; n >= 0; --n) acc = acc * x + c[n];
    return acc;
}

double csa_oracle_phi1(double x)
{
    if (fabs(x) < 0.1) return series_phi(x, 1);
    return expm1(x) / x;
}

double csa_oracle_phi2(double x)
{
    if (fabs(x) < 0.1) return series_phi(x, 2);
    return (expm1(x) - x) / (x * x);
}

/* log phi1, log phi2 without overflow for large positive x:
 *   x > 1:  phi1 = e^x (1 - e^{-x}) / x,  phi2 = e^x (1 - (1+x) e^{-x}) / x^2
 * so the logs are x + log1p(-...) - log x (or 2 log x).  phi1, phi2 > 0 for
 * every real x (both are integrals of positive functions, end of
 * "Preliminaries"), so the logs are always finite. */
double csa_oracle_log_phi1(double x)
{
    if (x > 1.0) return x + log1p(-exp(-x)) - log(x);
    if (x < -1.0) return log(-expm1(x)) - log(-x);
    return log(csa_oracle_phi1(x));
}

double csa_oracle_log_phi2(double x)
{
    if (x > 1.0) return x + log1p(-(1.0 + x) * exp(-x)) - 2.0 * log(x);
    if (x < -1.0) return log(expm1(x) - x) - 2.0 * log(-x);
    return log(csa_oracle_phi2(x));
}

/* ------------------------------------------------------------------------
 * Shared argument block and per-row helpers.
 * ---------------------------------------------------------------------- */
typedef struct {
    const float *q, *k, *v, *k0, *v0;
    double *out, *lse;
    int B, H, T, d;
    double scale;
    int mode;
    /* explicit row list (NULL = all rows) */
    const long long *rows;
    long long nrows;
    int form; /* 0 = eq.(8), 1 = eq.(11), 2 = eq.(12) standard, 3 = eq.(13) short conv,
               * 4 = eq.(8) over the symmetric interval [1/2, t + 1/2] */
} job_t;

typedef struct {
    const job_t *job;
    int index, count; /* this worker's index and the number of workers */
    int status;
} slice_t;

static double dot_fd(const float *x, const double *y, int d)
{
    double s = 0.0;
    for (int c = 0; c < d; ++c) s += (double)x[c] * y[c];
    return s;
}

/* Extended key/value sequence of row (bh, r): index 0 is the sink, index
 * i >= 1 is array key i-1 (page key i).  Fills a[0..t] with the logits. */
static const float *key_ptr(const job_t *jb, long long bh, int i, int h, const float *zero)
{
    if (i >= 1) return jb->k + ((size_t)bh * jb->T + (size_t)(i - 1)) * jb->d;
    if (jb->mode == ORACLE_COPY_FIRST) return jb->k + (size_t)bh * jb->T * jb->d;
    if (jb->mode == ORACLE_GIVEN) return jb->k0 + (size_t)h * jb->d;
    return zero;
}

static const float *val_ptr(const job_t *jb, long long bh, int i, int h, const float *zero)
{
    if (i >= 1) return jb->v + ((size_t)bh * jb->T + (size_t)(i - 1)) * jb->d;
    if (jb->mode == ORACLE_COPY_FIRST) return jb->v + (size_t)bh * jb->T * jb->d;
    if (jb->mode == ORACLE_GIVEN) return jb->v0 + (size_t)h * jb->d;
    return zero;
}

/* One output row.  buf holds (T+1) doubles of logits plus d doubles of
 * scratch for q and d doubles for the numerator. */
static void one_row(const job_t *jb, long long flat, double *out_row, double *lse_out,
                    double *a, double *qd, double *num, const float *zero)
{
    const int T = jb->T, d = jb->d;
    const long long bh = flat / T;
    const int r = (int)(flat % T);
    const int h = (int)(bh % jb->H);
    const float *qr = jb->q + ((size_t)bh * T + (size_t)r) * d;
    for (int c = 0; c < d; ++c) qd[c] = (double)qr[c];
    for (int c = 0; c < d; ++c) num[c] = 0.0;

    if (jb->form == 2) {
        /* eq.(12): o_t = sum_{i=1}^t e^{a_{t,i}} v_i / sum_{i=1}^t e^{a_{t,i}} */
        const int t = r + 1;
        double m = -INFINITY;
        for (int i = 1; i <= t; ++i) {
            a[i] = jb->scale * dot_fd(key_ptr(jb, bh, i, h, zero), qd, d);
            if (a[i] > m) m = a[i];
        }
        double den = 0.0;
        for (int i = 1; i <= t; ++i) {
            const double w = exp(a[i] - m);
            const float *vi = val_ptr(jb, bh, i, h, zero);
            for (int c = 0; c < d; ++c) num[c] += w * (double)vi[c];
            den += w;
        }
        for (int c = 0; c < d; ++c) out_row[c] = num[c] / den;
        if (lse_out) *lse_out = m + log(den);
        return;
    }

    if (jb->form == 4) {
        /* The symmetric interval [1/2, t + 1/2] of the original Continuum
         * Attention paper ("Problem Statement"): eq. (2)'s integrals with
         * eq. (3) inside [1, t] and constant half-cells [1/2, 1] (k_1, v_1)
         * and [t, t + 1/2] (k_t, v_t), since a causal row has no k_{t+1}; no
         * sink.  Segment i = 2..t contributes as in eq. (8); each half-cell
         * contributes e^{a} v / 2 and e^{a} / 2. */
        const int t = r + 1;
        double m = -INFINITY;
        for (int i = 1; i <= t; ++i) {
            a[i] = jb->scale * dot_fd(key_ptr(jb, bh, i, h, zero), qd, d);
            if (a[i] > m) m = a[i];
        }
        const float *v1 = val_ptr(jb, bh, 1, h, zero), *vt = val_ptr(jb, bh, t, h, zero);
        const double h1 = 0.5 * exp(a[1] - m), ht = 0.5 * exp(a[t] - m);
        double den = h1 + ht;
        for (int c = 0; c < d; ++c) num[c] = h1 * (double)v1[c] + ht * (double)vt[c];
        for (int i = 2; i <= t; ++i) {
            const double delta = a[i] - a[i - 1];
            const double e1 = exp(a[i - 1] - m + csa_oracle_log_phi1(delta));
            const double e2 = exp(a[i - 1] - m + csa_oracle_log_phi2(delta));
            const float *vi = val_ptr(jb, bh, i, h, zero);
            const float *vp = val_ptr(jb, bh, i - 1, h, zero);
            for (int c = 0; c < d; ++c)
                num[c] += e1 * (double)vi[c] + e2 * ((double)vp[c] - (double)vi[c]);
            den += e1;
        }
        for (int c = 0; c < d; ++c) out_row[c] = num[c] / den;
        if (lse_out) *lse_out = m + log(den);
        return;
    }

    /* Page token t = r + 1 sees keys i = 0..t (k_0 included). */
    const int t = r + 1;
    double m = -INFINITY;
    for (int i = 0; i <= t; ++i) {
        a[i] = jb->scale * dot_fd(key_ptr(jb, bh, i, h, zero), qd, d);
        if (a[i] > m) m = a[i];
    }

    if (jb->form == 0) {
        /* eq.(8): segment i in 1..t contributes, by eq.(4)/(5),
         *   numerator   e^{a_{i-1}} phi1(delta_i) v_i + e^{a_{i-1}} phi2(delta_i) (v_{i-1} - v_i)
         *   denominator e^{a_{i-1}} phi1(delta_i)
         * with delta_i = a_i - a_{i-1}; everything is scaled by e^{-m}. */
        double den = 0.0;
        for (int i = 1; i <= t; ++i) {
            const double delta = a[i] - a[i - 1];
            const double e1 = exp(a[i - 1] - m + csa_oracle_log_phi1(delta));
            const double e2 = exp(a[i - 1] - m + csa_oracle_log_phi2(delta));
            const float *vi = val_ptr(jb, bh, i, h, zero);
            const float *vp = val_ptr(jb, bh, i - 1, h, zero);
            for (int c = 0; c < d; ++c)
                num[c] += e1 * (double)vi[c] + e2 * ((double)vp[c] - (double)vi[c]);
            den += e1;
        }
        for (int c = 0; c < d; ++c) out_row[c] = num[c] / den;
        if (lse_out) *lse_out = m + log(den);
        return;
    }

    if (jb->form == 3) {
        /* The short-conv reading of eq.(13): b replaced by its first-order
         * Taylor term.  Interior keys: log(phi2(x) + phi2(y)) with
         * phi2(x) = 1/2 + x/6 + O(x^2) gives b_i = (a_{i-1} + a_{i+1} - 2 a_i)/6;
         * the end keys (one phi2 each): log phi2(x) = -log 2 + x/3 + O(x^2)
         * gives b_0 = -log 2 + (a_1 - a_0)/3, b_t = -log 2 + (a_{t-1} - a_t)/3.
         * Then a plain two-pass softmax over z = a + b. */
        double zmax = -INFINITY;
        double *z = a + (t + 1);
        for (int i = 0; i <= t; ++i) {
            double b;
            if (i == 0)
                b = -log(2.0) + (a[1] - a[0]) / 3.0;
            else if (i == t)
                b = -log(2.0) + (a[t - 1] - a[t]) / 3.0;
            else
                b = (a[i - 1] + a[i + 1] - 2.0 * a[i]) / 6.0;
            z[i] = a[i] + b;
            if (z[i] > zmax) zmax = z[i];
        }
        double den = 0.0;
        for (int i = 0; i <= t; ++i) {
            const double w = exp(z[i] - zmax);
            const float *vi = val_ptr(jb, bh, i, h, zero);
            for (int c = 0; c < d; ++c) num[c] += w * (double)vi[c];
            den += w;
        }
        for (int c = 0; c < d; ++c) out_row[c] = num[c] / den;
        if (lse_out) *lse_out = zmax + log(den);
        return;
    }

    /* eq.(10)/(11): z_i = a_i + b_i with
     *   e^{b_0} = phi2(a_1 - a_0),  e^{b_t} = phi2(a_{t-1} - a_t),
     *   e^{b_i} = phi2(a_{i-1} - a_i) + phi2(a_{i+1} - a_i)  (1 <= i <= t-1);
     * the sum inside the log is formed with logaddexp.  Then a plain
     * two-pass softmax over z. */
    double zmax = -INFINITY;
    double *z = a + (t + 1); /* second half of the buffer */
    for (int i = 0; i <= t; ++i) {
        double b;
        if (i == 0) {
            b = csa_oracle_log_phi2(a[1] - a[0]);
        } else if (i == t) {
            b = csa_oracle_log_phi2(a[t - 1] - a[t]);
        } else {
            const double l1 = csa_oracle_log_phi2(a[i - 1] - a[i]);
            const double l2 = csa_oracle_log_phi2(a[i + 1] - a[i]);
            const double hi = l1 > l2 ? l1 : l2, lo = l1 > l2 ? l2 : l1;
            b = hi + log1p(exp(lo - hi));
        }
        z[i] = a[i] + b;
        if (z[i] > zmax) zmax = z[i];
    }
    double den = 0.0;
    for (int i = 0; i <= t; ++i) {
        const double w = exp(z[i] - zmax);
        const float *vi = val_ptr(jb, bh, i, h, zero);
        for (int c = 0; c < d; ++c) num[c] += w * (double)vi[c];
        den += w;
    }
    for (int c = 0; c < d; ++c) out_row[c] = num[c] / den;
    if (lse_out) *lse_out = zmax + log(den);
}

static void *run_slice(void *arg)
{
    slice_t *s = (slice_t *)arg;
    const job_t *jb = s->job;
    const int d = jb->d;
    double *buf = (double *)malloc(sizeof(double) * (2 * ((size_t)jb->T + 2) + 2 * (size_t)d));
    float *zero = (float *)calloc((size_t)d, sizeof(float));
    if (!buf || !zero) {
        free(buf);
        free(zero);
        s->status = -2;
        return NULL;
    }
    double *a = buf;
    double *qd = buf + 2 * ((size_t)jb->T + 2);
    double *num = qd + d;
    const long long total = jb->rows ? jb->nrows : (long long)jb->B * jb->H * jb->T;
    /* Causal rows cost in proportion to their index, so workers take
     * blocks of 16 rows round-robin. */
    for (long long blk = s->index; blk * 16 < total; blk += s->count) {
      for (long long n = blk * 16; n < total && n < blk * 16 + 16; ++n) {
        long long flat = jb->rows ? jb->rows[n] : n;
        double *orow = jb->out + (size_t)n * d;
        double *lrow = jb->lse ? jb->lse + n : NULL;
        one_row(jb, flat, orow, lrow, a, qd, num, zero);
      }
    }
    free(buf);
    free(zero);
    s->status = 0;
    return NULL;
}

static int run_job(const job_t *jb, int nthreads)
{
    const long long total = jb->rows ? jb->nrows : (long long)jb->B * jb->H * jb->T;
    if (total == 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 1024) nthreads = 1024;
    if ((long long)nthreads * 16 > total) nthreads = (int)((total + 15) / 16);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    slice_t *sl = (slice_t *)malloc(sizeof(slice_t) * (size_t)nthreads);
    if (!th || !sl) {
        free(th);
        free(sl);
        return -2;
    }
    int rc = 0;
    unsigned char *joined = (unsigned char *)calloc((size_t)nthreads, 1);
    if (!joined) {
        free(th);
        free(sl);
        return -2;
    }
    for (int i = 0; i < nthreads; ++i) {
        sl[i].job = jb;
        sl[i].index = i;
        sl[i].count = nthreads;
        sl[i].status = 0;
    }
    for (int i = 0; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, run_slice, &sl[i]) == 0) {
            joined[i] = 1;
        } else {
            run_slice(&sl[i]); /* no thread available: run it here */
        }
    }
    for (int i = 0; i < nthreads; ++i)
        if (joined[i]) pthread_join(th[i], NULL);
    for (int i = 0; i < nthreads; ++i)
        if (sl[i].status != 0) rc = sl[i].status;
    free(joined);
    free(th);
    free(sl);
    return rc;
}

static int check_args(const float *q, const float *k, const float *v, const float *k0, const float *v0,
                      double *out, int B, int H, int T, int d, int mode)
{
    if (B < 0 || H < 0 || T < 0 || d < 1) return -1;
    if ((long long)B * H * T > 0 && (!q || !k || !v || !out)) return -1;
    if (mode < 0 || mode > 2) return -1;
    if (mode == ORACLE_GIVEN && (!k0 || !v0)) return -1;
    return 0;
}

static int forward_common(const float *q, const float *k, const float *v, const float *k0,
                          const float *v0, double *out, double *lse, int B, int H, int T, int d,
                          double scale, int mode, const long long *rows, long long nrows,
                          int form, int nthreads)
{
    if (check_args(q, k, v, k0, v0, out, B, H, T, d, mode) != 0) return -1;
    if (rows) {
        const long long total = (long long)B * H * T;
        for (long long n = 0; n < nrows; ++n)
            if (rows[n] < 0 || rows[n] >= total) return -1;
    }
    job_t jb;
    memset(&jb, 0, sizeof(jb));
    jb.q = q; jb.k = k; jb.v = v; jb.k0 = k0; jb.v0 = v0;
    jb.out = out; jb.lse = lse;
    jb.B = B; jb.H = H; jb.T = T; jb.d = d;
    jb.scale = scale; jb.mode = mode;
    jb.rows = rows; jb.nrows = nrows; jb.form = form;
    return run_job(&jb, nthreads);
}

/* Continuous attention by the segment sum of eq.(8). */
int csa_oracle_forward(const float *q, const float *k, const float *v, const float *k0,
                       const float *v0, double *out, double *lse, int B, int H, int T, int d,
                       double scale, int k0_mode, int nthreads)
{
    return forward_common(q, k, v, k0, v0, out, lse, B, H, T, d, scale, k0_mode, NULL, 0, 0, nthreads);
}

/* Continuous attention by the simplified softmax form of eq.(10)/(11). */
int csa_oracle_forward_eq11(const float *q, const float *k, const float *v, const float *k0,
                            const float *v0, double *out, double *lse, int B, int H, int T, int d,
                            double scale, int k0_mode, int nthreads)
{
    return forward_common(q, k, v, k0, v0, out, lse, B, H, T, d, scale, k0_mode, NULL, 0, 1, nthreads);
}

/* The short-conv reading of eq.(13): b replaced by its first-order term. */
int csa_oracle_forward_short_conv(const float *q, const float *k, const float *v, const float *k0,
                                  const float *v0, double *out, double *lse, int B, int H, int T,
                                  int d, double scale, int k0_mode, int nthreads)
{
    return forward_common(q, k, v, k0, v0, out, lse, B, H, T, d, scale, k0_mode, NULL, 0, 3, nthreads);
}

/* eq.(13) short conv for a list of rows only. */
int csa_oracle_forward_short_conv_rows(const float *q, const float *k, const float *v,
                                       const float *k0, const float *v0, const long long *rows,
                                       long long nrows, double *out, double *lse, int B, int H,
                                       int T, int d, double scale, int k0_mode, int nthreads)
{
    if (!rows && nrows > 0) return -1;
    return forward_common(q, k, v, k0, v0, out, lse, B, H, T, d, scale, k0_mode, rows, nrows, 3, nthreads);
}

/* eq.(8) over the symmetric interval [1/2, t + 1/2], no sink. */
int csa_oracle_forward_symmetric(const float *q, const float *k, const float *v, double *out,
                                 double *lse, int B, int H, int T, int d, double scale,
                                 int nthreads)
{
    return forward_common(q, k, v, NULL, NULL, out, lse, B, H, T, d, scale, 0, NULL, 0, 4, nthreads);
}

/* The symmetric interval for a list of rows only. */
int csa_oracle_forward_symmetric_rows(const float *q, const float *k, const float *v,
                                      const long long *rows, long long nrows, double *out,
                                      double *lse, int B, int H, int T, int d, double scale,
                                      int nthreads)
{
    if (!rows && nrows > 0) return -1;
    return forward_common(q, k, v, NULL, NULL, out, lse, B, H, T, d, scale, 0, rows, nrows, 4, nthreads);
}

/* Standard causal softmax attention, eq.(12). */
int csa_oracle_std_forward(const float *q, const float *k, const float *v, double *out,
                           double *lse, int B, int H, int T, int d, double scale, int nthreads)
{
    return forward_common(q, k, v, NULL, NULL, out, lse, B, H, T, d, scale, 0, NULL, 0, 2, nthreads);
}

/* eq.(8) for a list of rows only: rows[n] = (b*H + h)*T + r;
 * out is [nrows, d], lse is [nrows]. */
int csa_oracle_forward_rows(const float *q, const float *k, const float *v, const float *k0,
                            const float *v0, const long long *rows, long long nrows, double *out,
                            double *lse, int B, int H, int T, int d, double scale, int k0_mode,
                            int nthreads)
{
    if (!rows && nrows > 0) return -1;
    return forward_common(q, k, v, k0, v0, out, lse, B, H, T, d, scale, k0_mode, rows, nrows, 0, nthreads);
}

/* eq.(12) for a list of rows only. */
int csa_oracle_std_forward_rows(const float *q, const float *k, const float *v, const long long *rows,
                                long long nrows, double *out, double *lse, int B, int H, int T, int d,
                                double scale, int nthreads)
{
    if (!rows && nrows > 0) return -1;
    return forward_common(q, k, v, NULL, NULL, out, lse, B, H, T, d, scale, 0, rows, nrows, 2, nthreads);
}

/* Logits a_{t,0..t} and corrections b_{t,0..t} (eq.(10)) of one row, for
 * the tests of the Taylor form (13) and the sink cases.  a_out and b_out
 * must hold r + 2 doubles. */
int csa_oracle_row_bias(const float *q, const float *k, const float *k0, int B, int H, int T, int d,
                        double scale, int k0_mode, int b, int h, int r, double *a_out, double *b_out)
{
    if (check_args(q, k, k, k0, k0, a_out, B, H, T, d, k0_mode) != 0) return -1;
    if (b < 0 || b >= B || h < 0 || h >= H || r < 0 || r >= T || !b_out) return -1;
    job_t jb;
    memset(&jb, 0, sizeof(jb));
    jb.q = q; jb.k = k; jb.k0 = k0;
    jb.B = B; jb.H = H; jb.T = T; jb.d = d; jb.scale = scale; jb.mode = k0_mode;
    float *zero = (float *)calloc((size_t)d, sizeof(float));
    double *qd = (double *)malloc(sizeof(double) * (size_t)d);
    if (!zero || !qd) {
        free(zero);
        free(qd);
        return -2;
    }
    const long long bh = (long long)b * H + h;
    const float *qr = q + ((size_t)bh * T + (size_t)r) * d;
    for (int c = 0; c < d; ++c) qd[c] = (double)qr[c];
    const int t = r + 1;
    for (int i = 0; i <= t; ++i) a_out[i] = scale * dot_fd(key_ptr(&jb, bh, i, h, zero), qd, d);
    for (int i = 0; i <= t; ++i) {
        if (i == 0) {
            b_out[i] = csa_oracle_log_phi2(a_out[1] - a_out[0]);
        } else if (i == t) {
            b_out[i] = csa_oracle_log_phi2(a_out[t - 1] - a_out[t]);
        } else {
            const double l1 = csa_oracle_log_phi2(a_out[i - 1] - a_out[i]);
            const double l2 = csa_oracle_log_phi2(a_out[i + 1] - a_out[i]);
            const double hi = l1 > l2 ? l1 : l2, lo = l1 > l2 ? l2 : l1;
            b_out[i] = hi + log1p(exp(lo - hi));
        }
    }
    free(zero);
    free(qd);
    return 0;
}

int csa_oracle_abi_version(void) { return 1; }
