/*
 * Continuous Softmax Attention: gradients of the forward pass, CPU oracle,
 * double precision.
 *
 * TEST INFRASTRUCTURE ONLY (same rules as csa_oracle.c: only the tests, the
 * smoke check and the benchmark's CPU legs load this library; the CUDA
 * library shares no code with it).
 *
 * The pages do not write the backward pass out; they train models with the
 * method (Jianlin Su, "Continuous Softmax Attention", section "Simple
 * Experiments"), which needs it.  This file is the plain chain rule through
 * the forward pass as the page states it in eq. (10)/(11) ("Assembly and
 * Simplification"):
 *
 *   a_i = scale q . k_i (i = 0..t, k_0 the sink),
 *   E_i = [i >= 1] phi2(a_{i-1} - a_i) + [i <= t-1] phi2(a_{i+1} - a_i),
 *   z_i = a_i + log E_i,  P_i = e^{z_i} / sum_j e^{z_j},  o = sum_i P_i v_i.
 *
 * For a loss L with dL/do = dO (one row):
 *   dL/dv_i = P_i dO;
 *   dL/dz_i = P_i (dP_i - D),  dP_i = dO . v_i,  D = dO . o   (softmax);
 *   dL/da_j = dL/dz_j + sum_i dL/dz_i * d(log E_i)/da_j, where log E_i
 *   depends on a_{i-1}, a_i, a_{i+1} through phi2, so that (with
 *   phi2'(x) = d phi2 / dx and u_i = (dL/dz_i) / E_i):
 *     d(log E_i)/da_i     = -(phi2'(a_{i-1}-a_i) + phi2'(a_{i+1}-a_i)) / E_i,
 *     d(log E_i)/da_{i-1} =   phi2'(a_{i-1}-a_i) / E_i,
 *     d(log E_i)/da_{i+1} =   phi2'(a_{i+1}-a_i) / E_i;
 *   dL/dq = scale sum_i (dL/da_i) k_i,  dL/dk_i = scale (dL/da_i) q.
 * u_i phi2'(x) is formed as (dP_i - D) exp(a_i - lse + log phi2'(x)), since
 * P_i / E_i = e^{a_i - lse}; nothing overflows.
 *
 * phi2'(x) = int_0^1 s (1 - s) e^{sx} ds > 0 (differentiating eq. (6) under
 * the integral), = ((x - 2) e^x + x + 2) / x^3, with the power series
 * sum_m (m + 1) x^m / (m + 3)! near 0.
 *
 * Sink gradients: k_0, v_0 are trainable in mode 2 (the last paragraph of
 * "Analysis of the Result"): dk0, dv0 [H, d] sum over the batch and the
 * rows.  In mode 1 (k_0 = k_1, v_0 = v_1) the sink's gradient flows into
 * array key 0; in mode 0 the sink is a constant.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

double csa_oracle_log_phi2(double x); /* csa_oracle.c */

/* log phi2'(x), finite for every real x. */
double csa_oracle_log_dphi2(double x)
{
    if (fabs(x) < 0.5) {
        /* sum_{m=0}^{23} (m+1) x^m / (m+3)!; the first omitted term is below
         * 1e-30 at |x| = 0.5 */
        double c[24];
        double f = 6.0; /* 3! */
        for (int m = 0; m < 24; ++m) {
            if (m > 0) f *= (double)(m + 3);
            c[m] = (double)(m + 1) / f;
        }
        double acc = c[23];
        for (int m = 22; m >= 0; --m) acc = acc * x + c[m];
        return log(acc);
    }
    if (x > 0.0) /* e^x ((x - 2) + (x + 2) e^{-x}) / x^3 */
        return x + log((x - 2.0) + (x + 2.0) * exp(-x)) - 3.0 * log(x);
    /* x <= -0.5: numerator and x^3 are both negative */
    return log(((x - 2.0) * exp(x) + x + 2.0) / (x * x * x));
}

typedef struct {
    const float *q, *k, *v, *k0, *v0, *dout;
    double *dq, *dk, *dv, *dk0_part, *dv0_part; /* parts: [B*H, d] */
    int B, H, T, d, mode;
    double scale;
} bjob_t;

typedef struct {
    const bjob_t *job;
    int index, count, status;
} bslice_t;

static const float *sink_key(const bjob_t *jb, long long bh, int h, const float *zero)
{
    if (jb->mode == 1) return jb->k + (size_t)bh * jb->T * jb->d;
    if (jb->mode == 2) return jb->k0 + (size_t)h * jb->d;
    return zero;
}

static const float *sink_val(const bjob_t *jb, long long bh, int h, const float *zero)
{
    if (jb->mode == 1) return jb->v + (size_t)bh * jb->T * jb->d;
    if (jb->mode == 2) return jb->v0 + (size_t)h * jb->d;
    return zero;
}

/* All rows of one (b, h).  Work arrays: a, z, P, dP, da of T+1 doubles,
 * o and dsink_k / dsink_v of d doubles. */
static void one_head(const bjob_t *jb, long long bh, double *work, const float *zero)
{
    const int T = jb->T, d = jb->d, h = (int)(bh % jb->H);
    double *a = work, *z = a + (T + 1), *P = z + (T + 1), *dP = P + (T + 1), *da = dP + (T + 1);
    double *o = da + (T + 1), *gk0 = o + d, *gv0 = gk0 + d;
    const size_t base = (size_t)bh * T * d;
    for (int c = 0; c < d; ++c) gk0[c] = gv0[c] = 0.0;
    for (int r = 0; r < T; ++r) {
        const int t = r + 1;
        const float *qr = jb->q + base + (size_t)r * d;
        const float *gr = jb->dout + base + (size_t)r * d;
#define KEY(i) ((i) == 0 ? sink_key(jb, bh, h, zero) : jb->k + base + (size_t)((i) - 1) * d)
#define VAL(i) ((i) == 0 ? sink_val(jb, bh, h, zero) : jb->v + base + (size_t)((i) - 1) * d)
        for (int i = 0; i <= t; ++i) {
            const float *ki = KEY(i);
            double s = 0.0;
            for (int c = 0; c < d; ++c) s += (double)qr[c] * (double)ki[c];
            a[i] = jb->scale * s;
        }
        /* eq. (10): z_i = a_i + log E_i (the sum of two phi2 by logaddexp) */
        double zmax = -INFINITY;
        for (int i = 0; i <= t; ++i) {
            double lb;
            if (i == 0) {
                lb = csa_oracle_log_phi2(a[1] - a[0]);
            } else if (i == t) {
                lb = csa_oracle_log_phi2(a[t - 1] - a[t]);
            } else {
                const double l1 = csa_oracle_log_phi2(a[i - 1] - a[i]);
                const double l2 = csa_oracle_log_phi2(a[i + 1] - a[i]);
                const double hi = l1 > l2 ? l1 : l2, lo = l1 > l2 ? l2 : l1;
                lb = hi + log1p(exp(lo - hi));
            }
            z[i] = a[i] + lb;
            if (z[i] > zmax) zmax = z[i];
        }
        double den = 0.0;
        for (int i = 0; i <= t; ++i) den += exp(z[i] - zmax);
        const double lse = zmax + log(den);
        /* eq. (11) */
        for (int c = 0; c < d; ++c) o[c] = 0.0;
        for (int i = 0; i <= t; ++i) {
            P[i] = exp(z[i] - lse);
            const float *vi = VAL(i);
            for (int c = 0; c < d; ++c) o[c] += P[i] * (double)vi[c];
        }
        double D = 0.0;
        for (int c = 0; c < d; ++c) D += (double)gr[c] * o[c];
        for (int i = 0; i <= t; ++i) {
            const float *vi = VAL(i);
            double s = 0.0;
            for (int c = 0; c < d; ++c) s += (double)gr[c] * (double)vi[c];
            dP[i] = s;
        }
        /* dL/da_j: the softmax term plus the three logs E_{j-1}, E_j, E_{j+1}
         * that depend on a_j */
        for (int j = 0; j <= t; ++j) {
            double g = P[j] * (dP[j] - D);
            const double uj = dP[j] - D; /* times e^{a_j - lse} inside each term */
            if (j >= 1) {
                g -= uj * exp(a[j] - lse + csa_oracle_log_dphi2(a[j - 1] - a[j]));
                g += (dP[j - 1] - D) * exp(a[j - 1] - lse + csa_oracle_log_dphi2(a[j] - a[j - 1]));
            }
            if (j <= t - 1) {
                g -= uj * exp(a[j] - lse + csa_oracle_log_dphi2(a[j + 1] - a[j]));
                g += (dP[j + 1] - D) * exp(a[j + 1] - lse + csa_oracle_log_dphi2(a[j] - a[j + 1]));
            }
            da[j] = g;
        }
        /* dq_t, dk_i, dv_i */
        double *dqr = jb->dq + base + (size_t)r * d;
        for (int c = 0; c < d; ++c) dqr[c] = 0.0;
        for (int i = 0; i <= t; ++i) {
            const float *ki = KEY(i);
            const double ds = jb->scale * da[i];
            for (int c = 0; c < d; ++c) dqr[c] += ds * (double)ki[c];
            if (i >= 1) {
                double *dki = jb->dk + base + (size_t)(i - 1) * d;
                double *dvi = jb->dv + base + (size_t)(i - 1) * d;
                for (int c = 0; c < d; ++c) {
                    dki[c] += ds * (double)qr[c];
                    dvi[c] += P[i] * (double)gr[c];
                }
            } else {
                for (int c = 0; c < d; ++c) {
                    gk0[c] += ds * (double)qr[c];
                    gv0[c] += P[0] * (double)gr[c];
                }
            }
        }
#undef KEY
#undef VAL
    }
    if (jb->mode == 1) { /* the sink is array key 0 */
        for (int c = 0; c < d; ++c) {
            jb->dk[base + c] += gk0[c];
            jb->dv[base + c] += gv0[c];
        }
    } else if (jb->mode == 2) {
        for (int c = 0; c < d; ++c) {
            jb->dk0_part[(size_t)bh * d + c] = gk0[c];
            jb->dv0_part[(size_t)bh * d + c] = gv0[c];
        }
    }
}

static void *run_heads(void *arg)
{
    bslice_t *s = (bslice_t *)arg;
    const bjob_t *jb = s->job;
    const size_t n = 5 * ((size_t)jb->T + 1) + 3 * (size_t)jb->d;
    double *work = (double *)malloc(sizeof(double) * n);
    float *zero = (float *)calloc((size_t)jb->d, sizeof(float));
    if (!work || !zero) {
        free(work);
        free(zero);
        s->status = -2;
        return NULL;
    }
    const long long BH = (long long)jb->B * jb->H;
    for (long long bh = s->index; bh < BH; bh += s->count) one_head(jb, bh, work, zero);
    free(work);
    free(zero);
    s->status = 0;
    return NULL;
}

/* Gradients of L = sum dout . o for the forward pass of csa_oracle_forward.
 * q, k, v, dout: float32 [B, H, T, d]; k0, v0: float32 [H, d] (mode 2).
 * dq, dk, dv: double [B, H, T, d] (overwritten); dk0, dv0: double [H, d]
 * (mode 2 only; may be NULL otherwise).  Heads run in parallel on nthreads
 * threads.  Returns 0, or -1 on a bad argument, -2 when memory runs out. */
int csa_oracle_backward(const float *q, const float *k, const float *v, const float *k0,
                        const float *v0, const float *dout, double *dq, double *dk, double *dv,
                        double *dk0, double *dv0, int B, int H, int T, int d, double scale,
                        int k0_mode, int nthreads)
{
    if (B < 0 || H < 0 || T < 0 || d < 1 || k0_mode < 0 || k0_mode > 2) return -1;
    const long long BH = (long long)B * H;
    if (k0_mode == 2 && (!k0 || !v0 || !dk0 || !dv0)) return -1;
    if (k0_mode == 2) {
        memset(dk0, 0, sizeof(double) * (size_t)H * d);
        memset(dv0, 0, sizeof(double) * (size_t)H * d);
    }
    if (BH * T == 0) return 0;
    if (!q || !k || !v || !dout || !dq || !dk || !dv) return -1;
    const size_t n = (size_t)BH * T * d;
    memset(dq, 0, sizeof(double) * n);
    memset(dk, 0, sizeof(double) * n);
    memset(dv, 0, sizeof(double) * n);
    bjob_t jb;
    memset(&jb, 0, sizeof(jb));
    jb.q = q; jb.k = k; jb.v = v; jb.k0 = k0; jb.v0 = v0; jb.dout = dout;
    jb.dq = dq; jb.dk = dk; jb.dv = dv;
    jb.B = B; jb.H = H; jb.T = T; jb.d = d; jb.mode = k0_mode; jb.scale = scale;
    if (k0_mode == 2) {
        jb.dk0_part = (double *)calloc((size_t)BH * d, sizeof(double));
        jb.dv0_part = (double *)calloc((size_t)BH * d, sizeof(double));
        if (!jb.dk0_part || !jb.dv0_part) {
            free(jb.dk0_part);
            free(jb.dv0_part);
            return -2;
        }
    }
    if (nthreads < 1) nthreads = 1;
    if (nthreads > BH) nthreads = (int)BH;
    if (nthreads > 1024) nthreads = 1024;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    bslice_t *sl = (bslice_t *)malloc(sizeof(bslice_t) * (size_t)nthreads);
    unsigned char *joined = (unsigned char *)calloc((size_t)nthreads, 1);
    int rc = 0;
    if (!th || !sl || !joined) {
        rc = -2;
    } else {
        for (int i = 0; i < nthreads; ++i) {
            sl[i].job = &jb;
            sl[i].index = i;
            sl[i].count = nthreads;
            sl[i].status = 0;
        }
        for (int i = 0; i < nthreads; ++i) {
            if (pthread_create(&th[i], NULL, run_heads, &sl[i]) == 0)
                joined[i] = 1;
            else
                run_heads(&sl[i]);
        }
        for (int i = 0; i < nthreads; ++i)
            if (joined[i]) pthread_join(th[i], NULL);
        for (int i = 0; i < nthreads; ++i)
            if (sl[i].status != 0) rc = sl[i].status;
    }
    if (rc == 0 && k0_mode == 2) { /* the sink pair is shared across the batch */
        for (long long bh = 0; bh < BH; ++bh) {
            const int h = (int)(bh % H);
            for (int c = 0; c < d; ++c) {
                dk0[(size_t)h * d + c] += jb.dk0_part[(size_t)bh * d + c];
                dv0[(size_t)h * d + c] += jb.dv0_part[(size_t)bh * d + c];
            }
        }
    }
    free(th);
    free(sl);
    free(joined);
    free(jb.dk0_part);
    free(jb.dv0_part);
    return rc;
}
