/*
 * EvoAttention oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, float64 CPU statement of the 3D attention over the pair
 * representation that MegaFold's EvoFlash-3D kernel computes (MegaFold,
 * technical summary, "Methodik" section 1 "EvoFlash-3D": online, numerically
 * stable softmax over logits that carry an additively broadcast pair-bias
 * term).  For every (b, s, h) slice and every query row j:
 *
 *   x[j,k]  = sum_d q[j,d] k[k,d] / sqrt(D) + bias[b,h,j,k] + (mask[b,s,k] ? 0 : -1e9)
 *   p[j,k]  = exp(x[j,k] - max_k x[j,:]) / sum_k exp(x[j,:] - max_k x[j,:])
 *   lse[j]  = max_k x[j,:] + log sum_k exp(x[j,:] - max_k x[j,:])
 *   O[j,d]  = sum_k p[j,k] v[k,d]
 *   out     = sigmoid(g) * O       (or O when there is no gate)
 *
 * and the analytic backward of the same expression:
 *
 *   dOa     = dout * sigmoid(g)                 dgate = dout * O * sigmoid(g) (1 - sigmoid(g))
 *   dp[j,k] = sum_d dOa[j,d] v[k,d]             delta[j] = sum_k p[j,k] dp[j,k]
 *   ds[j,k] = p[j,k] (dp[j,k] - delta[j])
 *   dq[j]   = sum_k ds[j,k] k[k] / sqrt(D)      dk[k] = sum_j ds[j,k] q[j] / sqrt(D)
 *   dv[k]   = sum_j p[j,k] dOa[j]               dbias[b,h,j,k] = sum_s ds[j,k]  (s ascending)
 *
 * The pages fix neither the formula's scale nor the mask constant; the
 * readings taken are 1/sqrt(D) and an additive -1e9 on masked keys.
 *
 * Every array is dense and row-major in the shapes named below; the oracle
 * sees no strides (callers pass explicit contiguous copies).  The logits of a
 * whole (b,s,h) slice are materialised as a plain N x N matrix -- exactly the
 * O(N^3) activation that the tiled method avoids -- because that is the
 * plainest form of the definition.
 *
 * Nothing in the product library links, includes or calls this file; only
 * the test-suite, the smoke check and the benchmark's CPU-baseline leg do.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define MASK_BIAS (-1e9)

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

typedef struct {
    int B, S, H, N, D;
    const double *q, *k, *v, *bias, *gate;
    const uint8_t *mask;
} problem;

/* offset of element [b,s,h,n,0] of a dense [B,S,H,N,D] array */
static size_t off5(const problem *P, int b, int s, int h, int n) {
    return ((((size_t)b * P->S + s) * P->H + h) * P->N + n) * (size_t)P->D;
}
/* offset of row [b,s,h,n] of a dense [B,S,H,N] array */
static size_t off4(const problem *P, int b, int s, int h, int n) {
    return (((size_t)b * P->S + s) * P->H + h) * (size_t)P->N + n;
}

/*
 * Logits, probabilities and log-sum-exp of one (b,s,h) slice.
 * x and p are N x N scratch matrices owned by the caller; lse has N entries.
 */
static void slice_probs(const problem *P, int b, int s, int h,
                        double *x, double *p, double *lse) {
    const int N = P->N, D = P->D;
    const double scale = 1.0 / sqrt((double)D);
    for (int j = 0; j < N; ++j) {
        const double *qj = P->q + off5(P, b, s, h, j);
        for (int kk = 0; kk < N; ++kk) {
            const double *kv = P->k + off5(P, b, s, h, kk);
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += qj[d] * kv[d];
            double val = dot * scale;
            val += P->bias[(((size_t)b * P->H + h) * N + j) * N + kk];
            if (P->mask && !P->mask[((size_t)b * P->S + s) * N + kk]) val += MASK_BIAS;
            x[(size_t)j * N + kk] = val;
        }
    }
    for (int j = 0; j < N; ++j) {
        const double *xj = x + (size_t)j * N;
        double m = xj[0];
        for (int kk = 1; kk < N; ++kk) if (xj[kk] > m) m = xj[kk];
        double z = 0.0;
        for (int kk = 0; kk < N; ++kk) z += exp(xj[kk] - m);
        for (int kk = 0; kk < N; ++kk) p[(size_t)j * N + kk] = exp(xj[kk] - m) / z;
        lse[j] = m + log(z);
    }
}

/* O = P V for one slice; O is N x D. */
static void slice_pv(const problem *P, int b, int s, int h, const double *p, double *O) {
    const int N = P->N, D = P->D;
    for (int j = 0; j < N; ++j)
        for (int d = 0; d < D; ++d) {
            double acc = 0.0;
            for (int kk = 0; kk < N; ++kk)
                acc += p[(size_t)j * N + kk] * P->v[off5(P, b, s, h, kk) + d];
            O[(size_t)j * D + d] = acc;
        }
}

/*
 * Forward.  q,k,v,gate,out: [B,S,H,N,D]; bias: [B,H,N,N]; mask: [B,S,N]
 * (1 = keep, may be NULL = keep all); gate may be NULL; lse: [B,S,H,N].
 * Returns 0, or -1 on bad sizes / allocation failure.
 */
int oracle_fwd(const double *q, const double *k, const double *v, const double *bias,
               const uint8_t *mask, const double *gate, double *out, double *lse,
               int B, int S, int H, int N, int D) {
    if (B < 1 || S < 1 || H < 1 || N < 1 || D < 1) return -1;
    problem P = {B, S, H, N, D, q, k, v, bias, gate, mask};
    int fail = 0;
    const long nslices = (long)B * S * H;
#pragma omp parallel
    {
        double *x = malloc(sizeof(double) * (size_t)N * N);
        double *p = malloc(sizeof(double) * (size_t)N * N);
        double *O = malloc(sizeof(double) * (size_t)N * D);
        double *l = malloc(sizeof(double) * (size_t)N);
        if (!x || !p || !O || !l) {
#pragma omp atomic write
            fail = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (long t = 0; t < nslices; ++t) {
                int h = (int)(t % H), s = (int)((t / H) % S), b = (int)(t / ((long)H * S));
                slice_probs(&P, b, s, h, x, p, l);
                slice_pv(&P, b, s, h, p, O);
                for (int j = 0; j < N; ++j) {
                    lse[off4(&P, b, s, h, j)] = l[j];
                    for (int d = 0; d < D; ++d) {
                        size_t o = off5(&P, b, s, h, j) + d;
                        double g = gate ? sigmoid(gate[o]) : 1.0;
                        out[o] = g * O[(size_t)j * D + d];
                    }
                }
            }
        }
        free(x); free(p); free(O); free(l);
    }
    return fail ? -1 : 0;
}

/*
 * Backward of one slice: fills ds (N x N) and, when the pointers are not NULL,
 * this slice's dq/dk/dv/dgate rows.  p must hold the slice's probabilities.
 */
static void slice_backward(const problem *P, int b, int s, int h, const double *p,
                           const double *dout, double *ds, double *O, double *dOa,
                           double *dq, double *dk, double *dv, double *dgate) {
    const int N = P->N, D = P->D;
    const double scale = 1.0 / sqrt((double)D);
    slice_pv(P, b, s, h, p, O);
    for (int j = 0; j < N; ++j)
        for (int d = 0; d < D; ++d) {
            size_t o = off5(P, b, s, h, j) + d;
            double g = P->gate ? sigmoid(P->gate[o]) : 1.0;
            dOa[(size_t)j * D + d] = dout[o] * g;
            if (dgate) dgate[o] = dout[o] * O[(size_t)j * D + d] * g * (1.0 - g);
        }
    for (int j = 0; j < N; ++j) {
        double delta = 0.0;
        for (int kk = 0; kk < N; ++kk) {
            double dp = 0.0;
            for (int d = 0; d < D; ++d)
                dp += dOa[(size_t)j * D + d] * P->v[off5(P, b, s, h, kk) + d];
            ds[(size_t)j * N + kk] = dp;             /* dp for now */
            delta += p[(size_t)j * N + kk] * dp;
        }
        for (int kk = 0; kk < N; ++kk) {
            size_t e = (size_t)j * N + kk;
            ds[e] = p[e] * (ds[e] - delta);
        }
    }
    if (dq)
        for (int j = 0; j < N; ++j)
            for (int d = 0; d < D; ++d) {
                double acc = 0.0;
                for (int kk = 0; kk < N; ++kk)
                    acc += ds[(size_t)j * N + kk] * P->k[off5(P, b, s, h, kk) + d];
                dq[off5(P, b, s, h, j) + d] = acc * scale;
            }
    if (dk)
        for (int kk = 0; kk < N; ++kk)
            for (int d = 0; d < D; ++d) {
                double acc = 0.0;
                for (int j = 0; j < N; ++j)
                    acc += ds[(size_t)j * N + kk] * P->q[off5(P, b, s, h, j) + d];
                dk[off5(P, b, s, h, kk) + d] = acc * scale;
            }
    if (dv)
        for (int kk = 0; kk < N; ++kk)
            for (int d = 0; d < D; ++d) {
                double acc = 0.0;
                for (int j = 0; j < N; ++j)
                    acc += p[(size_t)j * N + kk] * dOa[(size_t)j * D + d];
                dv[off5(P, b, s, h, kk) + d] = acc;
            }
}

/*
 * Backward.  Inputs as in oracle_fwd plus dout [B,S,H,N,D].  Outputs dq, dk,
 * dv, dgate: [B,S,H,N,D] (dgate ignored when gate is NULL, may be NULL);
 * dbias: [B,H,N,N], the sum over s of ds taken in ascending s.  The forward is
 * recomputed here from the inputs.  Returns 0, or -1 on failure.
 */
int oracle_bwd(const double *q, const double *k, const double *v, const double *bias,
               const uint8_t *mask, const double *gate, const double *dout,
               double *dq, double *dk, double *dv, double *dbias, double *dgate,
               int B, int S, int H, int N, int D) {
    if (B < 1 || S < 1 || H < 1 || N < 1 || D < 1) return -1;
    problem P = {B, S, H, N, D, q, k, v, bias, gate, mask};
    int fail = 0;
    const long nslices = (long)B * S * H;
    /* (1) per-slice gradients dq, dk, dv, dgate */
#pragma omp parallel
    {
        double *x = malloc(sizeof(double) * (size_t)N * N);
        double *p = malloc(sizeof(double) * (size_t)N * N);
        double *ds = malloc(sizeof(double) * (size_t)N * N);
        double *O = malloc(sizeof(double) * (size_t)N * D);
        double *dOa = malloc(sizeof(double) * (size_t)N * D);
        double *l = malloc(sizeof(double) * (size_t)N);
        if (!x || !p || !ds || !O || !dOa || !l) {
#pragma omp atomic write
            fail = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (long t = 0; t < nslices; ++t) {
                int h = (int)(t % H), s = (int)((t / H) % S), b = (int)(t / ((long)H * S));
                slice_probs(&P, b, s, h, x, p, l);
                slice_backward(&P, b, s, h, p, dout, ds, O, dOa, dq, dk, dv,
                               gate ? dgate : NULL);
            }
        }
        free(x); free(p); free(ds); free(O); free(dOa); free(l);
    }
    if (fail) return -1;
    /* (2) dbias: for each (b,h) the s-slices are visited in ascending order and
     * their ds matrices added one after another; (b,h) pairs run in parallel. */
    const long nbh = (long)B * H;
#pragma omp parallel
    {
        double *x = malloc(sizeof(double) * (size_t)N * N);
        double *p = malloc(sizeof(double) * (size_t)N * N);
        double *ds = malloc(sizeof(double) * (size_t)N * N);
        double *O = malloc(sizeof(double) * (size_t)N * D);
        double *dOa = malloc(sizeof(double) * (size_t)N * D);
        double *l = malloc(sizeof(double) * (size_t)N);
        if (!x || !p || !ds || !O || !dOa || !l) {
#pragma omp atomic write
            fail = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (long t = 0; t < nbh; ++t) {
                int h = (int)(t % H), b = (int)(t / H);
                double *db = dbias + ((size_t)b * H + h) * (size_t)N * N;
                memset(db, 0, sizeof(double) * (size_t)N * N);
                for (int s = 0; s < S; ++s) {
                    slice_probs(&P, b, s, h, x, p, l);
                    slice_backward(&P, b, s, h, p, dout, ds, O, dOa, NULL, NULL, NULL, NULL);
                    for (size_t e = 0; e < (size_t)N * N; ++e) db[e] += ds[e];
                }
            }
        }
        free(x); free(p); free(ds); free(O); free(dOa); free(l);
    }
    return fail ? -1 : 0;
}

/* Number of OpenMP threads a parallel region of the oracle uses. */
int oracle_num_threads(void) {
    int n = 1;
#pragma omp parallel
    {
#pragma omp single
        {
#ifdef _OPENMP
            extern int omp_get_num_threads(void);
            n = omp_get_num_threads();
#endif
        }
    }
    return n;
}
