/*
 * ssm_oracle.c -- plain, slow, fp64 CPU oracle for the selective state space
 * (S6) scan and its single-step state update.
 *
 * THIS IS TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT PATH.  Only the test
 * suite, the smoke check and the CPU-baseline leg of the benchmark may load
 * it.  It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (Mamba paper, arXiv 2312.00752, as restated on the pages):
 *   - per channel (b,d) the SSM runs independently over a diagonal A
 *     ("Mamba / gitcode.csdn.net", section 2 "Structure and dimensions");
 *   - Delta = softplus(delta + delta_bias[d]) ("gitcode", section 3.2 for the
 *     softplus tau_Delta, section 3.6 for the bias; "docs.ifdog.com", section
 *     "Mamba: selective state space model", softplus(z) = log(1 + exp(z)));
 *   - Abar = exp(Delta * A) ("docs.ifdog.com", section "Discretisation", ZOH
 *     diagonal form);
 *   - Bbar * x = Delta * B * u (Euler form used by the same page's numpy
 *     selective-SSM listing); the exact ZOH form
 *     Bbar = (Delta A)^-1 (exp(Delta A) - 1) Delta B is a second mode;
 *   - h_t = Abar_t h_{t-1} + Bbar_t x_t, y_t = C_t . h_t + D x_t
 *     ("docs.ifdog.com", sections "Continuous state space model" and
 *     "Discretisation"; "gitcode", section 2, recurrent mode);
 *   - optional gate y_t *= silu(z_t) = z_t * sigmoid(z_t) ("docs.ifdog.com",
 *     section "Mamba architecture", steps 4-5);
 *   - the causal depthwise convolution (with optional SiLU) that feeds the
 *     SSM branch ("docs.ifdog.com", section "Mamba architecture", step 3a),
 *     as a separate function.
 * The hardware-aware scan of "gitcode" section 3.3.2 is an exact reordering
 * of this recurrence, so the oracle is the sequential definition itself.  A
 * second evaluation order (work-efficient tree scan of the associative
 * combine (a2*a1, a2*b1 + b2), "docs.ifdog.com", section "Hardware-aware
 * parallel scan"; Blelloch 1990) exists only so that tests can check the
 * two orders against each other.
 *
 * Complex A (the S4D-Lin initialisation A_n = -1/2 + n i, "gitcode", section
 * 3.6 "real vs complex" and "initialisation") is a separate function: the
 * state h and Abar = exp(Delta A) are complex, the Euler input term
 * Delta B u is real and enters the state as it is, and the output reads the
 * real part of the C contraction, y = Re(sum_n C h) + D u (then the gate).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - the gate multiplies the whole output C.h + D.u;
 *   - y_t uses the state after the update at step t;
 *   - the initial state is zero unless h0 is given;
 *   - softplus is exact: max(s,0) + log1p(exp(-|s|)), no linear threshold.
 *
 * Layout: every array is dense row-major.
 *   u, delta, z, y : (B, D, L)      Bm, Cm : (B, N, L)
 *   A : (D, N)    Dskip, delta_bias : (D)    h0, h_last, state : (B, D, N)
 * Nullable: z, Dskip, delta_bias, h0, h_last.
 */
#include <complex.h>
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_DISC_EULER 0
#define ORACLE_DISC_ZOH 1
#define ORACLE_ORDER_SEQUENTIAL 0
#define ORACLE_ORDER_TREE 1

/* softplus(s) = log(1 + exp(s)), written in the overflow-free form. */
static double softplus(double s) {
    return (s > 0.0 ? s : 0.0) + log1p(exp(-fabs(s)));
}

static double sigmoid(double v) { return 1.0 / (1.0 + exp(-v)); }

/* Delta for one (b,d,t): softplus(delta + bias) or, if disabled, the sum. */
static double discretisation_step(double delta, double bias, int use_softplus) {
    double s = delta + bias;
    return use_softplus ? softplus(s) : s;
}

/* Input coefficient Bbar * x for one state component. */
static double input_term(double dt, double a_cont, double b, double x, int disc) {
    if (disc == ORACLE_DISC_ZOH) {
        /* (Delta A)^-1 (exp(Delta A) - 1) Delta B = (exp(Delta A) - 1) / A * B */
        if (a_cont == 0.0) return dt * b * x;
        return expm1(dt * a_cont) / a_cont * b * x;
    }
    return dt * b * x; /* Euler: Bbar = Delta B */
}

typedef struct {
    int64_t B, D, L, N;
    const double *u, *delta, *z, *Bm, *Cm, *A, *Dskip, *delta_bias, *h0;
    int delta_softplus, disc, order;
    double *y, *h_last;
    int64_t first, last; /* channel range [first, last) over b*D + d */
    int status;
} scan_job_t;

/* Identity-padded work-efficient (Blelloch) scan over pairs (a, b), where
 * a pair stands for the affine map h -> a h + b and pairs are composed in
 * time order: combine(first, second) = (a2 a1, a2 b1 + b2).  On return
 * (ea[t], eb[t]) is the composition of pairs 0..t (inclusive prefix). */
static void tree_scan(int64_t L, const double *a, const double *b,
                      double *ea, double *eb, double *xa, double *xb, int64_t P) {
    for (int64_t i = 0; i < P; ++i) {
        xa[i] = i < L ? a[i] : 1.0;
        xb[i] = i < L ? b[i] : 0.0;
    }
    /* up-sweep: node (i + 2s - 1) := combine(left child, right child) */
    for (int64_t s = 1; s < P; s *= 2) {
        for (int64_t i = 0; i < P; i += 2 * s) {
            int64_t l = i + s - 1, r = i + 2 * s - 1;
            double na = xa[r] * xa[l];
            double nb = xa[r] * xb[l] + xb[r];
            xa[r] = na;
            xb[r] = nb;
        }
    }
    /* down-sweep with the identity at the root: exclusive prefixes */
    xa[P - 1] = 1.0;
    xb[P - 1] = 0.0;
    for (int64_t s = P / 2; s >= 1; s /= 2) {
        for (int64_t i = 0; i < P; i += 2 * s) {
            int64_t l = i + s - 1, r = i + 2 * s - 1;
            double la = xa[l], lb = xb[l];   /* total of the left subtree  */
            double pa = xa[r], pb = xb[r];   /* prefix before this subtree */
            xa[l] = pa;
            xb[l] = pb;
            xa[r] = la * pa;                 /* combine(prefix, left)      */
            xb[r] = la * pb + lb;
        }
    }
    /* inclusive prefix: combine(exclusive prefix, own pair) */
    for (int64_t t = 0; t < L; ++t) {
        ea[t] = a[t] * xa[t];
        eb[t] = a[t] * xb[t] + b[t];
    }
}

static void *scan_worker(void *arg) {
    scan_job_t *j = (scan_job_t *)arg;
    const int64_t L = j->L, N = j->N, D = j->D;
    double *h = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    double *dts = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
    double *hs = NULL, *ta = NULL, *tb = NULL, *ea = NULL, *eb = NULL, *xa = NULL, *xb = NULL;
    int64_t P = 1;
    if (j->order == ORACLE_ORDER_TREE) {
        while (P < L) P *= 2;
        hs = (double *)malloc(sizeof(double) * (size_t)(L * N + 1));
        ta = (double *)malloc(sizeof(double) * (size_t)(L + 1));
        tb = (double *)malloc(sizeof(double) * (size_t)(L + 1));
        ea = (double *)malloc(sizeof(double) * (size_t)(L + 1));
        eb = (double *)malloc(sizeof(double) * (size_t)(L + 1));
        xa = (double *)malloc(sizeof(double) * (size_t)P);
        xb = (double *)malloc(sizeof(double) * (size_t)P);
        if (!hs || !ta || !tb || !ea || !eb || !xa || !xb) { j->status = -1; goto done; }
    }
    if (!h || !dts) { j->status = -1; goto done; }

    for (int64_t c = j->first; c < j->last; ++c) {
        const int64_t b = c / D, d = c % D;
        const double *u = j->u + c * L;
        const double *dl = j->delta + c * L;
        const double *z = j->z ? j->z + c * L : NULL;
        const double *Bb = j->Bm + b * N * L;
        const double *Cb = j->Cm + b * N * L;
        const double *Ad = j->A + d * N;
        const double bias = j->delta_bias ? j->delta_bias[d] : 0.0;
        const double Dd = j->Dskip ? j->Dskip[d] : 0.0;
        double *y = j->y + c * L;

        for (int64_t t = 0; t < L; ++t)
            dts[t] = discretisation_step(dl[t], bias, j->delta_softplus);
        for (int64_t n = 0; n < N; ++n)
            h[n] = j->h0 ? j->h0[c * N + n] : 0.0;

        if (j->order == ORACLE_ORDER_SEQUENTIAL) {
            for (int64_t t = 0; t < L; ++t) {
                double acc = 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    double abar = exp(dts[t] * Ad[n]);
                    double bx = input_term(dts[t], Ad[n], Bb[n * L + t], u[t], j->disc);
                    h[n] = abar * h[n] + bx;
                    acc += Cb[n * L + t] * h[n];
                }
                y[t] = acc;
            }
        } else {
            for (int64_t n = 0; n < N; ++n) {
                for (int64_t t = 0; t < L; ++t) {
                    ta[t] = exp(dts[t] * Ad[n]);
                    tb[t] = input_term(dts[t], Ad[n], Bb[n * L + t], u[t], j->disc);
                }
                tree_scan(L, ta, tb, ea, eb, xa, xb, P);
                for (int64_t t = 0; t < L; ++t) hs[t * N + n] = ea[t] * h[n] + eb[t];
                if (L > 0) h[n] = hs[(L - 1) * N + n];
            }
            for (int64_t t = 0; t < L; ++t) {
                double acc = 0.0;
                for (int64_t n = 0; n < N; ++n) acc += Cb[n * L + t] * hs[t * N + n];
                y[t] = acc;
            }
        }
        for (int64_t t = 0; t < L; ++t) {
            double v = y[t] + Dd * u[t];
            if (z) v *= z[t] * sigmoid(z[t]);
            y[t] = v;
        }
        if (j->h_last)
            for (int64_t n = 0; n < N; ++n) j->h_last[c * N + n] = h[n];
    }
done:
    free(h); free(dts); free(hs); free(ta); free(tb); free(ea); free(eb); free(xa); free(xb);
    return NULL;
}

static int default_threads(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/* Returns the number of threads the host offers the oracle by default. */
int oracle_default_threads(void) { return default_threads(); }

/*
 * Selective scan over all channels.  Returns 0 on success, -1 on a bad
 * argument or an allocation failure.  nthreads <= 0 picks one per online
 * core; channels are split into contiguous blocks, one per thread.
 */
int oracle_selective_scan(int64_t B, int64_t D, int64_t L, int64_t N,
                          const double *u, const double *delta, const double *z,
                          const double *Bm, const double *Cm, const double *A,
                          const double *Dskip, const double *delta_bias,
                          const double *h0, int delta_softplus, int disc, int order,
                          double *y, double *h_last, int nthreads) {
    if (B < 0 || D < 0 || L < 0 || N < 0) return -1;
    if (!u || !delta || !Bm || !Cm || !A || !y) return -1;
    if (disc != ORACLE_DISC_EULER && disc != ORACLE_DISC_ZOH) return -1;
    if (order != ORACLE_ORDER_SEQUENTIAL && order != ORACLE_ORDER_TREE) return -1;
    const int64_t channels = B * D;
    if (channels == 0) return 0;
    if (nthreads <= 0) nthreads = default_threads();
    if (nthreads > channels) nthreads = (int)channels;

    scan_job_t *jobs = (scan_job_t *)calloc((size_t)nthreads, sizeof(scan_job_t));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) { free(jobs); free(tids); return -1; }
    for (int i = 0; i < nthreads; ++i) {
        scan_job_t *j = &jobs[i];
        j->B = B; j->D = D; j->L = L; j->N = N;
        j->u = u; j->delta = delta; j->z = z; j->Bm = Bm; j->Cm = Cm; j->A = A;
        j->Dskip = Dskip; j->delta_bias = delta_bias; j->h0 = h0;
        j->delta_softplus = delta_softplus; j->disc = disc; j->order = order;
        j->y = y; j->h_last = h_last;
        j->first = channels * i / nthreads;
        j->last = channels * (i + 1) / nthreads;
    }
    int rc = 0;
    if (nthreads == 1) {
        scan_worker(&jobs[0]);
    } else {
        int started = 0;
        for (int i = 0; i < nthreads; ++i) {
            if (pthread_create(&tids[i], NULL, scan_worker, &jobs[i]) != 0) break;
            ++started;
        }
        for (int i = 0; i < started; ++i) pthread_join(tids[i], NULL);
        for (int i = started; i < nthreads; ++i) scan_worker(&jobs[i]);
    }
    for (int i = 0; i < nthreads; ++i) if (jobs[i].status) rc = -1;
    free(jobs);
    free(tids);
    return rc;
}

/*
 * Selective scan with a complex diagonal A (S4D-Lin, "gitcode" section 3.6):
 * per channel the complex state runs
 *     h_t[n] = exp(Delta_t A[d,n]) h_{t-1}[n] + Delta_t B[b,n,t] u[b,d,t]
 *     y[b,d,t] = Re(sum_n C[b,n,t] h_t[n]) + Dskip[d] u[b,d,t]     (then * silu(z))
 * with A = A_re + i A_im (the real arrays of the real scan's layout, (D, N)).
 * h0 / h_last are complex (B, D, N), stored as interleaved (re, im) doubles;
 * both nullable.  Single-threaded per call block, sequential order only.
 */
int oracle_selective_scan_complex(int64_t B, int64_t D, int64_t L, int64_t N,
                                  const double *u, const double *delta, const double *z,
                                  const double *Bm, const double *Cm, const double *A_re,
                                  const double *A_im, const double *Dskip,
                                  const double *delta_bias, const double *h0,
                                  int delta_softplus, double *y, double *h_last) {
    if (B < 0 || D < 0 || L < 0 || N < 0) return -1;
    if (!u || !delta || !Bm || !Cm || !A_re || !A_im || !y) return -1;
    double complex *h = (double complex *)malloc(sizeof(double complex) * (size_t)(N > 0 ? N : 1));
    if (!h) return -1;
    for (int64_t c = 0; c < B * D; ++c) {
        const int64_t b = c / D, d = c % D;
        const double bias = delta_bias ? delta_bias[d] : 0.0;
        const double Dd = Dskip ? Dskip[d] : 0.0;
        for (int64_t n = 0; n < N; ++n)
            h[n] = h0 ? h0[2 * (c * N + n)] + I * h0[2 * (c * N + n) + 1] : 0.0;
        for (int64_t t = 0; t < L; ++t) {
            const double dt = discretisation_step(delta[c * L + t], bias, delta_softplus);
            const double ut = u[c * L + t];
            double complex acc = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                const double complex a = A_re[d * N + n] + I * A_im[d * N + n];
                const double complex abar = cexp(dt * a);
                h[n] = abar * h[n] + dt * Bm[b * N * L + n * L + t] * ut;
                acc += Cm[b * N * L + n * L + t] * h[n];
            }
            double v = creal(acc) + Dd * ut;
            if (z) v *= z[c * L + t] * sigmoid(z[c * L + t]);
            y[c * L + t] = v;
        }
        if (h_last)
            for (int64_t n = 0; n < N; ++n) {
                h_last[2 * (c * N + n)] = creal(h[n]);
                h_last[2 * (c * N + n) + 1] = cimag(h[n]);
            }
    }
    free(h);
    return 0;
}

/*
 * Mamba-2 state-space-dual (SSD) layer: the same selective recurrence with A a
 * scalar times the identity per head ("Mamba close reading", section on SSD
 * and Mamba-2: A simplified to a scalar times I, heads like multi-head
 * attention, larger states; "Mamba and state space models", section
 * "Mamba-2 and structured duality").  Heads h < H of P channels each
 * (channel d = h P + p), states n < N, per batch b and step t:
 *     Delta_t  = softplus(delta[b,h,t] + delta_bias[h])      (or the plain sum)
 *     abar_t   = exp(Delta_t a[h])                            (one scalar per head)
 *     h_t[p,n] = abar_t h_{t-1}[p,n] + Delta_t B[b,t,n] x[b,d,t]
 *     y[b,d,t] = (sum_n C[b,t,n] h_t[p,n] + Dskip[h] x[b,d,t]) * silu(z[b,d,t])
 * B and C are shared by all heads.  Layout (dense, row-major):
 *     x, z, y : (B, H*P, L)   delta : (B, H, L)   Bm, Cm : (B, L, N)
 *     a, Dskip, delta_bias : (H)   h0, h_last : (B, H, P, N)
 * Nullable: z, Dskip, delta_bias, h0, h_last.  Sequential in time, one
 * thread.  The pages' dual (masked-attention) form is a second evaluation
 * order of the same map, used by the tests as a pin.
 */
int oracle_ssd_scan(int64_t B, int64_t H, int64_t P, int64_t L, int64_t N,
                    const double *x, const double *delta, const double *z,
                    const double *Bm, const double *Cm, const double *a,
                    const double *Dskip, const double *delta_bias, const double *h0,
                    int delta_softplus, double *y, double *h_last) {
    if (B < 0 || H < 0 || P < 0 || L < 0 || N < 0) return -1;
    if (!x || !delta || !Bm || !Cm || !a || !y) return -1;
    double *h = (double *)malloc(sizeof(double) * (size_t)(P * N > 0 ? P * N : 1));
    if (!h) return -1;
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t hd = 0; hd < H; ++hd) {
            const double bias = delta_bias ? delta_bias[hd] : 0.0;
            const double Dh = Dskip ? Dskip[hd] : 0.0;
            for (int64_t i = 0; i < P * N; ++i)
                h[i] = h0 ? h0[((b * H + hd) * P) * N + i] : 0.0;
            for (int64_t t = 0; t < L; ++t) {
                const double dt = discretisation_step(delta[(b * H + hd) * L + t], bias, delta_softplus);
                const double abar = exp(dt * a[hd]);
                for (int64_t p = 0; p < P; ++p) {
                    const int64_t row = (b * H + hd) * P + p;   /* channel row of x, z, y */
                    const double xt = x[row * L + t];
                    double acc = 0.0;
                    for (int64_t n = 0; n < N; ++n) {
                        h[p * N + n] = abar * h[p * N + n] + dt * Bm[(b * L + t) * N + n] * xt;
                        acc += Cm[(b * L + t) * N + n] * h[p * N + n];
                    }
                    double v = acc + Dh * xt;
                    if (z) v *= z[row * L + t] * sigmoid(z[row * L + t]);
                    y[row * L + t] = v;
                }
            }
            if (h_last)
                for (int64_t i = 0; i < P * N; ++i) h_last[((b * H + hd) * P) * N + i] = h[i];
        }
    }
    free(h);
    return 0;
}

/*
 * One recurrent (decode) step for every channel, the loop body of the scan
 * applied once ("gitcode", section 1: constant time per step; section 2: the
 * recurrent mode used for autoregressive inference).
 *   state : (B, D, N), read and overwritten in place
 *   u, delta, z, y : (B, D)      Bm, Cm : (B, N)
 */
int oracle_state_update(int64_t B, int64_t D, int64_t N, double *state,
                        const double *u, const double *delta, const double *z,
                        const double *Bm, const double *Cm, const double *A,
                        const double *Dskip, const double *delta_bias,
                        int delta_softplus, int disc, double *y) {
    if (B < 0 || D < 0 || N < 0) return -1;
    if (!state || !u || !delta || !Bm || !Cm || !A || !y) return -1;
    if (disc != ORACLE_DISC_EULER && disc != ORACLE_DISC_ZOH) return -1;
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t d = 0; d < D; ++d) {
            const int64_t c = b * D + d;
            const double bias = delta_bias ? delta_bias[d] : 0.0;
            const double dt = discretisation_step(delta[c], bias, delta_softplus);
            double acc = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                double abar = exp(dt * A[d * N + n]);
                double bx = input_term(dt, A[d * N + n], Bm[b * N + n], u[c], disc);
                double hn = abar * state[c * N + n] + bx;
                state[c * N + n] = hn;
                acc += Cm[b * N + n] * hn;
            }
            double v = acc + (Dskip ? Dskip[d] : 0.0) * u[c];
            if (z) v *= z[c] * sigmoid(z[c]);
            y[c] = v;
        }
    }
    return 0;
}

/*
 * Causal depthwise 1-D convolution along time, optionally followed by SiLU:
 * the step in front of the selective SSM ("docs.ifdog.com", section "Mamba
 * architecture", step 3a: every channel is convolved on its own, with a
 * kernel of d_conv taps, typically 4, so that each position sees itself and
 * the d_conv - 1 positions before it; step 3b: that output enters the SSM).
 *
 *   out[b,d,t] = act(bias[d] + sum_{k=0}^{W-1} w[d,k] * x[b,d,t-(W-1)+k])
 *
 * Tap k = W-1 multiplies the current step (the order of a framework Conv1d
 * with W-1 steps of left padding, cut to the first L outputs).  Inputs before
 * t = 0 are x_hist[b,d,0..W-2] (oldest first) when given, else zero.
 * act is SiLU, v * sigmoid(v) ("docs.ifdog.com", same section, step 4), or
 * the identity.
 *   x, out : (B, D, L)   w : (D, W)   bias : (D) nullable
 *   x_hist : (B, D, W-1) nullable
 */
int oracle_causal_conv1d(int64_t B, int64_t D, int64_t L, int64_t W, const double *x,
                         const double *w, const double *bias, const double *x_hist,
                         int use_silu, double *out) {
    if (B < 0 || D < 0 || L < 0 || W < 1) return -1;
    if (B * D * L > 0 && (!x || !w || !out)) return -1;
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t d = 0; d < D; ++d) {
            const int64_t row = b * D + d;
            for (int64_t t = 0; t < L; ++t) {
                double v = bias ? bias[d] : 0.0;
                for (int64_t k = 0; k < W; ++k) {
                    const int64_t src = t - (W - 1) + k;   /* the input step tap k reads */
                    double xv;
                    if (src >= 0) xv = x[row * L + src];
                    else xv = x_hist ? x_hist[row * (W - 1) + (W - 1) + src] : 0.0;
                    v += w[d * W + k] * xv;
                }
                out[row * L + t] = use_silu ? v * sigmoid(v) : v;
            }
        }
    }
    return 0;
}

/*
 * d/dA of the exact-ZOH input coefficient g = (exp(Delta A) - 1) / A:
 *   dg/dA = (Delta e^{Delta A} A - (e^{Delta A} - 1)) / A^2 = Delta^2 psi(Delta A),
 *   psi(x) = (x e^x - (e^x - 1)) / x^2 = sum_{k>=1} k x^{k-1} / (k+1)!  (psi(0) = 1/2).
 * The closed form cancels for small |x|, so below |x| = 1e-3 the series is summed
 * (the dropped terms are below 1e-13 relative there).
 */
static double zoh_coef_dA(double dt, double a_cont) {
    const double x = dt * a_cont;
    double psi;
    if (fabs(x) < 1e-3) {
        psi = 0.5 + x / 3.0 + x * x / 8.0 + x * x * x / 30.0;
    } else {
        psi = (x * exp(x) - expm1(x)) / (x * x);
    }
    return dt * dt * psi;
}

/*
 * Reverse-mode derivative of the scan above (Euler or exact-ZOH input term), for training
 * with recomputation ("gitcode", section 3.3.2: the backward pass recomputes
 * the intermediate states instead of storing them; the oracle, being slow and
 * plain, simply keeps every state of one channel).  Given the upstream
 * gradient dy of y (and optionally dh_last of the final state) it returns the
 * gradient of every input.  Written out from the chain rule on
 *   Delta_t = softplus(s_t), s_t = delta_t + bias       dDelta/ds = sigmoid(s_t)
 *   a_t[n]  = exp(Delta_t A[n])                          da/dDelta = a A, da/dA = a Delta
 *   h_t[n]  = a_t[n] h_{t-1}[n] + g_t[n] B_t[n] u_t
 *   g = Delta (Euler: dg/dDelta = 1, dg/dA = 0) or g = (a - 1) / A (exact ZOH,
 *   "docs.ifdog.com", section "Discretisation": dg/dDelta = a, dg/dA = Delta^2 psi)
 *   p_t     = sum_n C_t[n] h_t[n] + D u_t,   y_t = p_t silu(z_t)
 *   silu'(z) = sigmoid(z) (1 + z (1 - sigmoid(z)))
 * with the adjoint lambda_t[n] = dL/dh_t[n] = (dy_t silu(z_t)) C_t[n]
 * + a_{t+1}[n] lambda_{t+1}[n], run backwards from lambda_{L-1} = dh_last
 * contributions.  dh0 = a_0 lambda_0.
 * Outputs, each overwritten (accumulated from zero over the batch and time):
 *   du, ddelta : (B, D, L)   dz : (B, D, L), only if z   dBm, dCm : (B, N, L)
 *   dA : (D, N)   dDskip : (D), only if Dskip   ddelta_bias : (D)   dh0 : (B, D, N) nullable
 */
int oracle_selective_scan_bwd(int64_t B, int64_t D, int64_t L, int64_t N,
                              const double *u, const double *delta, const double *z,
                              const double *Bm, const double *Cm, const double *A,
                              const double *Dskip, const double *delta_bias,
                              const double *h0, int delta_softplus,
                              const double *dy, const double *dh_last,
                              double *du, double *ddelta, double *dz, double *dBm, double *dCm,
                              double *dA, double *dDskip, double *ddelta_bias, double *dh0, int disc) {
    if (B < 0 || D < 0 || L < 0 || N < 0) return -1;
    if (!u || !delta || !Bm || !Cm || !A || !dy || !du || !ddelta || !dBm || !dCm || !dA || !ddelta_bias)
        return -1;
    if (disc != ORACLE_DISC_EULER && disc != ORACLE_DISC_ZOH) return -1;
    const int zoh = disc == ORACLE_DISC_ZOH;
    if (z && !dz) return -1;
    if (Dskip && !dDskip) return -1;
    memset(dBm, 0, sizeof(double) * (size_t)(B * N * L));
    memset(dCm, 0, sizeof(double) * (size_t)(B * N * L));
    memset(dA, 0, sizeof(double) * (size_t)(D * N));
    memset(ddelta_bias, 0, sizeof(double) * (size_t)D);
    if (dDskip) memset(dDskip, 0, sizeof(double) * (size_t)D);
    double *hs = (double *)malloc(sizeof(double) * (size_t)((L + 1) * N + 1));   /* h_{t-1} at row t */
    double *dts = (double *)malloc(sizeof(double) * (size_t)(L + 1));
    double *pre = (double *)malloc(sizeof(double) * (size_t)(L + 1));
    double *lam = (double *)malloc(sizeof(double) * (size_t)(N + 1));
    if (!hs || !dts || !pre || !lam) { free(hs); free(dts); free(pre); free(lam); return -1; }
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t d = 0; d < D; ++d) {
            const int64_t c = b * D + d;
            const double *uc = u + c * L, *dl = delta + c * L, *zc = z ? z + c * L : NULL;
            const double *dyc = dy + c * L;
            const double *Bb = Bm + b * N * L, *Cb = Cm + b * N * L, *Ad = A + d * N;
            const double bias = delta_bias ? delta_bias[d] : 0.0;
            const double Dd = Dskip ? Dskip[d] : 0.0;
            /* forward, keeping every state: hs[t*N + n] = h_{t-1}[n] */
            for (int64_t n = 0; n < N; ++n) hs[n] = h0 ? h0[c * N + n] : 0.0;
            for (int64_t t = 0; t < L; ++t) {
                dts[t] = discretisation_step(dl[t], bias, delta_softplus);
                double acc = 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    double hn = exp(dts[t] * Ad[n]) * hs[t * N + n] + input_term(dts[t], Ad[n], Bb[n * L + t], uc[t], disc);
                    hs[(t + 1) * N + n] = hn;
                    acc += Cb[n * L + t] * hn;
                }
                pre[t] = acc + Dd * uc[t];
            }
            /* backward */
            for (int64_t n = 0; n < N; ++n) lam[n] = dh_last ? dh_last[c * N + n] : 0.0;
            for (int64_t t = L - 1; t >= 0; --t) {
                double gate = 1.0;
                if (zc) {
                    const double sg = sigmoid(zc[t]);
                    gate = zc[t] * sg;
                    dz[c * L + t] = dyc[t] * pre[t] * sg * (1.0 + zc[t] * (1.0 - sg));
                }
                const double yt = dyc[t] * gate;   /* dL/dp_t */
                if (dDskip) dDskip[d] += yt * uc[t];
                double du_acc = yt * Dd, dDelta = 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    const double lt = lam[n] + yt * Cb[n * L + t];   /* lambda_t */
                    const double at = exp(dts[t] * Ad[n]);   /* Abar_t[n] */
                    const double hprev = hs[t * N + n];
                    const double bu = Bb[n * L + t] * uc[t];
                    /* the input coefficient g and its partial derivatives */
                    const double g = zoh ? (Ad[n] == 0.0 ? dts[t] : expm1(dts[t] * Ad[n]) / Ad[n]) : dts[t];
                    const double dg_dDelta = zoh ? at : 1.0;
                    const double dg_dA = zoh ? zoh_coef_dA(dts[t], Ad[n]) : 0.0;
                    dCm[b * N * L + n * L + t] += yt * hs[(t + 1) * N + n];
                    dA[d * N + n] += lt * (hprev * at * dts[t] + bu * dg_dA);
                    dDelta += lt * (hprev * at * Ad[n] + bu * dg_dDelta);
                    dBm[b * N * L + n * L + t] += lt * g * uc[t];
                    du_acc += lt * g * Bb[n * L + t];
                    lam[n] = lt * at;                               /* carried to step t-1 */
                }
                du[c * L + t] = du_acc;
                const double dd = delta_softplus ? dDelta * sigmoid(dl[t] + bias) : dDelta;
                ddelta[c * L + t] = dd;
                ddelta_bias[d] += dd;
            }
            if (dh0)
                for (int64_t n = 0; n < N; ++n) dh0[c * N + n] = lam[n];
        }
    }
    free(hs); free(dts); free(pre); free(lam);
    return 0;
}
