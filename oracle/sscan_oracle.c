/*
 * Selective-scan oracle: plain, slow, obviously correct, double precision.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or constant with the
 * CUDA library.
 *
 * What it computes (one function per definition on the pages):
 *
 *  - oracle_sscan_fwd: the causal selective scan, stepped one timestep at a
 *    time.  "Mamba 状态空间模型：从理论到生产级推理的 CUDA 内核优化实战" page, section 2.3 (the selective_scan
 *    pseudocode: discretise, update state, contract with C, add D*x) and
 *    section 7.1 (the PyTorch reference returning (y, h)); the mamba.py
 *    listing on the "图解Blelloch并行扫描" page, section 3.2 (deltaA =
 *    exp(delta*A), deltaB*x = delta*B*x, y = h.C + D*x).  Per (b, d):
 *        h[n] = h0[b,d,n]  (0 when h0 is absent)
 *        for t:  a = exp(delta[b,d,t]*A[d,n])
 *                h[n] = a*h[n] + delta[b,d,t]*B[b,n,t]*u[b,d,t]
 *                y[b,d,t] = sum_n C[b,n,t]*h[n] + D[d]*u[b,d,t]
 *        final_state[b,d,n] = h[n] after the last step.
 *    Readings where the pages are loose: B-bar is delta*B (the simplified
 *    discretisation of section 2.3, not the zero-order-hold form of
 *    section 1.2); delta is used as given (no softplus inside); y_t uses the
 *    state after the update at t; the D skip multiplies u, not delta*u.
 *
 *  - oracle_sscan_fwd_full: the same scan with the options the pages attach
 *    to it, each off by default:
 *      delta_bias  delta <- delta + delta_bias[d] (the per-channel bias of
 *                the projection that makes delta, section 2.2; NULL = none);
 *      SOFTPLUS  then delta <- softplus(delta) inside the op (the
 *                F.softplus(delta) of the section 7.1 reference and the
 *                delta = softplus(Linear(x)) of section 2.2);
 *      ZOH       the zero-order-hold B-bar of section 1.2,
 *                (delta*A)^-1 (exp(delta*A) - 1) delta*B, which for diagonal A
 *                is expm1(delta*A[d,n]) / A[d,n] * B (delta*B when A = 0);
 *      z         an output gate, out = (y + D*u) * silu(z) with
 *                silu(z) = z / (1 + exp(-z)): the sigmoid gate activation
 *                fused into the scan kernel on the "为什么Mamba的“并行扫描”
 *                不是真并行" page, section 2, read as Mamba's SiLU gate.
 *
 *  - oracle_pscan_seq: the first-order linear recurrence h_t = a_t*h_{t-1}
 *    + b_t, one row at a time (the pscan(deltaA, BX) primitive of the
 *    mamba.py listing, "图解Blelloch并行扫描" section 3.2; with a = 1 it is
 *    the prefix sum of section 1.1).
 *
 *  - oracle_pscan_blelloch: the same recurrence by Blelloch's work-efficient
 *    up-sweep / down-sweep ("图解Blelloch并行扫描" section 2) applied to the
 *    pairs (a, b) under the associative operator
 *        (a1, b1) o (a2, b2) = (a2*a1, a2*b1 + b2)      ("first 1, then 2")
 *    of the "并行扫描与硬件感知优化 (mhpq.cn/news/1077344)" page, section 2.2, and the
 *    "Mamba 状态空间模型：从理论到生产级推理的 CUDA 内核优化实战" page,
 *    section 3.2.  Each up-sweep level is recorded so that the 8-element
 *    trace printed on the Blelloch page can be checked.
 *
 * The compile flags keep -ffp-contract=off so that x86 and Arm hosts round
 * identically.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Planted-mistake switch used only by the oracle's own pin tests, which check
 * that every plausible slip is caught by at least one pin.  0 = the oracle. */
enum {
    MUT_NONE = 0,
    MUT_DROP_D = 1,          /* forget the D*u skip term                     */
    MUT_NO_DELTA_IN_B = 2,   /* B-bar*x = B*u instead of delta*B*u           */
    MUT_Y_BEFORE_UPDATE = 3, /* contract C with the state before the update  */
    MUT_EXP_SIGN = 4,        /* a = exp(-delta*A)                            */
    MUT_IGNORE_H0 = 5,       /* start from zero even when h0 is given        */
    MUT_B_NEXT_STEP = 6,     /* read B at t+1 (index slip)                   */
    MUT_C_FROM_B = 7,        /* contract with B instead of C (operand swap)  */
    MUT_D_TIMES_DU = 8,      /* skip term D*delta*u instead of D*u           */
    MUT_BIAS_AFTER_SOFTPLUS = 9, /* softplus(delta) + bias                   */
    MUT_GATE_SIGMOID = 10,   /* out = y * sigmoid(z) instead of y * silu(z)  */
    MUT_GATE_BEFORE_D = 11,  /* gate y, then add D*u ungated                 */
    MUT_ZOH_NO_DIV = 12,     /* ZOH B-bar = expm1(delta*A) * B (1/A dropped) */
    MUT_ZOH_DELTA_TWICE = 13, /* ZOH B-bar = expm1(delta*A)/A * delta*B      */
    MUT_COUNT = 14,
    MUT_COPY = 100           /* no mistake, but through the copy that carries
                                them: it must equal the definition exactly    */
};

enum { FLAG_SOFTPLUS = 1, FLAG_ZOH = 2 };

/* log(1 + exp(x)) without overflow */
static double softplus(double x) { return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x)); }

typedef struct {
    const double *u, *delta, *A, *B, *C, *D, *h0;
    double *out, *final_state;
    int64_t batch, dim, L, N;
    int64_t first, last; /* channel range [first, last) over batch*dim */
    int mutation;
    const double *z, *delta_bias; /* [batch, dim, L] and [dim], or NULL */
    int flags;                     /* FLAG_SOFTPLUS | FLAG_ZOH           */
} sscan_job;

/* The definition, one channel at a time and one step at a time (the
 * pseudocode of section 2.3 with the options listed above). */
static void sscan_channels(const sscan_job *j)
{
    const int64_t L = j->L, N = j->N, dim = j->dim;
    double *h = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
    for (int64_t ch = j->first; ch < j->last; ++ch) {
        const int64_t b = ch / dim, d = ch % dim;
        const double *u = j->u + ch * L;      /* u[b, d, :]     */
        const double *dl = j->delta + ch * L; /* delta[b, d, :] */
        const double *Ad = j->A + d * N;      /* A[d, :]        */
        const double *Bb = j->B + b * N * L;  /* B[b, :, :]     */
        const double *Cb = j->C + b * N * L;  /* C[b, :, :]     */
        double *y = j->out + ch * L;
        for (int64_t n = 0; n < N; ++n) h[n] = j->h0 ? j->h0[ch * N + n] : 0.0;
        const double bias = j->delta_bias ? j->delta_bias[d] : 0.0;
        for (int64_t t = 0; t < L; ++t) {
            double dt = dl[t] + bias;
            if (j->flags & FLAG_SOFTPLUS) dt = softplus(dt);
            for (int64_t n = 0; n < N; ++n) {
                const double a = exp(dt * Ad[n]); /* A-bar */
                double bbar = dt;                 /* B-bar per unit B: delta (Euler) ... */
                if ((j->flags & FLAG_ZOH) && Ad[n] != 0.0) bbar = expm1(dt * Ad[n]) / Ad[n]; /* ... or ZOH */
                h[n] = a * h[n] + bbar * Bb[n * L + t] * u[t];
            }
            double acc = 0.0;
            for (int64_t n = 0; n < N; ++n) acc += Cb[n * L + t] * h[n];
            const double skip = j->D ? j->D[d] * u[t] : 0.0;
            if (j->z) {
                const double zv = j->z[ch * L + t];
                acc = (acc + skip) * (zv * (1.0 / (1.0 + exp(-zv)))); /* (y + D u) silu(z) */
            } else {
                acc += skip;
            }
            y[t] = acc;
        }
        if (j->final_state)
            for (int64_t n = 0; n < N; ++n) j->final_state[ch * N + n] = h[n];
    }
    free(h);
}

/* A copy of sscan_channels carrying the planted mistakes of the pin tests
 * (which check that every plausible slip fails at least one pin); with
 * MUT_NONE it computes exactly what sscan_channels computes. */
static void sscan_channels_mutant(const sscan_job *j)
{
    const int64_t L = j->L, N = j->N, dim = j->dim;
    double *h = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
    double *hprev = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
    for (int64_t ch = j->first; ch < j->last; ++ch) {
        const int64_t b = ch / dim, d = ch % dim;
        const double *u = j->u + ch * L;
        const double *dl = j->delta + ch * L;
        const double *Ad = j->A + d * N;
        const double *Bb = j->B + b * N * L;
        const double *Cb = j->C + b * N * L;
        double *y = j->out + ch * L;
        for (int64_t n = 0; n < N; ++n)
            h[n] = (j->h0 && j->mutation != MUT_IGNORE_H0) ? j->h0[ch * N + n] : 0.0;
        const double bias = j->delta_bias ? j->delta_bias[d] : 0.0;
        for (int64_t t = 0; t < L; ++t) {
            double dt = dl[t];
            if (j->flags & FLAG_SOFTPLUS)
                dt = (j->mutation == MUT_BIAS_AFTER_SOFTPLUS) ? softplus(dt) + bias
                                                              : softplus(dt + bias);
            else
                dt += bias;
            double acc = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                hprev[n] = h[n];
                double a = exp(dt * Ad[n]);
                if (j->mutation == MUT_EXP_SIGN) a = exp(-dt * Ad[n]);
                int64_t tb = t;
                if (j->mutation == MUT_B_NEXT_STEP && t + 1 < L) tb = t + 1;
                /* B-bar per unit B: delta (Euler) or the zero-order hold */
                double bbar = dt;
                if (j->flags & FLAG_ZOH) {
                    if (Ad[n] == 0.0)
                        bbar = dt;
                    else if (j->mutation == MUT_ZOH_NO_DIV)
                        bbar = expm1(dt * Ad[n]);
                    else if (j->mutation == MUT_ZOH_DELTA_TWICE)
                        bbar = expm1(dt * Ad[n]) / Ad[n] * dt;
                    else
                        bbar = expm1(dt * Ad[n]) / Ad[n];
                }
                double bx = bbar * Bb[n * L + tb] * u[t];
                if (j->mutation == MUT_NO_DELTA_IN_B) bx = Bb[n * L + tb] * u[t];
                h[n] = a * h[n] + bx;
            }
            for (int64_t n = 0; n < N; ++n) {
                double hv = (j->mutation == MUT_Y_BEFORE_UPDATE) ? hprev[n] : h[n];
                double cv = (j->mutation == MUT_C_FROM_B) ? Bb[n * L + t] : Cb[n * L + t];
                acc += cv * hv;
            }
            double skip = 0.0;
            if (j->D && j->mutation != MUT_DROP_D)
                skip = (j->mutation == MUT_D_TIMES_DU) ? j->D[d] * dt * u[t] : j->D[d] * u[t];
            if (j->z) {
                const double zv = j->z[ch * L + t];
                const double sig = 1.0 / (1.0 + exp(-zv));
                const double gate = (j->mutation == MUT_GATE_SIGMOID) ? sig : zv * sig;
                if (j->mutation == MUT_GATE_BEFORE_D)
                    acc = acc * gate + skip;
                else
                    acc = (acc + skip) * gate;
            } else {
                acc += skip;
            }
            y[t] = acc;
        }
        if (j->final_state)
            for (int64_t n = 0; n < N; ++n) j->final_state[ch * N + n] = h[n];
    }
    free(h);
    free(hprev);
}

static void sscan_run(const sscan_job *j)
{
    if (j->mutation == MUT_NONE)
        sscan_channels(j);
    else
        sscan_channels_mutant(j);
}

static void *sscan_thread(void *arg)
{
    sscan_run((const sscan_job *)arg);
    return NULL;
}

/* Layouts (row-major, contiguous): u, delta, out [batch, dim, L]; A [dim, N];
 * B, C [batch, N, L]; D [dim] or NULL; h0, final_state [batch, dim, N] or NULL.
 * nthreads <= 1 runs on the calling thread.  Returns 0, or -1 on bad sizes. */
int oracle_sscan_fwd_full_mutant(const double *u, const double *delta, const double *A,
                                 const double *B, const double *C, const double *D,
                                 const double *z, const double *delta_bias,
                                 const double *h0, double *out, double *final_state,
                                 int64_t batch, int64_t dim, int64_t L, int64_t N,
                                 int flags, int nthreads, int mutation)
{
    if (batch < 0 || dim < 0 || L < 0 || N < 0) return -1;
    if ((mutation < 0 || mutation >= MUT_COUNT) && mutation != MUT_COPY) return -1;
    if (flags & ~(FLAG_SOFTPLUS | FLAG_ZOH)) return -1;
    const int64_t nch = batch * dim;
    if (nch == 0) return 0;
    sscan_job base = {u, delta, A, B, C, D, h0, out, final_state,
                      batch, dim, L, N, 0, nch, mutation, z, delta_bias, flags};
    if (nthreads <= 1 || nch == 1) {
        sscan_run(&base);
        return 0;
    }
    if (nthreads > nch) nthreads = (int)nch;
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    sscan_job *jobs = (sscan_job *)malloc(sizeof(sscan_job) * (size_t)nthreads);
    int started = 0;
    for (int i = 0; i < nthreads; ++i) {
        jobs[i] = base;
        jobs[i].first = nch * i / nthreads;
        jobs[i].last = nch * (i + 1) / nthreads;
        if (pthread_create(&tid[i], NULL, sscan_thread, &jobs[i]) == 0)
            started = i + 1;
        else
            break;
    }
    /* channels of threads that failed to start run here */
    if (started < nthreads) {
        sscan_job rest = base;
        rest.first = jobs[started].first;
        sscan_run(&rest);
    }
    for (int i = 0; i < started; ++i) pthread_join(tid[i], NULL);
    free(tid);
    free(jobs);
    return 0;
}

int oracle_sscan_fwd_mutant(const double *u, const double *delta, const double *A,
                            const double *B, const double *C, const double *D,
                            const double *h0, double *out, double *final_state,
                            int64_t batch, int64_t dim, int64_t L, int64_t N,
                            int nthreads, int mutation)
{
    return oracle_sscan_fwd_full_mutant(u, delta, A, B, C, D, NULL, NULL, h0, out, final_state,
                                        batch, dim, L, N, 0, nthreads, mutation);
}

int oracle_sscan_fwd(const double *u, const double *delta, const double *A,
                     const double *B, const double *C, const double *D,
                     const double *h0, double *out, double *final_state,
                     int64_t batch, int64_t dim, int64_t L, int64_t N, int nthreads)
{
    return oracle_sscan_fwd_mutant(u, delta, A, B, C, D, h0, out, final_state,
                                   batch, dim, L, N, nthreads, MUT_NONE);
}

/* The scan with its options: z [batch, dim, L] or NULL (output gate),
 * delta_bias [dim] or NULL, flags = FLAG_SOFTPLUS (1) | FLAG_ZOH (2). */
int oracle_sscan_fwd_full(const double *u, const double *delta, const double *A,
                          const double *B, const double *C, const double *D,
                          const double *z, const double *delta_bias,
                          const double *h0, double *out, double *final_state,
                          int64_t batch, int64_t dim, int64_t L, int64_t N,
                          int flags, int nthreads)
{
    return oracle_sscan_fwd_full_mutant(u, delta, A, B, C, D, z, delta_bias, h0, out,
                                        final_state, batch, dim, L, N, flags, nthreads,
                                        MUT_NONE);
}

int oracle_mutation_count(void) { return MUT_COUNT; }

/* h[r,t] = a[r,t]*h[r,t-1] + b[r,t], h[r,-1] = h0[r] (0 when h0 is NULL).
 * a, b, h: [rows, len]; h0: [rows] or NULL. */
int oracle_pscan_seq(const double *a, const double *b, const double *h0, double *h,
                     int64_t rows, int64_t len)
{
    if (rows < 0 || len < 0) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        double s = h0 ? h0[r] : 0.0;
        for (int64_t t = 0; t < len; ++t) {
            s = a[r * len + t] * s + b[r * len + t];
            h[r * len + t] = s;
        }
    }
    return 0;
}

/* (a1,b1) o (a2,b2): apply step 1, then step 2. */
static void pair_combine(double a1, double b1, double a2, double b2,
                         double *ao, double *bo)
{
    *ao = a2 * a1;
    *bo = a2 * b1 + b2;
}

/* One row by Blelloch's scan over (a, b) pairs.  The row is padded to the next
 * power of two with identity pairs (1, 0).  trace_a / trace_b, when not NULL,
 * receive the array after each up-sweep level d = 0 .. log2(P)-1, as
 * [levels, P] row-major (P = padded length); *levels_out gets the level count.
 * The down-sweep builds exclusive prefixes; the inclusive state is the
 * exclusive prefix applied to h0, followed by the element itself.
 * Returns 0, or -1 on bad sizes / allocation failure. */
int oracle_pscan_blelloch(const double *a, const double *b, double h0, double *h,
                          int64_t len, double *trace_a, double *trace_b,
                          int64_t *levels_out)
{
    if (len < 0) return -1;
    if (len == 0) {
        if (levels_out) *levels_out = 0;
        return 0;
    }
    int64_t P = 1, levels = 0;
    while (P < len) {
        P <<= 1;
        ++levels;
    }
    double *xa = (double *)malloc((size_t)P * sizeof(double));
    double *xb = (double *)malloc((size_t)P * sizeof(double));
    if (!xa || !xb) {
        free(xa);
        free(xb);
        return -1;
    }
    for (int64_t i = 0; i < P; ++i) {
        xa[i] = i < len ? a[i] : 1.0;
        xb[i] = i < len ? b[i] : 0.0;
    }
    /* up-sweep: node at k+2^(d+1)-1 absorbs its left sibling at k+2^d-1 */
    for (int64_t d = 0; d < levels; ++d) {
        const int64_t half = (int64_t)1 << d, stride = half << 1;
        for (int64_t k = 0; k < P; k += stride) {
            const int64_t l = k + half - 1, r = k + stride - 1;
            pair_combine(xa[l], xb[l], xa[r], xb[r], &xa[r], &xb[r]);
        }
        if (trace_a && trace_b) {
            memcpy(trace_a + d * P, xa, (size_t)P * sizeof(double));
            memcpy(trace_b + d * P, xb, (size_t)P * sizeof(double));
        }
    }
    if (levels_out) *levels_out = levels;
    /* down-sweep: the root gets the identity; a right child's prefix is its
     * parent's prefix followed by the left sibling's subtree */
    double *ea = (double *)malloc((size_t)P * sizeof(double));
    double *eb = (double *)malloc((size_t)P * sizeof(double));
    if (!ea || !eb) {
        free(xa);
        free(xb);
        free(ea);
        free(eb);
        return -1;
    }
    memcpy(ea, xa, (size_t)P * sizeof(double));
    memcpy(eb, xb, (size_t)P * sizeof(double));
    ea[P - 1] = 1.0;
    eb[P - 1] = 0.0;
    for (int64_t d = levels - 1; d >= 0; --d) {
        const int64_t half = (int64_t)1 << d, stride = half << 1;
        for (int64_t k = 0; k < P; k += stride) {
            const int64_t l = k + half - 1, r = k + stride - 1;
            const double la = ea[l], lb = eb[l]; /* left subtree aggregate */
            const double pa = ea[r], pb = eb[r]; /* parent's prefix        */
            ea[l] = pa;
            eb[l] = pb;
            pair_combine(pa, pb, la, lb, &ea[r], &eb[r]);
        }
    }
    for (int64_t i = 0; i < len; ++i) {
        const double before = ea[i] * h0 + eb[i]; /* state entering step i */
        h[i] = a[i] * before + b[i];
    }
    free(xa);
    free(xb);
    free(ea);
    free(eb);
    return 0;
}

/*
 * oracle_sscan_bwd: gradients of the selective scan (the backward pass whose
 * recompute strategy "并行扫描与硬件感知优化 (mhpq.cn/news/1077344)" section
 * 3.3 describes).  Given the forward of oracle_sscan_fwd and the upstream
 * gradients dy [batch, dim, L] and dhT [batch, dim, N] (NULL = 0) of the
 * outputs y and final_state, it returns the gradients of every input, by the
 * chain rule on the forward recurrence taken in reverse time:
 *
 *   g_t[n]   = dL/dh_t[n] = C[b,n,t]*dy_t + a_{t+1}[n]*g_{t+1}[n],
 *              g_{L-1} = C*dy + dhT                      (a_t = exp(delta_t*A[d,n]))
 *   ddelta_t = sum_n g_t[n]*(h_{t-1}[n]*a_t[n]*A[d,n] + u_t*B[b,n,t])
 *   du_t     = sum_n g_t[n]*delta_t*B[b,n,t] + D[d]*dy_t
 *   dB[b,n,t] += g_t[n]*delta_t*u_t         (summed over d)
 *   dC[b,n,t] += dy_t*h_t[n]                (summed over d)
 *   dA[d,n]   += g_t[n]*h_{t-1}[n]*a_t[n]*delta_t   (summed over b, t)
 *   dD[d]     += dy_t*u_t                   (summed over b, t)
 *   dh0[n]    = a_0[n]*g_0[n]
 *
 * The forward states are kept for every step (plain and slow).  Outputs are
 * overwritten: du, ddelta [batch, dim, L]; dA [dim, N]; dB, dC [batch, N, L];
 * dD [dim] and dh0 [batch, dim, N] may be NULL.  Returns 0, or -1 on bad
 * sizes.  BWD mutations plant deliberate slips for the oracle's own pins.
 */
enum {
    BMUT_NONE = 0,
    BMUT_NO_CARRY_DECAY = 1, /* g_t = C*dy + g_{t+1} (a_{t+1} dropped)       */
    BMUT_HT_FOR_HPREV = 2,   /* use h_t instead of h_{t-1} in dL/da_t       */
    BMUT_DU_NO_D = 3,        /* forget D*dy in du                            */
    BMUT_DB_NO_U = 4,        /* dB = g*delta (u dropped)                     */
    BMUT_DH0_NO_DECAY = 5,   /* dh0 = g_0                                    */
    BMUT_COUNT = 6
};

int oracle_bwd_mutation_count(void) { return BMUT_COUNT; }

int oracle_sscan_bwd_mutant(const double *u, const double *delta, const double *A,
                            const double *B, const double *C, const double *D,
                            const double *h0, const double *dy, const double *dhT,
                            double *du, double *ddelta, double *dA, double *dB, double *dC,
                            double *dD, double *dh0, int64_t batch, int64_t dim, int64_t L,
                            int64_t N, int mutation)
{
    if (batch < 0 || dim < 0 || L < 0 || N < 0) return -1;
    if (mutation < 0 || mutation >= BMUT_COUNT) return -1;
    memset(dA, 0, sizeof(double) * (size_t)(dim * N));
    memset(dB, 0, sizeof(double) * (size_t)(batch * N * L));
    memset(dC, 0, sizeof(double) * (size_t)(batch * N * L));
    if (dD) memset(dD, 0, sizeof(double) * (size_t)dim);
    const size_t nh = (size_t)(L + 1) * (size_t)(N > 0 ? N : 1);
    double *hs = (double *)malloc(nh * sizeof(double)); /* hs[(t+1)*N + n] = h_t, hs[n] = h_{-1} */
    double *g = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t d = 0; d < dim; ++d) {
            const int64_t ch = b * dim + d;
            const double *uu = u + ch * L, *dl = delta + ch * L, *dyy = dy + ch * L;
            const double *Ad = A + d * N, *Bb = B + b * N * L, *Cb = C + b * N * L;
            for (int64_t n = 0; n < N; ++n) hs[n] = h0 ? h0[ch * N + n] : 0.0;
            for (int64_t t = 0; t < L; ++t)
                for (int64_t n = 0; n < N; ++n)
                    hs[(t + 1) * N + n] = exp(dl[t] * Ad[n]) * hs[t * N + n] + dl[t] * Bb[n * L + t] * uu[t];
            for (int64_t n = 0; n < N; ++n) g[n] = dhT ? dhT[ch * N + n] : 0.0; /* G_{L-1} */
            for (int64_t t = L - 1; t >= 0; --t) {
                double sdu = 0.0, sdd = 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    const double a = exp(dl[t] * Ad[n]);
                    const double gt = Cb[n * L + t] * dyy[t] + g[n];
                    const double hprev = (mutation == BMUT_HT_FOR_HPREV) ? hs[(t + 1) * N + n] : hs[t * N + n];
                    sdd += gt * (hprev * a * Ad[n] + uu[t] * Bb[n * L + t]);
                    sdu += gt * dl[t] * Bb[n * L + t];
                    dB[b * N * L + n * L + t] += gt * dl[t] * ((mutation == BMUT_DB_NO_U) ? 1.0 : uu[t]);
                    dC[b * N * L + n * L + t] += dyy[t] * hs[(t + 1) * N + n];
                    dA[d * N + n] += gt * hprev * a * dl[t];
                    g[n] = (mutation == BMUT_NO_CARRY_DECAY) ? gt : a * gt; /* G_{t-1} */
                    if (t == 0 && dh0) dh0[ch * N + n] = (mutation == BMUT_DH0_NO_DECAY) ? gt : a * gt;
                }
                if (D && mutation != BMUT_DU_NO_D) sdu += D[d] * dyy[t];
                du[ch * L + t] = sdu;
                ddelta[ch * L + t] = sdd;
                if (dD && D) dD[d] += dyy[t] * uu[t];
            }
            if (L == 0 && dh0)
                for (int64_t n = 0; n < N; ++n) dh0[ch * N + n] = dhT ? dhT[ch * N + n] : 0.0;
        }
    }
    free(hs);
    free(g);
    return 0;
}

int oracle_sscan_bwd(const double *u, const double *delta, const double *A, const double *B,
                     const double *C, const double *D, const double *h0, const double *dy,
                     const double *dhT, double *du, double *ddelta, double *dA, double *dB,
                     double *dC, double *dD, double *dh0, int64_t batch, int64_t dim, int64_t L,
                     int64_t N)
{
    return oracle_sscan_bwd_mutant(u, delta, A, B, C, D, h0, dy, dhT, du, ddelta, dA, dB, dC,
                                   dD, dh0, batch, dim, L, N, BMUT_NONE);
}
