/*
 * Plain fp64 CPU oracle of the selective scan (S6) forward pass and of the
 * single-token decode state update.
 *
 * TEST INFRASTRUCTURE ONLY. It exists to check the CUDA library; only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg may load it. It
 * shares no code, header or table with the CUDA path.
 *
 * What it computes, per row (b, d) of the (batch, dim) grid, sequentially in l:
 *
 *   x      = delta[b,d,l] + bias[d]
 *   dt     = softplus(x)                    (or x itself when softplus is off)
 *   for n:  h[n] = exp(dt * A[d,n]) * h[n] + dt * B[b,n,l] * u[b,d,l]
 *   y      = sum_n C[b,n,l] * h[n] + D[d] * u[b,d,l]
 *   y     *= z * sigmoid(z)                 (when z is given)
 *   h_last[b,d,:] = h after the last step
 *
 * Sources, by page title and section:
 *  - "Mamba: Linear-Time Sequence Modeling with Selective State Spaces",
 *    section "Method": zero-order-hold discretisation, A_bar = exp(Delta A),
 *    and the recurrence h_t = A_bar h_{t-1} + B_bar x_t, y_t = C h_t.
 *  - same page, section "The Selection Mechanism (S6)": B_t and C_t are
 *    per-token projections of width N (shared by every channel d) and
 *    Delta_t = softplus(parameter + projection).
 *  - soft186.com, "Mamba选择性状态空间机制", section "动态参数化的状态空间": the
 *    step is dt = softplus(projection + delta_bias), dA = exp(dt * A), and the
 *    state update multiplies the state by dA and adds the input times dt*B
 *    (the simplified input matrix dt*B is used instead of the exact ZOH B_bar).
 *  - same Mamba page, section "Key terms" (Mamba block): a multiplicative
 *    gate follows the SSM; it is silu(z) here and multiplies C.h + D*u.
 *  - same Mamba page, section "Questions": decoding keeps only the fixed-size
 *    D x N state per layer and advances it by one step per token.
 *
 * Inputs are read exactly (fp32 as is, bf16 bit patterns widened exactly) and
 * all arithmetic is fp64 with the C library's exp and log1p.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_BF16 = 1 };

static double rd(const void *p, long long i, int dtype) {
    if (dtype == ORC_BF16) {
        uint32_t bits = ((uint32_t)((const uint16_t *)p)[i]) << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return (double)((const float *)p)[i];
}

/* softplus(x) = log(1 + e^x), evaluated without overflow or cancellation. */
double ss_oracle_softplus(double x) {
    return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x));
}

/* silu(z) = z * sigmoid(z) = z / (1 + e^-z). */
double ss_oracle_silu(double z) { return z / (1.0 + exp(-z)); }

typedef struct {
    /* geometry */
    long long nrows, seqlen;
    int dim, dstate, dtype;
    const int *row_b, *row_d;          /* (nrows): batch and channel of each row */
    /* inputs */
    const void *u, *delta, *z;         /* (nrows, seqlen); z may be NULL */
    const float *A;                    /* (dim, dstate) */
    const void *B, *C;                 /* (batch, dstate, seqlen) */
    const float *D, *bias;             /* (dim); may be NULL */
    int softplus;
    int zoh;                           /* 1: exact zero-order-hold input matrix */
    const double *h0;                  /* (nrows, dstate) or NULL */
    /* outputs */
    double *y;                         /* (nrows, seqlen) or NULL */
    double *h_last;                    /* (nrows, dstate) or NULL */
    /* work split */
    long long lo, hi;
} scan_job;

/*
 * The factor that turns B into the discrete input matrix, per state:
 *  - simplified (soft186.com article, "动态参数化的状态空间"): dt;
 *  - exact zero-order hold ("Mamba: Linear-Time Sequence Modeling with
 *    Selective State Spaces", section "Method": B_bar = (dt A)^-1 (exp(dt A) - I) dt B,
 *    diagonal A): (exp(dt a) - 1) / a, whose limit at a = 0 is dt.
 */
static double input_factor(double dt, double a, int zoh) {
    if (!zoh || a == 0.0) return dt;
    return expm1(dt * a) / a;
}

static void scan_rows(const scan_job *j) {
    const long long L = j->seqlen;
    const int N = j->dstate;
    double *h = (double *)malloc(sizeof(double) * (size_t)N);
    for (long long r = j->lo; r < j->hi; ++r) {
        const int b = j->row_b[r], d = j->row_d[r];
        const long long urow = r * L;
        const long long bcrow = (long long)b * N * L;
        for (int n = 0; n < N; ++n) h[n] = j->h0 ? j->h0[r * N + n] : 0.0;
        const double bias = j->bias ? (double)j->bias[d] : 0.0;
        const double Dd = j->D ? (double)j->D[d] : 0.0;
        for (long long l = 0; l < L; ++l) {
            const double uv = rd(j->u, urow + l, j->dtype);
            const double x = rd(j->delta, urow + l, j->dtype) + bias;
            const double dt = j->softplus ? ss_oracle_softplus(x) : x;
            double yv = 0.0;
            for (int n = 0; n < N; ++n) {
                const double a = (double)j->A[(long long)d * N + n];
                const double Bv = rd(j->B, bcrow + (long long)n * L + l, j->dtype);
                const double Cv = rd(j->C, bcrow + (long long)n * L + l, j->dtype);
                const double bbar = input_factor(dt, a, j->zoh);
                h[n] = exp(dt * a) * h[n] + bbar * Bv * uv;
                yv += Cv * h[n];
            }
            yv += Dd * uv;
            if (j->z) yv *= ss_oracle_silu(rd(j->z, urow + l, j->dtype));
            if (j->y) j->y[urow + l] = yv;
        }
        if (j->h_last)
            for (int n = 0; n < N; ++n) j->h_last[r * N + n] = h[n];
    }
    free(h);
}

static void *scan_thread(void *arg) {
    scan_rows((const scan_job *)arg);
    return NULL;
}

/*
 * Selective scan forward over an explicit list of rows.
 *
 * row_b/row_d give the (batch, channel) of each of the nrows rows; u, delta
 * and z hold those rows only, row-major (nrows, seqlen). B and C hold every
 * batch, (batch, dstate, seqlen). dtype: 0 = fp32, 1 = bf16 bit patterns.
 * h0 (nrows, dstate) or NULL for a zero initial state. y (nrows, seqlen) and
 * h_last (nrows, dstate) are written in fp64; either may be NULL.
 * nthreads <= 0 uses one thread. Returns 0, or -1 on a bad argument.
 */
int ss_oracle_scan(long long nrows, const int *row_b, const int *row_d, int dim,
                   int dstate, long long seqlen, int dtype, const void *u,
                   const void *delta, const void *z, const float *A, const void *B,
                   const void *C, const float *D, const float *delta_bias,
                   int delta_softplus, const double *h0, double *y, double *h_last,
                   int zoh, int nthreads) {
    if (nrows < 0 || dim <= 0 || dstate <= 0 || seqlen < 0) return -1;
    if (!row_b || !row_d || !u || !delta || !A || !B || !C) return -1;
    if (dtype != ORC_F32 && dtype != ORC_BF16) return -1;
    for (long long r = 0; r < nrows; ++r)
        if (row_d[r] < 0 || row_d[r] >= dim || row_b[r] < 0) return -1;
    scan_job base = {nrows, seqlen, dim, dstate, dtype, row_b, row_d, u, delta, z,
                     A, B, C, D, delta_bias, delta_softplus, zoh, h0, y, h_last, 0, nrows};
    if (nthreads <= 1 || nrows < 2) {
        scan_rows(&base);
        return 0;
    }
    if (nthreads > nrows) nthreads = (int)nrows;
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    scan_job *jobs = (scan_job *)malloc(sizeof(scan_job) * (size_t)nthreads);
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = base;
        jobs[t].lo = nrows * t / nthreads;
        jobs[t].hi = nrows * (t + 1) / nthreads;
        pthread_create(&tid[t], NULL, scan_thread, &jobs[t]);
    }
    for (int t = 0; t < nthreads; ++t) pthread_join(tid[t], NULL);
    free(jobs);
    free(tid);
    return 0;
}

/*
 * Decode: one token per row. The state (nrows, dstate) is read and replaced
 * by the state after the step; y (nrows) receives the gated output. x, dt, z
 * are (nrows); B, C are (batch, dstate). This is the scan above with one
 * time step and h0 = state.
 */
int ss_oracle_state_update(long long nrows, const int *row_b, const int *row_d,
                           int dim, int dstate, int dtype, double *state,
                           const void *x, const void *dt, const void *z,
                           const float *A, const void *B, const void *C,
                           const float *D, const float *dt_bias, int dt_softplus,
                           double *y, int zoh, int nthreads) {
    if (!state) return -1;
    double *h_new = (double *)malloc(sizeof(double) * (size_t)(nrows * dstate + 1));
    int rc = ss_oracle_scan(nrows, row_b, row_d, dim, dstate, 1, dtype, x, dt, z, A,
                            B, C, D, dt_bias, dt_softplus, state, y, h_new, zoh, nthreads);
    if (rc == 0) memcpy(state, h_new, sizeof(double) * (size_t)(nrows * dstate));
    free(h_new);
    return rc;
}

/*
 * Causal depthwise 1D convolution of the Mamba block, and its decode step.
 *
 * Sources, by page title and section:
 *  - "Mamba: Linear-Time Sequence Modeling with Selective State Spaces",
 *    section "Key terms" (Mamba block): the block combines the input
 *    projection, a 1D convolution, the selective SSM and a multiplicative
 *    gate.
 *  - soft186.com, "Mamba选择性状态空间机制", section "基础模型构建": the
 *    convolution width d_conv = 4, and the install line names the
 *    causal-conv1d package (the convolution looks only backwards in time).
 *
 * Per row (b, d), width W, weights w[d][0..W-1], inputs x[0..L-1]:
 *   out[l] = bias[d] + sum_{k=0}^{W-1} w[d][k] * xin(l - (W-1) + k)
 *   xin(j) = x[j] for j >= 0, and the given initial state s[(W-1) + j] for
 *            -(W-1) <= j < 0 (zero without a state)
 *   out[l] = silu(out[l]) when asked
 * The state after the row is its last W-1 inputs, xin(L-(W-1)) .. xin(L-1).
 */
static double conv_in(const void *x, long long row_off, long long j, int dtype,
                      const double *s, int W) {
    if (j >= 0) return rd(x, row_off + j, dtype);
    return s ? s[(W - 1) + j] : 0.0;
}

int ss_oracle_conv1d(long long nrows, const int *row_d, int width, long long seqlen, int dtype,
                     const void *x, const float *w, const float *bias,
                     const double *init_state, int silu, double *out, double *final_state) {
    if (nrows < 0 || width < 1 || seqlen < 0 || !row_d || (seqlen > 0 && (!x || !out)) || !w)
        return -1;
    for (long long r = 0; r < nrows; ++r) {
        const int d = row_d[r];
        const double *s = init_state ? init_state + r * (width - 1) : NULL;
        const float *wd = w + (long long)d * width;
        const long long off = r * seqlen;
        for (long long l = 0; l < seqlen; ++l) {
            double acc = bias ? (double)bias[d] : 0.0;
            for (int k = 0; k < width; ++k)
                acc += (double)wd[k] * conv_in(x, off, l - (width - 1) + k, dtype, s, width);
            out[off + l] = silu ? ss_oracle_silu(acc) : acc;
        }
        if (final_state) {
            double *fs = final_state + r * (width - 1);
            double tmp[64];
            if (width - 1 > 64) return -1;
            for (int j = 0; j < width - 1; ++j)
                tmp[j] = conv_in(x, off, seqlen - (width - 1) + j, dtype, s, width);
            for (int j = 0; j < width - 1; ++j) fs[j] = tmp[j];
        }
    }
    return 0;
}

/*
 * Decode step of the convolution: for each row, out = bias + w[W-1] * x
 * + sum_{k<W-1} w[k] * state[k] (then silu when asked), and the state drops
 * its oldest input and appends x. state is (nrows, W-1), oldest first.
 */
int ss_oracle_conv1d_update(long long nrows, const int *row_d, int width, int dtype,
                            const void *x, const float *w, const float *bias, int silu,
                            double *state, double *out) {
    if (nrows < 0 || width < 1 || !row_d || !x || !w || !out || (width > 1 && !state)) return -1;
    for (long long r = 0; r < nrows; ++r) {
        const int d = row_d[r];
        const float *wd = w + (long long)d * width;
        double *s = state + r * (width - 1);
        const double xv = rd(x, r, dtype);
        double acc = bias ? (double)bias[d] : 0.0;
        for (int k = 0; k < width - 1; ++k) acc += (double)wd[k] * s[k];
        acc += (double)wd[width - 1] * xv;
        out[r] = silu ? ss_oracle_silu(acc) : acc;
        for (int k = 0; k + 1 < width - 1; ++k) s[k] = s[k + 1];
        if (width > 1) s[width - 2] = xv;
    }
    return 0;
}

/*
 * Backward pass of the selective scan: the gradients of a scalar loss with
 * respect to every input, given dy = dL/dy and optionally dh_last = dL/dh_L.
 * This is reverse-mode differentiation of the forward recurrence above, row
 * by row, in fp64; the forward states of a row are recomputed and kept in full
 * (this oracle has no memory limit). With x = delta + bias, dt = softplus(x),
 * e_n = exp(dt a_n), s = sum_n C_n h_n + D u, y = s silu(z):
 *   gs   = dy silu(z)                     gz = dy s silu'(z)
 *   g_n  = dL/dh_n(t) = gs C_n + e_n(t+1) g_n(t+1)   (+ dh_last at t = L-1)
 *   dC_n += gs h_n(t)          dB_n += g_n f_n u      (f_n: dt, or the ZOH factor)
 *   du   += gs D + sum_n g_n f_n B_n                  dD += gs u
 *   ddt   = sum_n g_n (a_n e_n h_n(t-1) + df_n/ddt B_n u)
 *   dA_n += g_n (dt e_n h_n(t-1) + df_n/da_n B_n u)
 *   ddelta = ddt sigmoid(x) (softplus) or ddt;  dbias += ddelta
 *   dh0_n = e_n(0) g_n(0)
 * dA, dB, dC, dD and dbias are sums over rows and must be zeroed by the
 * caller; the per-row outputs are overwritten.
 */
int ss_oracle_scan_bwd(long long nrows, const int *row_b, const int *row_d, int dim,
                       int dstate, long long seqlen, int dtype, const void *u,
                       const void *delta, const void *z, const float *A, const void *B,
                       const void *C, const float *D, const float *delta_bias,
                       int delta_softplus, const double *h0, int zoh, const double *dy,
                       const double *dh_last, double *du, double *ddelta, double *dz,
                       double *dA, double *dB, double *dC, double *dD, double *dbias,
                       double *dh0) {
    if (nrows < 0 || dim <= 0 || dstate <= 0 || seqlen < 0) return -1;
    if (!row_b || !row_d || !u || !delta || !A || !B || !C || !dy) return -1;
    const long long L = seqlen;
    const int N = dstate;
    double *H = (double *)malloc(sizeof(double) * (size_t)((L + 1) * N + 1));  /* h(-1..L-1) */
    double *g = (double *)malloc(sizeof(double) * (size_t)N);
    for (long long r = 0; r < nrows; ++r) {
        const int b = row_b[r], d = row_d[r];
        const long long urow = r * L;
        const long long bcrow = (long long)b * N * L;
        const double bias = delta_bias ? (double)delta_bias[d] : 0.0;
        const double Dd = D ? (double)D[d] : 0.0;
        /* forward, keeping every state: H[(t+1)*N + n] = h_n(t), H[n] = h_n(-1) */
        for (int n = 0; n < N; ++n) H[n] = h0 ? h0[r * N + n] : 0.0;
        for (long long t = 0; t < L; ++t) {
            const double uv = rd(u, urow + t, dtype);
            const double x = rd(delta, urow + t, dtype) + bias;
            const double dt = delta_softplus ? ss_oracle_softplus(x) : x;
            for (int n = 0; n < N; ++n) {
                const double a = (double)A[(long long)d * N + n];
                const double Bv = rd(B, bcrow + (long long)n * L + t, dtype);
                H[(t + 1) * N + n] = exp(dt * a) * H[t * N + n] + input_factor(dt, a, zoh) * Bv * uv;
            }
        }
        /* reverse */
        for (int n = 0; n < N; ++n) g[n] = dh_last ? dh_last[r * N + n] : 0.0;
        double gD = 0.0, gbias = 0.0;
        for (long long t = L - 1; t >= 0; --t) {
            const double uv = rd(u, urow + t, dtype);
            const double x = rd(delta, urow + t, dtype) + bias;
            const double dt = delta_softplus ? ss_oracle_softplus(x) : x;
            double s = Dd * uv;
            for (int n = 0; n < N; ++n)
                s += rd(C, bcrow + (long long)n * L + t, dtype) * H[(t + 1) * N + n];
            double gs = dy[urow + t];
            if (z) {
                const double zv = rd(z, urow + t, dtype);
                const double sg = 1.0 / (1.0 + exp(-zv));
                if (dz) dz[urow + t] = dy[urow + t] * s * sg * (1.0 + zv * (1.0 - sg));
                gs = dy[urow + t] * zv * sg;
            }
            gD += gs * uv;
            double gu = gs * Dd, gdt = 0.0;
            for (int n = 0; n < N; ++n) {
                const double a = (double)A[(long long)d * N + n];
                const double Bv = rd(B, bcrow + (long long)n * L + t, dtype);
                const double Cv = rd(C, bcrow + (long long)n * L + t, dtype);
                const double e = exp(dt * a);
                const double hp = H[t * N + n];
                g[n] += gs * Cv;
                if (dC) dC[bcrow + (long long)n * L + t] += gs * H[(t + 1) * N + n];
                const double f = input_factor(dt, a, zoh);
                /* derivatives of the input factor f(dt, a) */
                double fdt = 1.0, fa = 0.0;
                if (zoh && a != 0.0) {
                    fdt = e;                                  /* d/ddt (e^{dt a}-1)/a */
                    fa = (dt * e) / a - expm1(dt * a) / (a * a);
                } else if (zoh) {
                    fa = 0.5 * dt * dt;                       /* its limit at a = 0 */
                }
                if (dB) dB[bcrow + (long long)n * L + t] += g[n] * f * uv;
                gu += g[n] * f * Bv;
                gdt += g[n] * (a * e * hp + fdt * Bv * uv);
                if (dA) dA[(long long)d * N + n] += g[n] * (dt * e * hp + fa * Bv * uv);
                g[n] *= e;
            }
            const double gx = delta_softplus ? gdt / (1.0 + exp(-x)) : gdt;
            if (du) du[urow + t] = gu;
            if (ddelta) ddelta[urow + t] = gx;
            gbias += gx;
        }
        if (dD) dD[d] += gD;
        if (dbias) dbias[d] += gbias;
        if (dh0)
            for (int n = 0; n < N; ++n) dh0[r * N + n] = g[n];
    }
    free(H);
    free(g);
    return 0;
}
