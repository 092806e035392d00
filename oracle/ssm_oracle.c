/*
 * ssm_oracle.c -- plain, slow, fp64 CPU oracle for the selective scan (S6).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: it exists so that tests, the smoke check and the CPU
 * baseline leg of the benchmark can compare the CUDA library against an
 * obviously correct sequential recurrence.  It shares no code, header,
 * table or helper with the CUDA library.
 *
 * What it computes (the plain definition, written out):
 *
 *   Discretisation (intvml.com "DL0170 Mamba Selective SSM vs Attention",
 *   Mathematical Formulation: zero-order-hold decay Abar = exp(Delta*A) for a
 *   diagonal A, and the simplified input term Bbar = Delta*B used in place of
 *   the exact zero-order-hold input matrix):
 *       Delta_t   = softplus(delta_t + dt_bias[d])
 *       Abar_t[n] = exp(Delta_t * A[d,n])
 *       Bbar_t[n] * x_t = Delta_t * B_t[n] * u_t
 *
 *   Recurrence and readout (eightmm.github.io "Mamba", Main Claim and Scan
 *   View; portpowered.github.io "Mamba Selective State-Space Module", Math Or
 *   Compute Schema, "Selective state-space step"):
 *       h_t = Abar_t * h_{t-1} + Bbar_t x_t        (elementwise over n)
 *       y_t = sum_n C_t[n] * h_t[n]
 *
 *   Skip and gate: the pages say only that a gate path modulates the block
 *   output (eightmm.github.io "Mamba", Block Structure).  The reading taken is
 *       y_t = (sum_n C_t[n] h_t[n] + Dskip[d] * u_t) * silu(z_t),
 *   with the gate dropped when z is NULL.
 *
 *   Initial condition: h_0 = 0 unless the caller passes h0 (intvml.com, where
 *   the formulation names a required initial condition whose value was lost).
 *
 *   Decode (cuishuaiwen.com "Mamba & State-Space Sequence Models", Core
 *   mechanics: inference runs the recurrence one token at a time with a state
 *   of constant size): the same body for a single t, with h read from and
 *   written back to the caller's state.
 *
 * Layouts (all row-major, contiguous, last index fastest):
 *   u, delta, z, y : [batch, dim, seqlen]
 *   A              : [dim, dstate]
 *   B, C           : [batch, ngroups, dstate, seqlen]   (decode: [batch, ngroups, dstate])
 *   Dskip, dt_bias : [dim]
 *   h0, h_final, state : [batch, dim, dstate]
 *   channel d reads group g = d / (dim / ngroups).
 *
 * Everything is double precision; inputs that the GPU sees as bf16 or fp32
 * arrive here widened exactly.  softplus has no threshold: it is evaluated as
 * max(x, 0) + log1p(exp(-|x|)).
 *
 * Parallelism: (batch, channel) pairs are split over POSIX threads; each
 * channel remains one sequential loop over time.
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdlib.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1

static double softplus(double x) {
    return (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x)));
}

static double silu(double z) {
    return z / (1.0 + exp(-z));
}

typedef struct {
    const double *u, *delta, *z, *A, *B, *C, *Dskip, *dt_bias, *h0;
    double *y, *h_final;
    int batch, dim, dstate, seqlen, ngroups;
    long first, last; /* range of flattened (b, d) handled by one worker */
} scan_job;

/* One channel: the sequential recurrence over time, state in a local array. */
static void scan_channel(const scan_job *J, int b, int d, double *h) {
    const int N = J->dstate, L = J->seqlen;
    const int g = d / (J->dim / J->ngroups);
    const size_t row = ((size_t)b * J->dim + d) * (size_t)L;
    const size_t bc = ((size_t)b * J->ngroups + g) * (size_t)N * (size_t)L;
    const double dskip = J->Dskip ? J->Dskip[d] : 0.0;
    const double bias = J->dt_bias ? J->dt_bias[d] : 0.0;

    for (int n = 0; n < N; n++)
        h[n] = J->h0 ? J->h0[((size_t)b * J->dim + d) * N + n] : 0.0;

    for (int t = 0; t < L; t++) {
        const double ut = J->u[row + t];
        const double dt = softplus(J->delta[row + t] + bias);
        double acc = 0.0;
        for (int n = 0; n < N; n++) {
            const double abar = exp(dt * J->A[(size_t)d * N + n]);
            const double bx = dt * J->B[bc + (size_t)n * L + t] * ut;
            h[n] = abar * h[n] + bx;
            acc += J->C[bc + (size_t)n * L + t] * h[n];
        }
        double yt = acc + dskip * ut;
        if (J->z) yt *= silu(J->z[row + t]);
        J->y[row + t] = yt;
    }
    if (J->h_final)
        for (int n = 0; n < N; n++)
            J->h_final[((size_t)b * J->dim + d) * N + n] = h[n];
}

static void *scan_worker(void *arg) {
    const scan_job *J = (const scan_job *)arg;
    double *h = (double *)malloc(sizeof(double) * (size_t)J->dstate);
    if (!h) return NULL;
    for (long i = J->first; i < J->last; i++)
        scan_channel(J, (int)(i / J->dim), (int)(i % J->dim), h);
    free(h);
    return NULL;
}

static int check_dims(int batch, int dim, int dstate, int seqlen, int ngroups) {
    if (batch <= 0 || dim <= 0 || dstate <= 0 || seqlen < 0 || ngroups <= 0) return 0;
    if (dim % ngroups != 0) return 0;
    return 1;
}

/* Selective scan over a whole sequence.  z, Dskip, dt_bias, h0 and h_final
 * may be NULL.  Returns ORACLE_OK or ORACLE_BAD_ARG. */
int oracle_scan(const double *u, const double *delta, const double *z,
                const double *A, const double *B, const double *C,
                const double *Dskip, const double *dt_bias, const double *h0,
                double *y, double *h_final,
                int batch, int dim, int dstate, int seqlen, int ngroups,
                int nthreads) {
    if (!check_dims(batch, dim, dstate, seqlen, ngroups)) return ORACLE_BAD_ARG;
    if (!u || !delta || !A || !B || !C || !y) return ORACLE_BAD_ARG;
    const long total = (long)batch * dim;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > total) nthreads = (int)total;

    scan_job *jobs = (scan_job *)malloc(sizeof(scan_job) * (size_t)nthreads);
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!jobs || !tid) { free(jobs); free(tid); return ORACLE_BAD_ARG; }
    for (int k = 0; k < nthreads; k++) {
        scan_job J = {u, delta, z, A, B, C, Dskip, dt_bias, h0, y, h_final,
                      batch, dim, dstate, seqlen, ngroups,
                      total * k / nthreads, total * (k + 1) / nthreads};
        jobs[k] = J;
    }
    if (nthreads == 1) {
        scan_worker(&jobs[0]);
    } else {
        for (int k = 0; k < nthreads; k++) pthread_create(&tid[k], NULL, scan_worker, &jobs[k]);
        for (int k = 0; k < nthreads; k++) pthread_join(tid[k], NULL);
    }
    free(jobs);
    free(tid);
    return ORACLE_OK;
}

/* One decode step: state[b,d,:] is read, advanced by one token and written
 * back; y[b,d] receives the gated readout.  Token tensors are u, delta, z:
 * [batch, dim]; B, C: [batch, ngroups, dstate]. */
int oracle_state_update(double *state, const double *u, const double *delta,
                        const double *z, const double *A, const double *B,
                        const double *C, const double *Dskip,
                        const double *dt_bias, double *y,
                        int batch, int dim, int dstate, int ngroups) {
    if (!check_dims(batch, dim, dstate, 1, ngroups)) return ORACLE_BAD_ARG;
    if (!state || !u || !delta || !A || !B || !C || !y) return ORACLE_BAD_ARG;
    const int N = dstate;
    for (int b = 0; b < batch; b++) {
        for (int d = 0; d < dim; d++) {
            const int g = d / (dim / ngroups);
            const size_t bd = (size_t)b * dim + d;
            const size_t bc = ((size_t)b * ngroups + g) * (size_t)N;
            const double ut = u[bd];
            const double dt = softplus(delta[bd] + (dt_bias ? dt_bias[d] : 0.0));
            double acc = 0.0;
            for (int n = 0; n < N; n++) {
                double *h = &state[bd * N + n];
                *h = exp(dt * A[(size_t)d * N + n]) * (*h) + dt * B[bc + n] * ut;
                acc += C[bc + n] * (*h);
            }
            double yt = acc + (Dskip ? Dskip[d] : 0.0) * ut;
            if (z) yt *= silu(z[bd]);
            y[bd] = yt;
        }
    }
    return ORACLE_OK;
}

/*
 * Short causal convolution in front of the scan.
 *
 * The pages place a local convolution between the input projection and the
 * selective SSM (eightmm.github.io "Mamba", Block Structure: it adds
 * short-range local context; aipedia.org "Mamba: State Space Models", What a
 * Mamba Block Contains: a short convolution for local mixing) but give
 * neither its width nor its form.  The reading taken: one filter per channel
 * (depthwise), causal, W taps, a per-channel bias, then silu, so that its
 * output is the scan's input u:
 *
 *     out[b,d,l] = act( bias[d] + sum_{k=0}^{W-1} w[d,k] * x[b,d,l-(W-1)+k] )
 *
 * A time before 0 reads the caller's history x_prev[b,d,:] (the W-1 inputs
 * that preceded the sequence, oldest first) or 0 without one.  act is silu
 * when `silu_act` is set, else the identity.  x_last (optional) receives the
 * last W-1 inputs of history + sequence: the history of the next segment.
 *
 * Layouts: x, out [batch, dim, seqlen]; w [dim, W]; bias [dim];
 * x_prev, x_last [batch, dim, W-1].
 */
static double conv_input(const double *x, const double *x_prev, size_t row, size_t prow,
                         int W, long t) {
    if (t >= 0) return x[row + (size_t)t];
    /* t in [-(W-1), -1]: history slot (W-1) + t */
    return x_prev ? x_prev[prow + (size_t)((W - 1) + t)] : 0.0;
}

int oracle_causal_conv1d(const double *x, const double *w, const double *bias,
                         const double *x_prev, double *out, double *x_last,
                         int batch, int dim, int seqlen, int width, int silu_act) {
    if (batch <= 0 || dim <= 0 || seqlen < 0 || width < 1) return ORACLE_BAD_ARG;
    if (!w || (seqlen > 0 && (!x || !out))) return ORACLE_BAD_ARG;
    const int W = width;
    for (int b = 0; b < batch; b++) {
        for (int d = 0; d < dim; d++) {
            const size_t bd = (size_t)b * dim + d;
            const size_t row = bd * (size_t)seqlen;
            const size_t prow = bd * (size_t)(W - 1);
            for (long l = 0; l < seqlen; l++) {
                double acc = bias ? bias[d] : 0.0;
                for (int k = 0; k < W; k++)
                    acc += w[(size_t)d * W + k] * conv_input(x, x_prev, row, prow, W, l - (W - 1) + k);
                out[row + (size_t)l] = silu_act ? silu(acc) : acc;
            }
            if (x_last) {
                for (int k = 0; k < W - 1; k++)
                    x_last[prow + k] = conv_input(x, x_prev, row, prow, W, (long)seqlen - (W - 1) + k);
            }
        }
    }
    return ORACLE_OK;
}

/* One decode token of the convolution: the window is the W-1 inputs held in
 * conv_state[b,d,:] (oldest first) followed by x[b,d]; out[b,d] = act(bias +
 * sum_k w[d,k] window[k]), and the state drops its oldest input and appends
 * x[b,d]. */
int oracle_causal_conv1d_update(double *conv_state, const double *x, const double *w,
                                const double *bias, double *out,
                                int batch, int dim, int width, int silu_act) {
    if (batch <= 0 || dim <= 0 || width < 1) return ORACLE_BAD_ARG;
    if (!x || !w || !out || (width > 1 && !conv_state)) return ORACLE_BAD_ARG;
    const int W = width;
    for (int b = 0; b < batch; b++) {
        for (int d = 0; d < dim; d++) {
            const size_t bd = (size_t)b * dim + d;
            double *st = conv_state ? conv_state + bd * (size_t)(W - 1) : NULL;
            double acc = bias ? bias[d] : 0.0;
            for (int k = 0; k < W - 1; k++) acc += w[(size_t)d * W + k] * st[k];
            acc += w[(size_t)d * W + (W - 1)] * x[bd];
            out[bd] = silu_act ? silu(acc) : acc;
            for (int k = 0; k + 1 < W - 1; k++) st[k] = st[k + 1];
            if (W > 1) st[W - 2] = x[bd];
        }
    }
    return ORACLE_OK;
}

/*
 * Packed variable-length batch (serving: a batch of sequences of different
 * lengths without padding).  The pages treat the layer as sequence in,
 * sequence out with a recurrent state per sequence (eightmm.github.io
 * "Mamba", Architecture Contract); packing several sequences end to end along
 * time is the plainest layout for a batch of unequal lengths, and each
 * sequence is then its own run of the recurrence:
 *
 *   sequence s occupies times [cu_seqlens[s], cu_seqlens[s+1]) of one row;
 *   its state starts from h0[s] (or 0) at its first token, every token is the
 *   step of oracle_scan, and its end state goes to h_final[s].
 *
 * Layouts: u, delta, z, y [dim, T]; B, C [ngroups, dstate, T];
 * h0, h_final [nseq, dim, dstate]; cu_seqlens [nseq + 1], non-decreasing,
 * cu_seqlens[0] = 0 and cu_seqlens[nseq] <= T (T is the row length; times
 * past the last sequence are padding, read by nothing and left unwritten).
 */
int oracle_scan_varlen(const double *u, const double *delta, const double *z,
                       const double *A, const double *B, const double *C,
                       const double *Dskip, const double *dt_bias, const double *h0,
                       const int *cu_seqlens, double *y, double *h_final,
                       int dim, int dstate, int total, int ngroups, int nseq) {
    if (dim <= 0 || dstate <= 0 || total < 0 || ngroups <= 0 || nseq < 1 || dim % ngroups != 0)
        return ORACLE_BAD_ARG;
    if (!cu_seqlens || !A || (total > 0 && (!u || !delta || !B || !C || !y))) return ORACLE_BAD_ARG;
    if (cu_seqlens[0] != 0 || cu_seqlens[nseq] > total) return ORACLE_BAD_ARG;
    for (int s = 0; s < nseq; s++)
        if (cu_seqlens[s + 1] < cu_seqlens[s]) return ORACLE_BAD_ARG;
    const int N = dstate, T = total;
    double *h = (double *)malloc(sizeof(double) * (size_t)N);
    if (!h) return ORACLE_BAD_ARG;
    for (int d = 0; d < dim; d++) {
        const int g = d / (dim / ngroups);
        const size_t row = (size_t)d * (size_t)T;
        const size_t bc = (size_t)g * (size_t)N * (size_t)T;
        const double dskip = Dskip ? Dskip[d] : 0.0;
        const double bias = dt_bias ? dt_bias[d] : 0.0;
        for (int s = 0; s < nseq; s++) {
            for (int n = 0; n < N; n++)
                h[n] = h0 ? h0[((size_t)s * dim + d) * N + n] : 0.0;
            for (int t = cu_seqlens[s]; t < cu_seqlens[s + 1]; t++) {
                const double ut = u[row + t];
                const double dt = softplus(delta[row + t] + bias);
                double acc = 0.0;
                for (int n = 0; n < N; n++) {
                    h[n] = exp(dt * A[(size_t)d * N + n]) * h[n] + dt * B[bc + (size_t)n * T + t] * ut;
                    acc += C[bc + (size_t)n * T + t] * h[n];
                }
                double yv = acc + dskip * ut;
                if (z) yv *= silu(z[row + t]);
                y[row + t] = yv;
            }
            if (h_final)
                for (int n = 0; n < N; n++) h_final[((size_t)s * dim + d) * N + n] = h[n];
        }
    }
    free(h);
    return ORACLE_OK;
}

/* One decode step on a pool of states (continuous batching): batch row b
 * advances state slot state_indices[b] of state_pool [nslots, dim, dstate]
 * by its token; a negative index marks a padding row, which touches no state
 * and leaves y[b, :] unwritten.  Otherwise the step of oracle_state_update. */
int oracle_state_update_indexed(double *state_pool, const int *state_indices, int nslots,
                                const double *u, const double *delta, const double *z,
                                const double *A, const double *B, const double *C,
                                const double *Dskip, const double *dt_bias, double *y,
                                int batch, int dim, int dstate, int ngroups) {
    if (!check_dims(batch, dim, dstate, 1, ngroups) || nslots < 1) return ORACLE_BAD_ARG;
    if (!state_pool || !state_indices || !u || !delta || !A || !B || !C || !y) return ORACLE_BAD_ARG;
    const int N = dstate;
    for (int b = 0; b < batch; b++) {
        const int slot = state_indices[b];
        if (slot < 0) continue;
        if (slot >= nslots) return ORACLE_BAD_ARG;
        for (int d = 0; d < dim; d++) {
            const int g = d / (dim / ngroups);
            const size_t bd = (size_t)b * dim + d;
            const size_t bc = ((size_t)b * ngroups + g) * (size_t)N;
            double *h = &state_pool[((size_t)slot * dim + d) * N];
            const double ut = u[bd];
            const double dt = softplus(delta[bd] + (dt_bias ? dt_bias[d] : 0.0));
            double acc = 0.0;
            for (int n = 0; n < N; n++) {
                h[n] = exp(dt * A[(size_t)d * N + n]) * h[n] + dt * B[bc + n] * ut;
                acc += C[bc + n] * h[n];
            }
            double yv = acc + (Dskip ? Dskip[d] : 0.0) * ut;
            if (z) yv *= silu(z[bd]);
            y[bd] = yv;
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------
 * Backward pass of the scan: the gradients of a scalar loss with respect to
 * every input, given its gradient dy with respect to y (and, optionally, dhf
 * with respect to the final state).
 *
 * The pages say that training keeps the states on chip and recomputes them in
 * the backward pass (intvml.com "DL0170 Mamba Selective SSM vs Attention",
 * the paragraphs after the list of key points); they print no gradient
 * formulas.  The reading taken is the plain chain rule through the forward
 * definition above, written out per channel.  With s_t the ungated output
 * (sum_n C_t[n] h_t[n] + Dskip u_t), g_t = dy_t * silu(z_t) its gradient,
 * and lam_t[n] the gradient of the loss with respect to h_t[n]:
 *
 *   lam_t[n]   = g_t C_t[n] + Abar_{t+1}[n] lam_{t+1}[n]   (lam_{L-1} gets + dhf[n])
 *   dz_t       = dy_t * s_t * silu'(z_t),  silu'(z) = sig(z) (1 + z (1 - sig(z)))
 *   dC_t[n]    = g_t h_t[n]
 *   dB_t[n]    = lam_t[n] Delta_t u_t
 *   du_t       = g_t Dskip + Delta_t sum_n lam_t[n] B_t[n]
 *   dDelta_t   = sum_n lam_t[n] (B_t[n] u_t + A[n] Abar_t[n] h_{t-1}[n])
 *   ddelta_t   = dDelta_t * sig(delta_t + dt_bias)        (softplus' = sigmoid)
 *   dA[n]     += lam_t[n] Delta_t Abar_t[n] h_{t-1}[n]
 *   dDskip    += g_t u_t,   ddt_bias += ddelta_t,   dh0[n] = Abar_0[n] lam_0[n]
 *
 * dB, dC sum over the channels of a group, dA, dDskip, ddt_bias over the
 * batch (and time).  Each channel first runs the forward recurrence keeping
 * every state, then walks time backwards.
 * ---------------------------------------------------------------------- */

static double sigmoid(double x) {
    return x >= 0.0 ? 1.0 / (1.0 + exp(-x)) : exp(x) / (1.0 + exp(x));
}

typedef struct {
    const double *u, *delta, *z, *A, *B, *C, *Dskip, *dt_bias, *h0, *dy, *dhf;
    double *du, *ddelta, *dz, *dh0;
    double *dA, *dB, *dC, *dDskip, *ddt_bias; /* this worker's private sums */
    int batch, dim, dstate, seqlen, ngroups;
    long first, last;
    int ok;
} bwd_job;

static void *bwd_worker(void *arg) {
    bwd_job *J = (bwd_job *)arg;
    const int N = J->dstate, L = J->seqlen;
    /* hs[t * N + n] = h_t[n] for t = -1 .. L-1 (row 0 holds h_{-1} = h0) */
    double *hs = (double *)malloc(sizeof(double) * (size_t)(L + 1) * (size_t)N);
    double *dts = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
    double *lam = (double *)malloc(sizeof(double) * (size_t)N);
    if (!hs || !dts || !lam) { free(hs); free(dts); free(lam); J->ok = 0; return NULL; }
    for (long i = J->first; i < J->last; i++) {
        const int b = (int)(i / J->dim), d = (int)(i % J->dim);
        const int g = d / (J->dim / J->ngroups);
        const size_t row = ((size_t)b * J->dim + d) * (size_t)L;
        const size_t bc = ((size_t)b * J->ngroups + g) * (size_t)N * (size_t)L;
        const size_t st = ((size_t)b * J->dim + d) * (size_t)N;
        const double *Ad = J->A + (size_t)d * N;
        const double dskip = J->Dskip ? J->Dskip[d] : 0.0;
        const double bias = J->dt_bias ? J->dt_bias[d] : 0.0;

        /* forward, keeping every state */
        for (int n = 0; n < N; n++) hs[n] = J->h0 ? J->h0[st + n] : 0.0;
        for (int t = 0; t < L; t++) {
            const double x = J->delta[row + t] + bias;
            const double dt = softplus(x);
            dts[t] = dt;
            for (int n = 0; n < N; n++)
                hs[(size_t)(t + 1) * N + n] = exp(dt * Ad[n]) * hs[(size_t)t * N + n]
                                              + dt * J->B[bc + (size_t)n * L + t] * J->u[row + t];
        }

        /* backward over time */
        for (int n = 0; n < N; n++) lam[n] = J->dhf ? J->dhf[st + n] : 0.0;  /* carried from t+1 */
        for (int t = L - 1; t >= 0; t--) {
            const double ut = J->u[row + t], dt = dts[t];
            const double *hprev = hs + (size_t)t * N, *hcur = hs + (size_t)(t + 1) * N;
            double s = dskip * ut;
            for (int n = 0; n < N; n++) s += J->C[bc + (size_t)n * L + t] * hcur[n];
            double gt = J->dy[row + t];
            if (J->z) {
                const double zt = J->z[row + t], sg = sigmoid(zt);
                J->dz[row + t] = J->dy[row + t] * s * sg * (1.0 + zt * (1.0 - sg));
                gt *= silu(zt);
            }
            double dsum_b = 0.0, ddelta_t = 0.0;
            for (int n = 0; n < N; n++) {
                const size_t k = bc + (size_t)n * L + t;
                const double abar = exp(dt * Ad[n]);
                const double l = gt * J->C[k] + lam[n];     /* lam_t[n] */
                J->dC[k] += gt * hcur[n];
                J->dB[k] += l * dt * ut;
                dsum_b += l * J->B[k];
                ddelta_t += l * (J->B[k] * ut + Ad[n] * abar * hprev[n]);
                J->dA[(size_t)d * N + n] += l * dt * abar * hprev[n];
                lam[n] = abar * l;                           /* passes to t-1 */
            }
            J->du[row + t] = gt * dskip + dt * dsum_b;
            const double dd = ddelta_t * sigmoid(J->delta[row + t] + bias);
            J->ddelta[row + t] = dd;
            J->dDskip[d] += gt * ut;
            J->ddt_bias[d] += dd;
        }
        if (J->dh0)
            for (int n = 0; n < N; n++) J->dh0[st + n] = lam[n];
    }
    free(hs); free(dts); free(lam);
    J->ok = 1;
    return NULL;
}

/* Gradients of the scan.  Inputs as oracle_scan plus dy [batch, dim, L] and
 * dhf [batch, dim, N] (may be NULL: zero).  Outputs (all overwritten): du,
 * ddelta [batch, dim, L]; dz [batch, dim, L] (ignored when z is NULL); dA
 * [dim, N]; dB, dC [batch, G, N, L]; dDskip, ddt_bias [dim]; dh0 [batch, dim,
 * N] (may be NULL). */
int oracle_scan_bwd(const double *u, const double *delta, const double *z,
                    const double *A, const double *B, const double *C,
                    const double *Dskip, const double *dt_bias, const double *h0,
                    const double *dy, const double *dhf,
                    double *du, double *ddelta, double *dz, double *dA, double *dB, double *dC,
                    double *dDskip, double *ddt_bias, double *dh0,
                    int batch, int dim, int dstate, int seqlen, int ngroups, int nthreads) {
    if (!check_dims(batch, dim, dstate, seqlen, ngroups)) return ORACLE_BAD_ARG;
    if (!u || !delta || !A || !B || !C || !dy || !du || !ddelta || !dA || !dB || !dC || !dDskip || !ddt_bias)
        return ORACLE_BAD_ARG;
    if (z && !dz) return ORACLE_BAD_ARG;
    const long total = (long)batch * dim;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > total) nthreads = (int)total;
    const size_t nA = (size_t)dim * dstate, nBC = (size_t)batch * ngroups * dstate * (size_t)seqlen;
    const size_t per = nA + 2 * nBC + 2 * (size_t)dim; /* private sums of one worker */
    bwd_job *jobs = (bwd_job *)malloc(sizeof(bwd_job) * (size_t)nthreads);
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    double *sums = (double *)calloc((size_t)nthreads * per, sizeof(double));
    if (!jobs || !tid || !sums) { free(jobs); free(tid); free(sums); return ORACLE_BAD_ARG; }
    for (int k = 0; k < nthreads; k++) {
        double *p = sums + (size_t)k * per;
        bwd_job J = {u, delta, z, A, B, C, Dskip, dt_bias, h0, dy, dhf,
                     du, ddelta, dz, dh0,
                     p, p + nA, p + nA + nBC, p + nA + 2 * nBC, p + nA + 2 * nBC + dim,
                     batch, dim, dstate, seqlen, ngroups,
                     total * k / nthreads, total * (k + 1) / nthreads, 0};
        jobs[k] = J;
    }
    if (nthreads == 1) {
        bwd_worker(&jobs[0]);
    } else {
        for (int k = 0; k < nthreads; k++) pthread_create(&tid[k], NULL, bwd_worker, &jobs[k]);
        for (int k = 0; k < nthreads; k++) pthread_join(tid[k], NULL);
    }
    int ok = 1;
    for (int k = 0; k < nthreads; k++) ok &= jobs[k].ok;
    /* add up the workers' sums */
    for (size_t i = 0; i < nA; i++) dA[i] = 0.0;
    for (size_t i = 0; i < nBC; i++) { dB[i] = 0.0; dC[i] = 0.0; }
    for (int i = 0; i < dim; i++) { dDskip[i] = 0.0; ddt_bias[i] = 0.0; }
    for (int k = 0; k < nthreads; k++) {
        const bwd_job *J = &jobs[k];
        for (size_t i = 0; i < nA; i++) dA[i] += J->dA[i];
        for (size_t i = 0; i < nBC; i++) { dB[i] += J->dB[i]; dC[i] += J->dC[i]; }
        for (int i = 0; i < dim; i++) { dDskip[i] += J->dDskip[i]; ddt_bias[i] += J->ddt_bias[i]; }
    }
    free(jobs); free(tid); free(sums);
    return ok ? ORACLE_OK : ORACLE_BAD_ARG;
}

/* ------------------------------------------------------------------------
 * Structured state space duality (SSD, the Mamba-2 layer): the same
 * recurrence with a scalar decay per head.  eightmm.github.io "Mamba",
 * Relation to Mamba-2: Mamba-2 computes the causal matrix mixer
 * y_t = sum_{i<=t} C_t (prod_{j=i+1..t} A_j) B_i x_i with faster block/chunk
 * algorithms, and intvml.com (engineering paragraph) has it raise the state
 * size N from 16 to as much as 256.  The reading taken here (the pages give
 * no formula for the per-head parameters): head h owns headdim channels
 * d = h * headdim + p that share one scalar A[h], one step
 *     Delta_t = softplus(delta[b, h, t] + dt_bias[h])
 * and one skip weight Dskip[h]; B and C are shared by the heads of a group
 * (g = h / (nheads / ngroups)); per channel d and state n
 *     H_t[p, n] = exp(Delta_t * A[h]) * H_{t-1}[p, n] + Delta_t * B_t[n] * x_t[p]
 *     y_t[p]    = (sum_n C_t[n] * H_t[p, n] + Dskip[h] * x_t[p]) * silu(z_t[p])
 * with the gate dropped when z is NULL.
 *
 * Layouts: x, z, y [batch, nheads * headdim, L]; delta [batch, nheads, L];
 * A, Dskip, dt_bias [nheads]; B, C [batch, ngroups, N, L]; h0, h_final
 * [batch, nheads * headdim, N].
 * ------------------------------------------------------------------------ */
typedef struct {
    const double *x, *delta, *z, *A, *B, *C, *Dskip, *dt_bias, *h0;
    double *y, *h_final;
    int batch, nheads, headdim, dstate, seqlen, ngroups;
    long first, last; /* range of flattened (b, h) handled by one worker */
} ssd_job;

static void ssd_head(const ssd_job *J, int b, int h, double *H) {
    const int P = J->headdim, N = J->dstate, L = J->seqlen;
    const int dim = J->nheads * P;
    const int g = h / (J->nheads / J->ngroups);
    const size_t bc = ((size_t)b * J->ngroups + g) * (size_t)N * (size_t)L;
    const size_t drow = ((size_t)b * J->nheads + h) * (size_t)L;
    const double a = J->A[h];
    const double dskip = J->Dskip ? J->Dskip[h] : 0.0;
    const double bias = J->dt_bias ? J->dt_bias[h] : 0.0;

    for (int p = 0; p < P; p++)
        for (int n = 0; n < N; n++)
            H[(size_t)p * N + n] = J->h0 ? J->h0[((size_t)b * dim + (size_t)h * P + p) * N + n] : 0.0;

    for (int t = 0; t < L; t++) {
        const double dt = softplus(J->delta[drow + t] + bias);
        const double abar = exp(dt * a);
        for (int p = 0; p < P; p++) {
            const size_t row = ((size_t)b * dim + (size_t)h * P + p) * (size_t)L;
            const double xt = J->x[row + t];
            double acc = 0.0;
            for (int n = 0; n < N; n++) {
                double *hp = &H[(size_t)p * N + n];
                *hp = abar * *hp + dt * J->B[bc + (size_t)n * L + t] * xt;
                acc += J->C[bc + (size_t)n * L + t] * *hp;
            }
            double yt = acc + dskip * xt;
            if (J->z) yt = yt * silu(J->z[row + t]);
            J->y[row + t] = yt;
        }
    }
    if (J->h_final)
        for (int p = 0; p < P; p++)
            for (int n = 0; n < N; n++)
                J->h_final[((size_t)b * dim + (size_t)h * P + p) * N + n] = H[(size_t)p * N + n];
}

static void *ssd_worker(void *arg) {
    const ssd_job *J = (const ssd_job *)arg;
    double *H = (double *)malloc(sizeof(double) * (size_t)J->headdim * (size_t)J->dstate);
    if (!H) return NULL;
    for (long i = J->first; i < J->last; i++)
        ssd_head(J, (int)(i / J->nheads), (int)(i % J->nheads), H);
    free(H);
    return NULL;
}

/* SSD layer over whole sequences.  z, Dskip, dt_bias, h0 and h_final may be
 * NULL.  Returns ORACLE_OK or ORACLE_BAD_ARG. */
int oracle_ssd(const double *x, const double *delta, const double *z,
               const double *A, const double *B, const double *C,
               const double *Dskip, const double *dt_bias, const double *h0,
               double *y, double *h_final,
               int batch, int nheads, int headdim, int dstate, int seqlen, int ngroups,
               int nthreads) {
    if (batch <= 0 || nheads <= 0 || headdim <= 0 || dstate <= 0 || seqlen < 0 || ngroups <= 0) return ORACLE_BAD_ARG;
    if (nheads % ngroups != 0) return ORACLE_BAD_ARG;
    if (!x || !delta || !A || !B || !C || !y) return ORACLE_BAD_ARG;
    const long total = (long)batch * nheads;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > total) nthreads = (int)total;
    ssd_job *jobs = (ssd_job *)malloc(sizeof(ssd_job) * (size_t)nthreads);
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!jobs || !tid) { free(jobs); free(tid); return ORACLE_BAD_ARG; }
    for (int k = 0; k < nthreads; k++) {
        ssd_job *J = &jobs[k];
        J->x = x; J->delta = delta; J->z = z; J->A = A; J->B = B; J->C = C;
        J->Dskip = Dskip; J->dt_bias = dt_bias; J->h0 = h0; J->y = y; J->h_final = h_final;
        J->batch = batch; J->nheads = nheads; J->headdim = headdim; J->dstate = dstate;
        J->seqlen = seqlen; J->ngroups = ngroups;
        J->first = total * k / nthreads;
        J->last = total * (k + 1) / nthreads;
        pthread_create(&tid[k], NULL, ssd_worker, J);
    }
    for (int k = 0; k < nthreads; k++) pthread_join(tid[k], NULL);
    free(jobs);
    free(tid);
    return ORACLE_OK;
}
