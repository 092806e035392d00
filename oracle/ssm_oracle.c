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
