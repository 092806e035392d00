/*
 * ssm_scan.h -- C ABI of the B300 selective-scan (S6) library, libssmscan.so.
 *
 * The library computes, per channel d of every sequence b, the selective
 * state-space recurrence and its gated readout:
 *
 *   Delta_t   = softplus(delta_t + dt_bias[d])
 *   Abar_t[n] = exp(Delta_t * A[d,n])                  zero-order-hold decay of a diagonal A
 *   h_t[n]    = Abar_t[n] * h_{t-1}[n] + Delta_t * B_t[n] * u_t
 *   y_t       = (sum_n C_t[n] * h_t[n] + Dskip[d] * u_t) * silu(z_t)
 *
 * Sources: the recurrence h_t = Abar_t h_{t-1} + Bbar_t x_t and readout
 * y_t = C_t h_t are stated in eightmm.github.io "Mamba" (Main Claim; Scan View)
 * and portpowered.github.io "Mamba Selective State-Space Module" (Math Or
 * Compute Schema, "Selective state-space step").  The zero-order-hold decay
 * exp(Delta A) and the simplified input term Bbar = Delta B, used in place of
 * the exact zero-order-hold input matrix, are glossed in intvml.com "DL0170
 * Mamba Selective SSM vs Attention" (Mathematical Formulation).  Delta, B and C
 * depend on the token (aipedia.org "Mamba: State Space Models", The Key
 * Innovation: Selectivity); here they arrive precomputed as tensors.  The
 * softplus step, the Dskip term and the silu gate are this library's reading
 * of the "gate path modulates output" stage (eightmm.github.io "Mamba", Block
 * Structure), whose formula the pages do not print.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All pointers are DEVICE pointers (cudaMalloc / torch CUDA memory) on the
 *   current device, except where stated.  The caller owns every buffer; the
 *   library allocates nothing and keeps no pointer after a call returns.
 * - Every tensor is dense and contiguous, row-major, last index fastest:
 *     u, delta, z, y  : [batch, dim, seqlen]          (io type)
 *     A               : [dim, dstate]                 (fp32)
 *     B, C            : [batch, ngroups, dstate, seqlen] (io type)
 *     Dskip, dt_bias  : [dim]                         (fp32)
 *     h0, h_final     : [batch, dim, dstate]          (fp32)
 *   Channel d reads the B/C rows of group g = d / (dim / ngroups).
 * - io: SSM_F32 or SSM_BF16 selects the element type of u, delta, z, B, C, y
 *   (and of the decode token tensors).  Arithmetic and the state are fp32.
 *   bf16 outputs are rounded to nearest even.
 * - Every pointer must be 16-byte aligned (SSM_ERR_MISALIGNED otherwise).
 *   Any seqlen is accepted; rows whose length is not a multiple of the
 *   vector width take a slower element-wise path.
 * - Outputs (y, h_final) must not overlap any input.
 * - stream is a cudaStream_t (NULL = legacy default stream).  Every call is
 *   asynchronous on that stream; argument errors are returned before anything
 *   is enqueued.
 * - Supported dstate: 4, 8, 16, 32, 64, 128, 256 (others return SSM_ERR_UNSUPPORTED),
 *   on every scan entry point and any seqlen (rows that are not whole 16-byte
 *   packets, and the packed sequences of ssm_scan_fwd_varlen, take the
 *   register-staged kernel, which holds the B/C tile of dstate 128 and 256 in
 *   dynamic shared memory).
 * - batch == 0 is an empty problem: the call returns SSM_OK without touching
 *   any pointer.  seqlen == 0 is accepted: nothing is read or written except
 *   h_final (which then equals h0, or zeros).
 * - Environment variables read at each call, for tests and tuning only (the
 *   defaults are the measured best; results differ at most in fp32 rounding
 *   order): SSM_FORCE_PATH=generic (register-staged scan and decode kernels),
 *   SSM_FORCE_LANES, SSM_FORCE_CHUNKS, SSM_FORCE_AGG_LANES (the launch plan),
 *   SSM_FORCE_NW (consumer warps of the warp-specialised pass),
 *   SSM_FORCE_SEG (its time-segmented variant), SSM_SCAN_KERNEL=tma (the
 *   CTA-synchronous pass for single-pass plans), SSM_FUSED_KERNEL=ws (the
 *   warp-specialised fused pass for chunked plans), SSM_DECODE_KERNEL=tma and
 *   SSM_DECODE_TILE=<channels>x<stages> (the bulk-staged decode); and, to
 *   test the bounded waits, SSM_DEBUG_STOP_LOADS_AT_TILE and
 *   SSM_DEBUG_WAIT_BUDGET_US (the warp-specialised pass stops loading at that
 *   tile, and its waits give up after that many microseconds).
 */
#ifndef SSM_SCAN_H
#define SSM_SCAN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SSM_ABI_VERSION 1

typedef enum {
    SSM_OK = 0,
    SSM_ERR_INVALID_ARG = 1,        /* null required pointer, bad size, dim % ngroups != 0 */
    SSM_ERR_UNSUPPORTED = 2,        /* dstate not in {4, 8, ..., 256}, unknown io type */
    SSM_ERR_MISALIGNED = 3,         /* a pointer is not 16-byte aligned */
    SSM_ERR_WORKSPACE_TOO_SMALL = 4,/* workspace_bytes below the size query's answer */
    SSM_ERR_TIMEOUT = 5,            /* a bounded device-side wait gave up (see ssm_workspace_status) */
    SSM_ERR_CUDA = 6                /* a CUDA runtime call or launch failed (see ssm_last_cuda_error) */
} ssm_status_t;

typedef enum {
    SSM_F32 = 0,
    SSM_BF16 = 1
} ssm_dtype_t;

/* SSM_ABI_VERSION of the built library. */
int ssm_abi_version(void);

/* Static, human-readable name of a status code. */
const char *ssm_status_string(ssm_status_t status);

/* The cudaError_t of the most recent SSM_ERR_CUDA returned on this host
 * thread (0 if none). */
int ssm_last_cuda_error(void);

/*
 * ssm_scan_fwd -- selective scan over whole sequences, state starting at 0.
 *
 * Discretisation, recurrence, readout, skip and gate run fused in one kernel;
 * the state h stays in registers and is never written to memory.
 *   u, delta : [batch, dim, seqlen] io type              (required)
 *   z        : [batch, dim, seqlen] io type, or NULL (no gate)
 *   A        : [dim, dstate] fp32                          (required)
 *   B, C     : [batch, ngroups, dstate, seqlen] io type    (required)
 *   Dskip    : [dim] fp32, or NULL (treated as 0)
 *   dt_bias  : [dim] fp32, or NULL (treated as 0)
 *   y        : [batch, dim, seqlen] io type, written       (required)
 * Returns SSM_OK once the work is enqueued on stream.
 */
ssm_status_t ssm_scan_fwd(const void *u, const void *delta, const void *z,
                          const float *A, const void *B, const void *C,
                          const float *Dskip, const float *dt_bias, void *y,
                          int batch, int dim, int dstate, int seqlen, int ngroups,
                          ssm_dtype_t io, void *stream);

/*
 * Bytes of device workspace ssm_scan_fwd_chunked needs for this problem
 * (0 for invalid arguments).  The answer depends only on the arguments.
 */
size_t ssm_scan_fwd_chunked_workspace_size(int batch, int dim, int dstate, int seqlen,
                                           int ngroups, ssm_dtype_t io);

/*
 * The launch plan ssm_scan_fwd_chunked (chunked != 0) or ssm_scan_fwd
 * (chunked == 0) uses for this problem on the current process environment:
 * *lanes = lanes sharing one channel's states, *chunks = time chunks, and
 * *kernels = kernels one call enqueues (3 when chunks > 1: the summary pass,
 * the carry pass and the fused pass; 1 otherwise).  *staged = 1 if the TMA-staged kernels
 * run (row byte length a multiple of 16), 0 for the register-staged fallback.
 * Host-only; returns SSM_ERR_INVALID_ARG / SSM_ERR_UNSUPPORTED like the scan.
 */
ssm_status_t ssm_scan_plan(int batch, int dim, int dstate, int seqlen, int ngroups, ssm_dtype_t io,
                           int chunked, int *lanes, int *chunks, int *kernels, int *staged);

/*
 * ssm_scan_fwd_chunked -- selective scan with a caller-supplied initial state
 * and the final state returned; long sequences are split into time chunks
 * that run in parallel and are stitched by carrying each chunk's state into
 * the next (eightmm.github.io "Mamba", Scan View: the recurrence is a scan
 * over the pairs (Abar_t, Bbar_t x_t), so chunk results compose).
 *
 * Same tensors as ssm_scan_fwd, plus:
 *   h0        : [batch, dim, dstate] fp32 initial state, or NULL (zeros)
 *   h_final   : [batch, dim, dstate] fp32, written with h at t = seqlen-1
 *               (or NULL if not wanted)
 *   workspace : device buffer of at least
 *               ssm_scan_fwd_chunked_workspace_size(...) bytes (always at
 *               least 256), 16-byte aligned; owned by the caller, contents
 *               need not be initialised, must not be shared by calls that
 *               may run concurrently.  It holds a status word and, for
 *               time-chunked runs, one summary (P, E) per channel and chunk:
 *               P[n] = exp(A[d,n] * sum of Delta over the chunk) and E = the
 *               chunk's end state from a zero start (after the call, E of
 *               chunk c holds the state entering chunk c + 1).
 * When the sequence is long relative to the number of channels, the call
 * enqueues three kernels: a summary pass over every chunk but the last, a
 * carry pass that turns the summaries into the state entering each chunk
 * (h0 folded through the summaries of chunks 0..c-1), then the fused pass.  Device-side waits are bounded; if one gives up, the
 * kernel records SSM_ERR_TIMEOUT in the workspace, which ssm_workspace_status
 * reports.
 */
ssm_status_t ssm_scan_fwd_chunked(const void *u, const void *delta, const void *z,
                                  const float *A, const void *B, const void *C,
                                  const float *Dskip, const float *dt_bias,
                                  const float *h0, void *y, float *h_final,
                                  int batch, int dim, int dstate, int seqlen, int ngroups,
                                  ssm_dtype_t io, void *workspace, size_t workspace_bytes,
                                  void *stream);

/*
 * Synchronises stream, then returns the device-side status that the last
 * ssm_scan_fwd_chunked call on this workspace recorded: SSM_OK or
 * SSM_ERR_TIMEOUT (SSM_ERR_CUDA if the read itself failed).
 */
ssm_status_t ssm_workspace_status(const void *workspace, size_t workspace_bytes, void *stream);

/*
 * ssm_scan_fwd_chunked_static -- ssm_scan_fwd_chunked for callers that cannot
 * allocate device memory.  The source pages have no counterpart to this entry
 * point; it exists for integration only.
 *
 * Who needs it: code that is handed only input and output pointers and has no
 * way to obtain a scratch buffer.  Examples are a plugin inside an inference
 * runtime or graph executor whose memory planner owns every device allocation
 * (allocating behind its back breaks its budget, or fails once the pool is
 * reserved), and latency-critical decode or streaming loops that must not call
 * cudaMalloc/cudaFree, which can block until in-flight GPU work finishes.
 *
 * Arguments and results are exactly those of ssm_scan_fwd_chunked without
 * workspace / workspace_bytes; inputs and outputs are still the caller's.  The
 * chunk summaries and the status word live instead in one library-owned
 * scratch array of SSM_STATIC_SCRATCH_BYTES in device global memory:
 *   - every GPU that loads the library holds that array until the process exits;
 *   - the first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current, so make the first call on
 *     a device before any stream capture; the address is looked up again when
 *     the thread's current context is not the one it was found in (after a
 *     cudaDeviceReset, or under a caller's own driver context, where the
 *     library's module and its array are a different instance);
 *   - all calls share the array, which keeps the previous call's contents (each
 *     call clears the status word; the summaries are rewritten before they are
 *     read): calls that can overlap on the GPU -- other streams, other host
 *     threads -- race on it and must be serialised by the caller;
 *   - the call allocates nothing: no cudaMalloc, cudaFree or allocating library.
 * The launch plan uses at most as many time chunks as the array holds
 * summaries for ((chunks - 1) * batch * dim * 2 * dstate * 4 bytes plus 256),
 * down to a single unsplit pass, so no problem is rejected for its size; the
 * result differs from ssm_scan_fwd_chunked's only where that cap changes the
 * chunking (fp32 rounding order).
 * A device-side timeout is reported by ssm_device_status.
 */
#define SSM_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)
ssm_status_t ssm_scan_fwd_chunked_static(const void *u, const void *delta, const void *z,
                                         const float *A, const void *B, const void *C,
                                         const float *Dskip, const float *dt_bias,
                                         const float *h0, void *y, float *h_final,
                                         int batch, int dim, int dstate, int seqlen, int ngroups,
                                         ssm_dtype_t io, void *stream);

/*
 * Synchronises stream, then returns the library's device-wide error word for
 * the current device: SSM_OK, SSM_ERR_TIMEOUT if any kernel of this library
 * gave up on a bounded device-side wait since the word was last cleared, or
 * SSM_ERR_INVALID_ARG if a kernel found an access outside its tensor (packed
 * sequence offsets that do not describe the row, say) and skipped it; the
 * outputs are then unreliable.  clear != 0 resets the word afterwards.
 * SSM_ERR_CUDA if the read itself failed.
 */
ssm_status_t ssm_device_status(int clear, void *stream);

/*
 * Measurement hook.  Registers two CUDA events (cudaEvent_t, created by the
 * caller, who keeps ownership) that every later forward scan call
 * (ssm_scan_fwd, ssm_scan_fwd_chunked, ssm_scan_fwd_chunked_static) made from
 * the calling host thread records on its stream: begin_event immediately
 * before the launch of the fused pass (the kernel that writes y), end_event
 * immediately after it.  cudaEventElapsedTime(begin, end) is then that
 * kernel's device time.  The record between the passes stops the fused pass
 * from starting early (programmatic dependent launch), so use it for timing
 * the kernel, not the call.  NULL, NULL clears the hook.
 * Errors: SSM_ERR_INVALID_ARG when exactly one of the two is NULL.
 */
ssm_status_t ssm_set_pass_timer(void *begin_event, void *end_event);

/*
 * ssm_state_update -- one decode step: every sequence of the batch consumes
 * one token (cuishuaiwen.com "Mamba & State-Space Sequence Models", Core
 * mechanics: inference runs the recurrence, O(1) per step, with a state whose
 * size does not grow with the context; intvml.com, point (5)).
 *   state   : [batch, dim, dstate] fp32, read and overwritten in place
 *   u, delta: [batch, dim] io type                       (required)
 *   z       : [batch, dim] io type, or NULL
 *   A       : [dim, dstate] fp32
 *   B, C    : [batch, ngroups, dstate] io type
 *   Dskip, dt_bias : [dim] fp32, or NULL
 *   y       : [batch, dim] io type, written
 */
ssm_status_t ssm_state_update(float *state, const void *u, const void *delta, const void *z,
                              const float *A, const void *B, const void *C,
                              const float *Dskip, const float *dt_bias, void *y,
                              int batch, int dim, int dstate, int ngroups,
                              ssm_dtype_t io, void *stream);

/*
 * ssm_state_update_pooled -- the decode step on a pool of states (continuous
 * batching: sequences join and leave a serving batch between steps, each
 * keeping its state in a slot of one pool).  Batch row b advances state slot
 * state_indices[b]; an index outside [0, nslots) (a negative one, say) marks a
 * padding row, which touches no state and leaves y[b, :] unwritten.
 *   state_pool    : [nslots, dim, dstate] fp32, the rows' slots read and
 *                   overwritten in place
 *   state_indices : [batch] int32; the ones in [0, nslots) must be distinct
 *   nslots        : slots in the pool (>= 1)
 *   other arguments as in ssm_state_update.
 * ssm_state_update is this call with state_indices = NULL (row b uses slot b,
 * nslots = batch).  With state_indices, nslots must be >= 1; without, it must
 * equal batch (SSM_ERR_INVALID_ARG otherwise).
 */
ssm_status_t ssm_state_update_pooled(float *state_pool, const int *state_indices, int nslots, const void *u,
                                     const void *delta, const void *z, const float *A, const void *B,
                                     const void *C, const float *Dskip, const float *dt_bias, void *y,
                                     int batch, int dim, int dstate, int ngroups, ssm_dtype_t io, void *stream);

/*
 * ssm_scan_fwd_varlen -- the scan over a packed batch of sequences of
 * different lengths (serving: no padding).  The sequences lie end to end
 * along time in one row; sequence s occupies times
 * [cu_seqlens[s], cu_seqlens[s+1]) and is its own run of the recurrence
 * (eightmm.github.io "Mamba", Architecture Contract: sequence in, sequence
 * out, a recurrent state per sequence): its state starts from h0[s] (or 0) and
 * its end state goes to h_final[s].
 *   u, delta, z, y : [dim, total] io type (z nullable)
 *   A              : [dim, dstate] fp32
 *   B, C           : [ngroups, dstate, total] io type
 *   Dskip, dt_bias : [dim] fp32, or NULL
 *   h0, h_final    : [nseq, dim, dstate] fp32, or NULL
 *   cu_seqlens     : [nseq + 1] int32 on the device, cu_seqlens[0] = 0,
 *                    non-decreasing, cu_seqlens[nseq] <= total
 * total is the row length (the stride of every [.., total] tensor); times past
 * the last sequence are padding, read by nothing, and y there is left
 * unwritten.  A total that is a multiple of 8 (bf16) or 4 (fp32) keeps every
 * row on the 16-byte packet grid: the kernel then loads whole packets.
 * The offsets are not read on the host; offsets outside [0, total] are
 * clamped into it on the device (the result is then meaningless, but every
 * access stays in bounds).  One CTA scans one channel block of one sequence,
 * so the parallelism is channel blocks x sequences: a long sequence is not
 * split in time.  Errors as for ssm_scan_fwd (batch is 1); nseq < 1 or a NULL
 * cu_seqlens is SSM_ERR_INVALID_ARG.
 */
ssm_status_t ssm_scan_fwd_varlen(const void *u, const void *delta, const void *z, const float *A,
                                 const void *B, const void *C, const float *Dskip, const float *dt_bias,
                                 const float *h0, const int *cu_seqlens, void *y, float *h_final, int dim,
                                 int dstate, int total, int ngroups, int nseq, ssm_dtype_t io, void *stream);

/*
 * ssm_causal_conv1d_fwd -- the short causal convolution in front of the scan.
 * The pages place a local convolution between the input projection and the
 * selective SSM (eightmm.github.io "Mamba", Block Structure: it adds
 * short-range local context; aipedia.org "Mamba: State Space Models", What a
 * Mamba Block Contains: a short convolution for local mixing) without fixing
 * its form.  This library reads it as one filter of `width` taps per channel
 * (depthwise), causal, with a per-channel bias, followed by silu, so that its
 * output is the scan's u:
 *     out[b,d,l] = act(bias[d] + sum_{k<width} w[d,k] * x[b,d,l-(width-1)+k])
 * Times before 0 read x_prev (the width-1 inputs that preceded the sequence,
 * oldest first) or 0 when x_prev is NULL.
 *   x       : [batch, dim, seqlen] io type
 *   w       : [dim, width] fp32, width in 1..SSM_CONV_MAX_WIDTH
 *   bias    : [dim] fp32, or NULL (0)
 *   x_prev  : [batch, dim, width-1] io type, or NULL
 *   out     : [batch, dim, seqlen] io type, written; must not overlap x
 *   x_last  : [batch, dim, width-1] io type, or NULL; receives the last width-1
 *             inputs of x_prev + x (the history of the next segment); must not
 *             overlap x_prev
 *   silu    : nonzero applies silu, 0 returns the convolution alone
 * All pointers 16-byte aligned (SSM_ERR_MISALIGNED); x == out or
 * x_prev == x_last is SSM_ERR_INVALID_ARG; width outside 1..4 or an unknown io
 * type is SSM_ERR_UNSUPPORTED.  Checks run before anything is enqueued; the
 * call is asynchronous on stream and allocates nothing.
 */
#define SSM_CONV_MAX_WIDTH 4
ssm_status_t ssm_causal_conv1d_fwd(const void *x, const float *w, const float *bias, const void *x_prev,
                                   void *out, void *x_last, int batch, int dim, int seqlen, int width,
                                   int silu, ssm_dtype_t io, void *stream);

/*
 * ssm_causal_conv1d_update -- one decode token of the same convolution
 * (cuishuaiwen.com "Mamba & State-Space Sequence Models", Core mechanics: a
 * decode step works on a state of constant size).  The window is the width-1
 * inputs held in conv_state followed by x; out = act(bias + sum_k w[d,k]
 * window[k]), and conv_state drops its oldest input and appends x.
 *   conv_state : [batch, dim, width-1] io type, read and overwritten in place
 *                (may be NULL when width == 1)
 *   x          : [batch, dim] io type
 *   w, bias    : as in ssm_causal_conv1d_fwd
 *   out        : [batch, dim] io type, written; must not be x
 * Errors as in ssm_causal_conv1d_fwd.
 */
ssm_status_t ssm_causal_conv1d_update(void *conv_state, const void *x, const float *w, const float *bias,
                                      void *out, int batch, int dim, int width, int silu, ssm_dtype_t io,
                                      void *stream);

/*
 * ssm_scan_bwd -- gradients of the selective scan (training).  The pages keep
 * the states on chip and recompute them in the backward pass rather than
 * storing them (intvml.com "DL0170 Mamba Selective SSM vs Attention", the
 * paragraphs after the key points); the gradients are the chain rule through
 * the forward definition of ssm_scan_fwd_chunked.  With s_t the ungated
 * output, g_t = dy_t silu(z_t) and lam_t[n] = dLoss/dh_t[n]
 * (= g_t C_t[n] + Abar_{t+1}[n] lam_{t+1}[n], plus dh_final at the last step):
 *   du_t = g_t D + Delta_t sum_n lam_t[n] B_t[n]
 *   ddelta_t = sigmoid(delta_t + dt_bias) sum_n lam_t[n] (B_t[n] u_t + A[n] Abar_t[n] h_{t-1}[n])
 *   dz_t = dy_t s_t silu'(z_t);  dB_t[n] = sum over the group's channels of lam_t[n] Delta_t u_t;
 *   dC_t[n] = sum over the group's channels of g_t h_t[n];
 *   dA[n] = sum over batch and time of lam_t[n] Delta_t Abar_t[n] h_{t-1}[n];
 *   dDskip = sum g_t u_t;  ddt_bias = sum ddelta_t;  dh0[n] = Abar_0[n] lam_0[n].
 * Inputs: the forward call's inputs (u, delta, z, A, B, C, Dskip, dt_bias, h0
 *   as in ssm_scan_fwd_chunked; z, Dskip, dt_bias, h0 may be NULL), plus
 *   dy         : [batch, dim, seqlen] io type, dLoss/dy
 *   dh_final   : [batch, dim, dstate] fp32, dLoss/dh_final, or NULL (zero)
 * Outputs (all overwritten, none may alias an input):
 *   du, ddelta : [batch, dim, seqlen] io type
 *   dz         : [batch, dim, seqlen] io type; required when z is given, else ignored
 *   dA         : [dim, dstate] fp32
 *   dB, dC     : [batch, ngroups, dstate, seqlen] fp32 (sums over channels)
 *   dDskip     : [dim] fp32; required when Dskip is given, may be NULL otherwise
 *   ddt_bias   : [dim] fp32; required when dt_bias is given, may be NULL otherwise
 *   dh0        : [batch, dim, dstate] fp32, or NULL (not wanted)
 * workspace: device memory of at least ssm_scan_bwd_workspace_size() bytes
 *   (the chunk summaries; 12 * dstate bytes per channel and time chunk: 128 to
 *   160 steps, chosen from the arguments, or 64 from dstate 64 on); may be NULL
 *   when that size is 0.
 * The sums over channels and time are accumulated with fp32 atomic adds, so
 * dA, dB, dC, dDskip and ddt_bias may differ in the last bits between runs.
 * Errors: SSM_ERR_INVALID_ARG (bad size, missing required pointer, an output
 * aliasing an input), SSM_ERR_UNSUPPORTED, SSM_ERR_MISALIGNED,
 * SSM_ERR_WORKSPACE_TOO_SMALL, SSM_ERR_CUDA.
 */
size_t ssm_scan_bwd_workspace_size(int batch, int dim, int dstate, int seqlen, int ngroups, ssm_dtype_t io);

ssm_status_t ssm_scan_bwd(const void *u, const void *delta, const void *z, const float *A, const void *B,
                          const void *C, const float *Dskip, const float *dt_bias, const float *h0,
                          const void *dy, const float *dh_final, void *du, void *ddelta, void *dz, float *dA,
                          float *dB, float *dC, float *dDskip, float *ddt_bias, float *dh0, int batch, int dim,
                          int dstate, int seqlen, int ngroups, ssm_dtype_t io, void *workspace,
                          size_t workspace_bytes, void *stream);

/*
 * ssm_ssd_fwd -- the SSD (structured state space duality, Mamba-2) layer:
 * the selective recurrence with a scalar decay per head, computed chunk by
 * chunk as dense contractions on the tensor cores (eightmm.github.io
 * "Mamba", Relation to Mamba-2: the layer is the causal matrix mixer
 * y_t = sum_{s<=t} C_t (prod_{j=s+1..t} A_j) B_s x_s, evaluated with block/chunk
 * algorithms; intvml.com, engineering paragraph: state sizes up to 256).
 *
 * Head h owns the headdim channels d = h * headdim + p, which share one scalar
 * A[h], the step Delta_t = softplus(delta[b, h, t] + dt_bias[h]) and the skip
 * Dskip[h]; B, C belong to group g = h / (nheads / ngroups).  Per channel and
 * state n:
 *   H_t[p, n] = exp(Delta_t A[h]) H_{t-1}[p, n] + Delta_t B_t[n] x_t[p]
 *   y_t[p]    = (sum_n C_t[n] H_t[p, n] + Dskip[h] x_t[p]) * silu(z_t[p])
 *   x, z, y    : [batch, nheads * headdim, seqlen] bf16 (z may be NULL: no gate)
 *   delta      : [batch, nheads, seqlen] bf16
 *   A          : [nheads] fp32 (required); Dskip, dt_bias : [nheads] fp32 or NULL (0)
 *   B, C       : [batch, ngroups, dstate, seqlen] bf16
 *   h0, h_final: [batch, nheads * headdim, dstate] fp32, or NULL (zeros / not wanted)
 * Supported: io = SSM_BF16, headdim = 64, dstate = 16, 32, 64 or 128 (the
 * smaller sizes run on the 128-state tiles with zero rows: the same time as
 * 128), seqlen a multiple of 8 (16-byte rows); anything else returns
 * SSM_ERR_UNSUPPORTED.  All pointers
 * 16-byte aligned (SSM_ERR_MISALIGNED); outputs must not alias inputs.  The
 * contractions take bf16 operands (the chunk's decayed mixer and the carried
 * state are rounded to bf16 for them) and accumulate in fp32; the carried
 * state itself stays fp32.  Asynchronous on stream; allocates nothing.
 */
ssm_status_t ssm_ssd_fwd(const void *x, const void *delta, const void *z, const float *A, const void *B,
                         const void *C, const float *Dskip, const float *dt_bias, const float *h0, void *y,
                         float *h_final, int batch, int nheads, int headdim, int dstate, int seqlen,
                         int ngroups, ssm_dtype_t io, void *stream);

/*
 * ssm_probe_alu_rates -- measurement helper (no counterpart on the source
 * pages): the arithmetic rates that bound the scan on the current device.
 * One state update needs one MUFU.EX2 (the decay exp(Delta A)) and four fp32
 * FMA-pipe operations (Delta*A, (Delta u)*B, the recurrence's FMA and the
 * readout's FMA).  Runs two short kernels on stream, each with every SM fully
 * occupied by independent chains of one operation, synchronises, and writes:
 *   *ex2_per_sm_ns  : MUFU.EX2 results per SM per nanosecond
 *   *ffma_per_sm_ns : fp32 FMAs per SM per nanosecond
 *   *mix_updates_per_sm_ns (may be NULL): state updates per SM per nanosecond
 *                     of the scan's own per-state instruction mix (B, C from
 *                     shared memory, eight state pairs per thread, eight warps
 *                     per scheduler): what that mix can issue at best
 * sink: a device float the kernels may write (they never do in practice).
 * Errors: SSM_ERR_INVALID_ARG (NULL pointer), SSM_ERR_CUDA.
 */
ssm_status_t ssm_probe_alu_rates(float *sink, double *ex2_per_sm_ns, double *ffma_per_sm_ns,
                                 double *mix_updates_per_sm_ns, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SSM_SCAN_H */
