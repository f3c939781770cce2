/*
 * ssd.h -- C ABI of the GB300 (sm_103a) Mamba-2 SSD chunked forward.
 *
 * The operation.  The public call of the "Mamba-2 SSD for Ascend NPU" README
 * ("Usage", "Implementation": mamba2_ssd_fwd(x, dt, A, B, C, chunk_size,
 * dt_softplus, return_final_state) with D, z, dt_bias, dt_limit and
 * initial_states): for every batch b, head h and token t, with group
 * g = h / (H/G),
 *
 *     d_t = clamp(softplus(dt[b,t,h] + dt_bias[h]))   bias / softplus / clamp optional
 *     h_t = exp(d_t * A[h]) * h_{t-1} + d_t * x[b,t,h,:] (outer) B[b,t,g,:]
 *     y[b,t,h,:] = (h_t . C[b,t,g,:] + D[h] * x[b,t,h,:]) * silu(z[b,t,h,:])
 *
 * with h_{-1} = initial_state[b,h] (or 0) and final_state[b,h] = h_{L-1}.
 * It is computed chunk by chunk (ops-transformer MambaV2 article, section 2:
 * chunk_cumsum -> chunk_state -> chunk_state_passing -> chunk_scan), which
 * reorders floating-point sums but not the result.
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers (except ssd_fwd_host), dense and
 *    contiguous in the stated layout (row-major, last index fastest).
 *  - The caller owns every buffer, including the workspace.  The library
 *    allocates no memory and never synchronises the stream except where an
 *    entry point says so.
 *  - Work is enqueued on `stream` (a cudaStream_t passed as void*; NULL is the
 *    legacy default stream) and runs asynchronously.
 *  - Arguments are validated on the host before anything is enqueued.  A bad
 *    argument returns SSD_ERR_INVALID_ARG or SSD_ERR_UNSUPPORTED and enqueues
 *    nothing; ssd_last_error_detail() then names the offending field.
 *  - A CUDA launch error returns SSD_ERR_CUDA.  No kernel traps or asserts.
 *  - Results are bitwise deterministic run to run (no floating atomics).
 */
#ifndef SSD_GB300_SSD_H
#define SSD_GB300_SSD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SSD_ABI_VERSION 4

/* Element types of the public tensors. */
typedef enum { SSD_F32 = 0, SSD_F16 = 1, SSD_BF16 = 2 } ssd_dtype;

/* Operand precision of the contractions (accumulation is always fp32).
 * SSD_OPS_F32: every product in fp32 on the CUDA cores ("exact" path).
 * SSD_OPS_F16 / SSD_OPS_BF16: x, B, C and the derived operands are rounded to
 * fp16 / bf16 (round to nearest even) and multiplied on the tensor cores with
 * fp32 accumulation; the cumulative decay, the exponentials and the
 * inter-chunk recurrence stay fp32.  This is the README's "FP16 operands with
 * FP32 accumulation" ("Benchmark" notes). */
typedef enum { SSD_OPS_F32 = 0, SSD_OPS_F16 = 1, SSD_OPS_BF16 = 2 } ssd_operand_mode;

/* Execution plan.  CHUNKED runs the four chunk steps as separate launches
 * with the chunk states in the workspace; FUSED runs one persistent
 * tensor-core kernel per call that keeps every state on chip (it needs
 * P = N = chunk = 64, an even number of heads per group, fp16/bf16 operands
 * and 16-byte aligned x, B, C and y).  AUTO picks the fastest plan the
 * arguments support. */
typedef enum { SSD_PLAN_AUTO = 0, SSD_PLAN_CHUNKED = 1, SSD_PLAN_FUSED = 2 } ssd_plan;

typedef enum {
    SSD_OK = 0,
    SSD_ERR_INVALID_ARG = 1, /* null required pointer, dim <= 0, H % G != 0, ... */
    SSD_ERR_UNSUPPORTED = 2, /* valid but outside what the kernels implement   */
    SSD_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required      */
    SSD_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed            */
    SSD_ERR_TIMEOUT = 5      /* a bounded device-side wait gave up              */
} ssd_status;

/*
 * Arguments of one SSD forward.  Shapes (B batch, L tokens, H heads, P head
 * dim, N state dim, G groups, chunk = chunk_size):
 *   x              [B,L,H,P]  x_dtype                         required
 *   dt             [B,L,H]    fp32                            required
 *   A              [H]        fp32 (per-head decay rate)      required
 *   Bm, Cm         [B,L,G,N]  bc_dtype                        required
 *   D              [H]        fp32 (skip, per head)           optional (NULL)
 *   z              [B,L,H,P]  z_dtype  (gate: y *= silu(z))   optional (NULL)
 *   dt_bias        [H]        fp32                            optional (NULL)
 *   initial_state  [B,H,P,N]  fp32                            optional (NULL = 0)
 *   y              [B,L,H,P]  y_dtype                         required output
 *   final_state    [B,H,P,N]  fp32                            optional output
 *                  (NULL = return_final_state false)
 * Constraints: all dims > 0, H % G == 0, 16 <= chunk <= 256 with chunk % 16
 * == 0, P and N multiples of 16 no larger than 128.  x, B, C, z and y share
 * one dtype.  L need not be a multiple of chunk: the ragged tail is computed
 * as if padded with dt' = 0 and x = 0 (nothing is read or written past L).
 * dt_min/dt_max: the clamp of d_t, applied only when (dt_min, dt_max) differs
 * from the no-op default (0, +inf).
 */
typedef struct ssd_fwd_args {
    int64_t B, L, H, P, N, G, chunk;
    const void *x;
    const float *dt;
    const float *A;
    const void *Bm;
    const void *Cm;
    const float *D;
    const void *z;
    const float *dt_bias;
    const float *initial_state;
    void *y;
    float *final_state;
    int32_t x_dtype, bc_dtype, z_dtype, y_dtype; /* ssd_dtype */
    int32_t ops;                                  /* ssd_operand_mode */
    int32_t plan;                                 /* ssd_plan */
    int32_t dt_softplus;                          /* nonzero: softplus(dt + bias) */
    float dt_min, dt_max;
    void *workspace;                              /* device, 256-byte aligned */
    size_t workspace_bytes;
    /* Optional gated RMSNorm on the output (ops-transformer MambaV2 article,
     * section 4.6), the step after the SSD in a Mamba-2 block.  When
     * norm_weight (fp32 [H*P]) is non-NULL, z is required and
     *   y[b,t,:] = rmsnorm_g(ssd[b,t,:] * silu(z[b,t,:])) * norm_weight,
     * where ssd is the output above without its own z gate and rmsnorm_g
     * divides each run of (H/G)*P consecutive channels (the heads of one B/C
     * group) by sqrt(mean of squares + norm_eps).  The fused plan does it in
     * its store stage when H/G <= 4; other plans (and wider groups) run the
     * same arithmetic as a second kernel over y.  Not supported by ssd_bwd. */
    const float *norm_weight;
    float norm_eps;
    /* Optional causal depthwise conv1d + SiLU in front of the SSD
     * (ops-transformer MambaV2 article, sections 1.4 and 4.1: the step before
     * chunk_cumsum in a Mamba-2 block).  When conv_width > 0, x, Bm and Cm hold
     * the activations BEFORE the convolution and the SSD runs on
     *   x'[b,t,c] = silu(conv_x_bias[c] + sum_{k<W} conv_x_weight[c,k] x[b,t-(W-1)+k,c])
     * with x = 0 before t = 0, and likewise B' and C' with their own weights;
     * c runs over the H*P (x) or G*N (B, C) channels of a token, W = conv_width
     * (1..4).  Weights fp32 [channels, W] (all three required), biases fp32
     * [channels] or NULL.  The fused plan at N = 64 convolves the tiles it
     * stages, in the kernel; other plans convolve x, B and C into the
     * workspace first (ssd_causal_conv1d_tokens), then run the SSD.  Not
     * supported by ssd_fwd_host, ssd_fwd_varlen or ssd_bwd (SSD_ERR_UNSUPPORTED);
     * x, B and C must be 16-byte aligned. */
    const float *conv_x_weight, *conv_x_bias;
    const float *conv_b_weight, *conv_b_bias;
    const float *conv_c_weight, *conv_c_bias;
    int32_t conv_width;
} ssd_fwd_args;

/* ABI version of the loaded library (SSD_ABI_VERSION). */
int32_t ssd_abi_version(void);

/* Bytes of device workspace ssd_fwd needs for these arguments (pointers are
 * not inspected).  Returns INVALID_ARG / UNSUPPORTED like ssd_fwd. */
ssd_status ssd_fwd_workspace_size(const ssd_fwd_args *args, size_t *bytes);

/* The plan ssd_fwd would run for these arguments (SSD_PLAN_CHUNKED or
 * SSD_PLAN_FUSED), after resolving SSD_PLAN_AUTO. */
ssd_status ssd_fwd_resolve_plan(const ssd_fwd_args *args, int32_t *plan);

/* Names of the kernels ssd_fwd would launch for these arguments, in order,
 * as a NUL-terminated comma-separated list written into `out` (capacity
 * `cap` bytes, truncated if shorter), e.g. "chunk_cumsum,chunk_state_tc,
 * state_passing,chunk_scan_tc" or "ssd_fused_kernel".  Pointers are
 * inspected only for the alignment the tensor-core kernels need. */
ssd_status ssd_fwd_describe(const ssd_fwd_args *args, char *out, size_t cap);

/* The whole forward: y (and final_state when non-NULL).  Enqueue only. */
ssd_status ssd_fwd(const ssd_fwd_args *args, void *stream);

/*
 * The four chunk steps, callable one at a time (ops-transformer MambaV2
 * article, sections 4.2-4.5).  c = ceil(L / chunk).  Intermediate layouts:
 *   dtp, cs  [B,H,c,chunk] fp32   processed step d_t and the inclusive
 *                                 within-chunk cumulative sum of d_t*A[h]
 *                                 (past L: d = 0, cs holds its last value)
 *   states   [B,c,H,P,N]   fp32
 * These entry points need no workspace and ignore args->workspace.
 */

/* Step 1, chunk_cumsum (article section 4.2): writes dtp and cs. */
ssd_status ssd_chunk_cumsum(const ssd_fwd_args *args, float *dtp, float *cs, void *stream);

/* Step 2, chunk_state (article section 4.3): states[b,k,h] =
 *   sum_{i in chunk k} exp(cs[k,last] - cs[k,i]) * dtp[k,i] * x_i (outer) B_i,
 * the state chunk k produces from a zero start. */
ssd_status ssd_chunk_state(const ssd_fwd_args *args, const float *dtp, const float *cs,
                           float *states, void *stream);

/* Step 3, chunk_state_passing (article section 4.4): in place, replaces each
 * chunk's own state by the state ENTERING that chunk:
 *   S_0 = initial_state (or 0),  S_{k+1} = exp(cs[k,last]) * S_k + states[k],
 * and writes S_c to args->final_state when it is non-NULL. */
ssd_status ssd_state_passing(const ssd_fwd_args *args, const float *cs, float *states,
                             void *stream);

/* Step 4, chunk_scan (article section 4.5): writes args->y from the entering
 * states:  y_i = exp(cs_i) C_i . S_k + sum_{j<=i} (C_i . B_j) exp(cs_i - cs_j)
 * dtp_j x_j, then + D x_i and * silu(z_i). */
ssd_status ssd_chunk_scan(const ssd_fwd_args *args, const float *dtp, const float *cs,
                          const float *states, void *stream);

/*
 * End-to-end call with HOST buffers: every tensor pointer in args is host
 * memory (pinned for overlap; pageable works but serialises).  The library
 * copies the inputs into the device workspace, runs ssd_fwd there and copies
 * y and final_state back; the host outputs are valid after the caller
 * synchronises `stream`.  The call is cut into slices: with the fused plan at
 * N = 64 or the chunked plan, along the sequence (up to 16 slices of whole
 * chunks over every batch row, the fp32 state handed from slice to slice, so
 * the outputs equal ssd_fwd's bit for bit); otherwise along the batch (up to 8
 * slices; one when a per-batch stride is not a multiple of 256 bytes).  The
 * copies in run on an internal stream (one 2-D copy per tensor and sequence
 * slice), each slice's forward on `stream` once its inputs are in, its copies
 * out on a second internal stream, so both copy directions and the kernels
 * overlap.  Work enqueued on `stream` before the call is ordered before
 * it, and the call as a whole is complete on `stream`.  The two internal
 * streams and four events are created once per device on first use and kept
 * until exit; concurrent calls from several threads are serialised while they
 * enqueue.  The workspace (device) must hold ssd_fwd_host_workspace_size()
 * bytes; the host buffers must stay valid until the stream completes.
 */
ssd_status ssd_fwd_host_workspace_size(const ssd_fwd_args *args, size_t *bytes);
ssd_status ssd_fwd_host(const ssd_fwd_args *args, void *stream);

/*
 * ssd_fwd without a caller-provided workspace, for callers that cannot
 * allocate device memory (code that runs under an allocator it does not own,
 * plugins barred from cudaMalloc, latency-critical paths that must not
 * allocate).  The pages have no counterpart; this is a convenience of this
 * library.  args->workspace and args->workspace_bytes are ignored: the scratch
 * comes from a 64 MiB buffer built into the library, which every GPU that
 * loads the library holds until the process exits.  A call whose
 * ssd_fwd_workspace_size() exceeds 64 MiB returns SSD_ERR_WORKSPACE and
 * enqueues nothing.  Nothing is allocated: no cudaMalloc, no cudaFree.
 *  - The first call on a device, with that device current, looks up the
 *    buffer's device address (cudaGetSymbolAddress); make that first call
 *    before any stream capture.
 *  - All calls share the one buffer, so calls that may overlap on the GPU
 *    (different streams, other threads) race and must be serialised by the
 *    caller.  Everything that must start at zero is cleared by each call.
 *  - Device-side wait timeouts of these calls are not reachable through
 *    ssd_check_device_error, which needs the workspace.
 */
ssd_status ssd_fwd_noalloc(const ssd_fwd_args *args, void *stream);

/*
 * Decode: one recurrent step for a single new token of each of B sequences,
 * continuing from their carried states (the final_state of a forward, or of
 * the previous step) -- the "final_state for the decode stage" of the
 * ops-transformer MambaV2 article, section 4.4.  For every (b, h), g = h/(H/G):
 *
 *     d      = clamp(softplus(dt[b,h] + dt_bias[h]))   bias / softplus / clamp optional
 *     S[p,:] = exp(d A[h]) S[p,:] + d x[b,h,p] B[b,g,:]     S = state[b,h], updated IN PLACE
 *     y[b,h,p] = (S[p,:] . C[b,g,:] + D[h] x[b,h,p]) * silu(z[b,h,p])
 *
 * i.e. the forward's recurrence for L = 1 with initial_state = final_state =
 * state.  Shapes and types:
 *   x, z, y  [B,H,P]   x_dtype (z optional)
 *   dt       [B,H]     fp32        A, D, dt_bias  [H] fp32 (D, dt_bias optional)
 *   Bm, Cm   [B,G,N]   x_dtype
 *   state    [B,H,P,N] fp32, read and written
 * Every product is fp32 on the CUDA cores.  N <= 128, any P, H % G == 0.
 * No workspace; enqueue only; the same validation rules as ssd_fwd.
 */
typedef struct {
    int64_t B, H, P, N, G;
    const void *x;
    const float *dt;
    const float *A;
    const void *Bm;
    const void *Cm;
    const float *D;
    const void *z;
    const float *dt_bias;
    float *state;
    void *y;
    int32_t x_dtype;     /* ssd_dtype of x, B, C, z and y */
    int32_t dt_softplus; /* nonzero: softplus(dt + bias) */
    float dt_min, dt_max;
} ssd_decode_args;

ssd_status ssd_decode_step(const ssd_decode_args *args, void *stream);

/*
 * Backward of the forward: gradients of L = sum(dy * y) + sum(dfinal *
 * final_state) with respect to x, dt, A, B, C, D, z, dt_bias and the initial
 * state (the SSD backward of the "Mamba-2 SSD for Ascend NPU" README,
 * "Limitations and roadmap").  Chunked like the forward: the chunk states
 * are recomputed by its first three steps, the adjoint state is passed
 * backwards between chunks, and one kernel per (batch, head, chunk) forms the
 * local gradients; all arithmetic is fp32 on the CUDA cores (args.fwd.ops
 * and .plan are ignored).  Needs chunk <= 64, P <= 64, N <= 64.
 *   fwd        the forward's arguments: shapes, dtypes, x, dt, A, Bm, Cm and
 *              the optional D, z, dt_bias, initial_state, dt_softplus,
 *              dt_limit (y, final_state, workspace of fwd are ignored)
 *   dy         [B,L,H,P] x_dtype          dfinal  [B,H,P,N] fp32 or NULL
 *   dx         [B,L,H,P] x_dtype          ddt     [B,L,H] fp32 (raw dt)
 *   dB, dC     [B,L,G,N] x_dtype          dA      [H] fp32
 *   dD         [H] fp32, required with D  dz      [B,L,H,P] x_dtype, required with z
 *   ddt_bias   [H] fp32, required with dt_bias
 *   dh0        [B,H,P,N] fp32 or NULL
 *   workspace  device, 256-byte aligned, ssd_bwd_workspace_size() bytes
 * Every sum runs in a fixed order: bitwise reproducible.  Enqueue only.
 */
typedef struct {
    ssd_fwd_args fwd;
    const void *dy;
    const float *dfinal;
    void *dx;
    float *ddt;
    float *dA;
    void *dB;
    void *dC;
    float *dD;
    void *dz;
    float *ddt_bias;
    float *dh0;
    void *workspace;
    size_t workspace_bytes;
} ssd_bwd_args;

ssd_status ssd_bwd_workspace_size(const ssd_bwd_args *args, size_t *bytes);
ssd_status ssd_bwd(const ssd_bwd_args *args, void *stream);

/*
 * Packed variable-length sequences ("varlen"): nseq sequences of different
 * lengths stored back to back along L of a B = 1 call, sequence s holding
 * tokens [cu_seqlens[s], cu_seqlens[s+1]).  Each sequence is an independent
 * forward: the state starts at initial_state[s] (or 0) at its first token and
 * final_state[s] is the state after its last token; nothing crosses a
 * boundary.  Equivalent to nseq separate ssd_fwd calls with B = 1.
 *   args          as for ssd_fwd with B = 1 and L = cu_seqlens[nseq]; except
 *                 initial_state, final_state  [nseq,H,P,N] fp32
 *   cu_seqlens    HOST array of nseq + 1 int64 offsets, cu_seqlens[0] = 0,
 *                 non-decreasing (empty sequences allowed); read during the
 *                 call only (copied into the workspace when the fused plan runs)
 * The fused plan takes the call when its shape rules hold (the chunked plan
 * otherwise, one sequence after another).  Returns INVALID_ARG for B != 1 or
 * malformed offsets; the workspace must hold ssd_fwd_varlen_workspace_size()
 * bytes.  Enqueue only.
 */
ssd_status ssd_fwd_varlen_workspace_size(const ssd_fwd_args *args, const int64_t *cu_seqlens, int64_t nseq,
                                         size_t *bytes);
ssd_status ssd_fwd_varlen(const ssd_fwd_args *args, const int64_t *cu_seqlens, int64_t nseq, void *stream);

/*
 * Sequence-parallel exchange.  A sequence split into consecutive token
 * segments (one per rank) is composed from each segment's affine state map
 *     S_out = exp(a) * S_in + S_seg
 * per (b, h): a = the segment's total sum of d_t * A[h], S_seg = the segment's
 * final state from a zero start -- the rule chunk_state_passing applies
 * between chunks (ops-transformer MambaV2 article, section 4.4), here between
 * segments.  A rank computes (a, S_seg) for its segment, all ranks exchange
 * them, each folds the maps of the segments before its own into the state
 * entering its segment and reruns its segment from there.
 */

/* a[b,h] = sum over the L tokens of args of d_t * A[h], d_t processed as in
 * ssd_fwd (bias, softplus, clamp), accumulated in fp64 in token order.
 * log_decay: [B,H] fp32, device.  Needs x-free args: only dt, A, dt_bias and
 * the shape are read.  Enqueue only. */
ssd_status ssd_segment_log_decay(const ssd_fwd_args *args, float *log_decay, void *stream);

/* out = fold of nseg consecutive segment maps from a zero start:
 *     S = 0;  for q = 0 .. nseg-1:  S = exp(log_decay[q]) * S + states[q]
 * log_decay [nseg,B,H], states [nseg,B,H,P,N], out [B,H,P,N]; fp32, device.
 * nseg = 0 writes zeros.  Enqueue only. */
ssd_status ssd_state_fold(int64_t nseg, int64_t B, int64_t H, int64_t P, int64_t N, const float *log_decay,
                          const float *states, float *out, void *stream);

/*
 * The SSD's neighbours in the Mamba-2 block (ops-transformer MambaV2 article,
 * sections 1.4, 4.1 and 4.6).  fp32 arithmetic; x, z and out share `dtype`
 * (ssd_dtype); weights and biases are fp32.  Enqueue only.
 *
 * Causal conv1d + SiLU: a depthwise convolution of width W along the
 * sequence, with W-1 zeros before the first step, plus bias, then SiLU:
 *     out[b,d,t] = silu(bias[d] + sum_{k<W} w[d,k] x[b,d,t-(W-1)+k])
 * x, out [B,D,S]; w [D,W]; bias [D] or NULL; 1 <= W <= 8; silu = 0 skips SiLU.
 */
ssd_status ssd_causal_conv1d(int64_t B, int64_t D, int64_t S, int64_t W, int32_t dtype, const void *x,
                             const float *w, const float *bias, int32_t silu, void *out, void *stream);

/* The same convolution over token-major activations, the layout of a
 * Mamba-2 block's x, B and C (and of ssd_fwd_args.conv_*):
 *   out[b,t,c] = silu(bias[c] + sum_{k<W} w[c,k] x[b,t-(W-1)+k,c])  (SiLU if silu)
 * x, out [B, S, C] (dtype, contiguous); w [C, W] fp32 (1 <= W <= 4); bias [C]
 * fp32 or NULL; C % 4 == 0 and 16-byte aligned x and out.  out must not
 * overlap x. */
ssd_status ssd_causal_conv1d_tokens(int64_t B, int64_t S, int64_t C, int64_t W, int32_t dtype, const void *x,
                                    const float *w, const float *bias, int32_t silu, void *out, void *stream);

/* Gated grouped RMSNorm: v = x * silu(z), normalised by the root mean square
 * of v over each of `groups` runs of D/groups consecutive channels (eps inside
 * the root), times w:  out = v / sqrt(mean(v^2) + eps) * w.
 * x, z, out [rows, D]; w [D]; D % groups == 0; eps >= 0. */
ssd_status ssd_gated_rmsnorm(int64_t rows, int64_t D, int64_t groups, float eps, int32_t dtype, const void *x,
                             const void *z, const float *w, void *out, void *stream);

/* Self-test of the bounded device-side waits (no counterpart on the pages;
 * the pages' kernels report errors only as exceptions on the host).  Every
 * mbarrier wait in the tensor-core kernels gives up after a time limit
 * instead of hanging, records the timeout in the workspace error word and
 * lets the kernel finish; ssd_check_device_error then returns
 * SSD_ERR_TIMEOUT.  This call exercises that path on purpose: it clears the
 * first 256 bytes of `workspace` (device, 256-byte aligned, caller-owned,
 * at least 256 bytes) and launches one CTA whose thread waits, through the
 * same bounded wait, on an mbarrier that nothing arrives on, for
 * timeout_us microseconds (1 .. 1e6).  With `arrive` nonzero the thread
 * arrives first, so the wait succeeds and the word stays clear.  Nothing else
 * (no copy, no tensor-core operation) is in flight.  Asynchronous on `stream`;
 * read the outcome with ssd_check_device_error on args whose workspace is
 * this buffer.  Returns SSD_OK, SSD_ERR_INVALID_ARG or SSD_ERR_CUDA. */
ssd_status ssd_selftest_wait_timeout(void *workspace, uint32_t timeout_us, int32_t arrive, void *stream);

/* A measurement kernel, not part of the SSD: `grid` CTAs of 256 threads, each
 * thread running 8 independent fp32 FMA chains of `iters` steps (a multiple
 * of 8 in [8, 2^22]), 2 * 8 * iters * 256 * grid flops in all, and storing
 * one float per thread into `out` (device, caller-owned, at least grid * 256
 * floats; the values carry no meaning).  Timed with CUDA events on `stream`
 * it gives the GPU's fp32 CUDA-core throughput, the peak against which the
 * backward (fp32 on the CUDA cores) is reported.  Asynchronous; returns
 * SSD_OK, SSD_ERR_INVALID_ARG (before anything is enqueued) or SSD_ERR_CUDA. */
ssd_status ssd_selftest_fma_rate(float *out, int64_t out_count, int32_t iters, int32_t grid, void *stream);

/* Synchronises `stream`, then reads the device error word the last ssd_fwd
 * on this workspace left behind (bounded waits that gave up set it).
 * Returns SSD_OK or SSD_ERR_TIMEOUT (or SSD_ERR_CUDA). */
ssd_status ssd_check_device_error(const ssd_fwd_args *args, void *stream);

/* Short static description of a status code. */
const char *ssd_status_string(ssd_status status);

/* Thread-local detail of the last failing call on this thread ("" if none). */
const char *ssd_last_error_detail(void);

#ifdef __cplusplus
}
#endif

#endif /* SSD_GB300_SSD_H */
