/*
 * ssm_scan.h -- C ABI of the B300 (sm_103a) selective-scan library
 * (libssmscan.so).
 *
 * Two operations of the Mamba selective state-space model at the core:
 *
 *   ssm_scan_fwd      the full-sequence selective scan (prefill / training
 *                     forward): "Efficient Scan" of the Mamba README
 *                     ("Mamba: Selective State Space Models",
 *                     eeshsaxena/mamba-ssm-implementation), together with the
 *                     "Selective Mechanism" (input-dependent Delta, B, C) and the
 *                     state-space equations of "Mathematical Foundation";
 *   ssm_state_update  the single-token recurrent update used for
 *                     constant-memory inference ("Efficient Scan", item 2:
 *                     sequential scan, O(1) memory).
 *
 * and around them: the scan from a given state (ssm_scan_fwd_from_state), B
 * and C per channel group (the *_grouped calls), the scan's backward
 * (ssm_scan_bwd, ssm_scan_bwd_from_state), the depthwise causal conv1d that
 * produces the scan input (ssm_conv1d_fwd, ssm_conv1d_update), and the scan
 * without a caller workspace (ssm_scan_fwd_noalloc).
 *
 * Per (batch b, channel d) both compute, with h = 0 before the first step:
 *
 *   Delta_t = softplus(delta_raw[t] + delta_bias[d])     (softplus optional)
 *   h_t[n]  = exp(Delta_t * A[d][n]) * h_{t-1}[n] + Delta_t * B[n][t] * u[t]
 *   y_t     = sum_n C[n][t] * h_t[n] + D[d] * u[t]
 *   out[t]  = y_t * silu(z[t])                           (gate optional)
 *
 * The pages name the discretisation step but print no formula; this library
 * uses zero-order hold for A (exp(Delta A)) and the Euler rule for B
 * (Delta B), and reads the gate of the "Mamba block with gated residuals" as
 * a multiplication of y by silu(z).  Internally the state is float32 and
 * exp is evaluated as exp2 of Delta * (A * log2 e).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Memory: every array pointer is DEVICE memory owned by the caller.  The
 *   library never allocates, frees, copies to the host or synchronises; it
 *   only enqueues kernels on `stream` (a cudaStream_t; NULL = the legacy
 *   default stream) and returns.  The caller must keep the buffers alive
 *   until the work on `stream` has completed.
 * - dtype: SSM_F32 or SSM_BF16 selects the element type of the activation
 *   tensors (u/x, delta/dt, z, B, C, out).  A, D, delta_bias/dt_bias and the
 *   SSM state are always float32.  bf16 outputs are rounded to nearest even.
 * - Errors: every argument is validated on the host before anything is
 *   enqueued; on any error nothing is written and nothing is launched.
 *   A launch failure reported by the CUDA runtime returns SSM_ERR_LAUNCH.
 *   Faults inside a kernel (e.g. a pointer to freed memory) surface as a CUDA
 *   error at the caller's next synchronisation, as for any CUDA kernel.
 * - Aliasing: `out` must not overlap any input array (SSM_ERR_ALIAS);
 *   `last_state` must not overlap any input or `out`.  The decode `state` is
 *   read and written in place by definition and must not overlap anything
 *   else.
 * - Alignment: every pointer must be aligned to its element size; the decode
 *   state and A must be 16-byte aligned (SSM_ERR_ALIGN).
 * - Supported d_state: 4, 8 or 16 (SSM_ERR_UNSUPPORTED otherwise).
 * - Sizes are element counts; each must be > 0 (an empty tensor is
 *   SSM_ERR_SHAPE), dim must stay below 2^31 and batch*seqlen*dim below 2^40.
 */
#ifndef SSM_SCAN_H
#define SSM_SCAN_H

#include <stdint.h>

#if defined(__GNUC__)
#define SSM_API __attribute__((visibility("default")))
#else
#define SSM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum ssm_status {
    SSM_OK = 0,
    SSM_ERR_NULL = 1,         /* a required pointer is NULL                      */
    SSM_ERR_SHAPE = 2,        /* a size is <= 0 or the problem is too large      */
    SSM_ERR_ALIGN = 3,        /* a pointer is not aligned as documented          */
    SSM_ERR_UNSUPPORTED = 4,  /* d_state not in {4, 8, 16}                        */
    SSM_ERR_DTYPE = 5,        /* dtype is not SSM_F32 / SSM_BF16                 */
    SSM_ERR_ALIAS = 6,        /* an output overlaps an input (or another output) */
    SSM_ERR_LAUNCH = 7,       /* the CUDA runtime rejected a kernel launch       */
    SSM_ERR_DEVICE = 8,       /* no usable CUDA device / attribute query failed  */
    SSM_ERR_SCRATCH = 9       /* ssm_scan_fwd_noalloc: the sizes need more scratch
                                 than the library's fixed array holds             */
} ssm_status;

typedef enum ssm_dtype {
    SSM_F32 = 0,
    SSM_BF16 = 1
} ssm_dtype;

/*
 * ssm_scan_fwd -- full-sequence selective scan, from h = 0.
 *
 *   u           [batch][seqlen][dim]     dtype   input x of the SSM
 *   delta       [batch][seqlen][dim]     dtype   Delta_raw (already projected)
 *   A           [dim][dstate]            f32     state matrix (diagonal), < 0
 *   B, C        [batch][dstate][seqlen]  dtype   input-dependent B_t, C_t
 *                                                (shared by all channels)
 *   D           [dim]                    f32     skip weight; NULL = 0
 *   z           [batch][seqlen][dim]     dtype   gate input; NULL = no gate
 *   delta_bias  [dim]                    f32     added to delta; NULL = 0
 *   softplus_flag                                nonzero: Delta = softplus(.)
 *   out         [batch][seqlen][dim]     dtype   written once (never read)
 *   last_state  [batch][dim][dstate]     f32     h after the last step;
 *                                                NULL = not written
 *   workspace   device scratch, 16-byte aligned, workspace_bytes long, owned
 *               by the caller; may be NULL (workspace_bytes 0).  With at least
 *               ssm_scan_workspace_bytes(...) bytes the fast path runs (TMA
 *               staging; each warp scans a group of channels through
 *               segments of the sequence, chained through the workspace); it also
 *               needs 16-byte aligned u/delta/z/out/A/last_state and
 *               dim * sizeof(dtype) a multiple of 16.  Otherwise a generic
 *               kernel with the same results runs.  The workspace is
 *               overwritten; it must not overlap any other argument.
 *
 * Returns SSM_OK once the work is enqueued on `stream`.
 */
SSM_API ssm_status ssm_scan_fwd(const void* u, const void* delta, const float* A,
                        const void* B, const void* C, const float* D,
                        const void* z, const float* delta_bias, int softplus_flag,
                        void* out, float* last_state,
                        int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                        int dtype, void* workspace, int64_t workspace_bytes, void* stream);

/*
 * ssm_scan_fwd_from_state -- the same scan, starting from a given state
 * instead of zero: h_{-1} = initial_state.  A scan that continues an earlier
 * one -- a long prompt processed in pieces, or a sequence resumed after
 * ssm_state_update steps -- passes the state the earlier part left
 * ("Mamba: Selective State Space Models" README, "Efficient Scan": the
 * recurrent mode carries a constant-size state).
 *
 *   initial_state  [batch][dim][dstate]  f32   read once per channel before its
 *                                              first step; NULL = zero (exactly
 *                                              ssm_scan_fwd)
 *
 * Every other argument is as in ssm_scan_fwd.  initial_state may be the same
 * array as last_state (resume in place: each channel's initial state is read
 * before its final state is written); otherwise it must not overlap any
 * output, input or the workspace (SSM_ERR_ALIAS).  It must be aligned to 4
 * bytes, and to 16 bytes for the fast paths.  Scanning a sequence in pieces,
 * each from the previous piece's last_state, gives the whole scan's output
 * and final state up to float32 rounding.
 */
SSM_API ssm_status ssm_scan_fwd_from_state(const void* u, const void* delta, const float* A,
                                           const void* B, const void* C, const float* D,
                                           const void* z, const float* delta_bias, int softplus_flag,
                                           const float* initial_state, void* out, float* last_state,
                                           int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                           int dtype, void* workspace, int64_t workspace_bytes,
                                           void* stream);

/*
 * ssm_scan_workspace_bytes -- bytes of workspace the fast paths of
 * ssm_scan_fwd need for these sizes: the larger of (a) B and C staged in the
 * activation dtype as rows, batch * round_up(seqlen, 64) * 2 * dstate
 * elements, the state handed between sequence segments of each chain
 * (chains * cw * dstate * 4 bytes, cw = 128 / dstate channels per chain,
 * chains = batch * ceil(dim / cw)) and one int flag per chain (segmented
 * kernel); and, for bf16 with dstate 16, (b) the tensor-memory kernels'
 * staged operand (batch * round_up(seqlen, 64) * 32 * 4 bytes), their
 * segment state (groups * 32 * 16 * 4 bytes, groups = batch * ceil(dim / 32))
 * and groups * 8 int flags; each part rounded up to 256 bytes.  Returns -1
 * for sizes or a dtype that ssm_scan_fwd would reject.  Pure host computation.
 */
SSM_API int64_t ssm_scan_workspace_bytes(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                         int dtype);

/*
 * ssm_scan_fwd_grouped -- the scan with B and C per channel group.  The
 * pages' B_t and C_t are functions of the input shared by every channel of a
 * sequence ("Selective Mechanism"); here the dim channels are cut into
 * ngroups equal consecutive blocks of gch = dim / ngroups channels, and each
 * block has its own B_t and C_t:
 *
 *   B, C   [batch][ngroups][dstate][seqlen]  dtype   channel d reads block
 *                                                    [b][d / gch]
 *
 * ngroups = 1 is exactly ssm_scan_fwd_from_state.  ngroups must divide dim
 * (SSM_ERR_SHAPE otherwise, and for ngroups <= 0).  Every other argument is
 * as in ssm_scan_fwd_from_state.  Path choice: the tensor-memory kernels take
 * bf16 / dstate 16 when gch is a multiple of 32 and batch * ngroups <= 65535;
 * the segmented kernel when gch is a multiple of 128 / dstate; any other
 * group size runs on the generic kernel (no workspace needed there).  The
 * workspace is sized by ssm_scan_workspace_bytes_grouped.
 */
SSM_API ssm_status ssm_scan_fwd_grouped(const void* u, const void* delta, const float* A, const void* B,
                                        const void* C, const float* D, const void* z, const float* delta_bias,
                                        int softplus_flag, const float* initial_state, void* out,
                                        float* last_state, int64_t batch, int64_t dim, int64_t seqlen,
                                        int64_t dstate, int64_t ngroups, int dtype, void* workspace,
                                        int64_t workspace_bytes, void* stream);

/*
 * ssm_scan_workspace_bytes_grouped -- ssm_scan_workspace_bytes for B and C
 * with ngroups groups: the staged B/C parts (a), (b) and the staged operand
 * of (c) grow by the factor ngroups, the rest is unchanged.  -1 also when
 * ngroups does not divide dim.
 */
SSM_API int64_t ssm_scan_workspace_bytes_grouped(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                                 int64_t ngroups, int dtype);

/*
 * ssm_device_error -- the library's device error word: 0 if no kernel has
 * reported a problem, otherwise a bit set (1: a staged-data wait timed out,
 * 2: a state hand-off between warps of a CTA timed out, 4: a state hand-off
 * between sequence segments timed out; the affected outputs are then
 * incomplete).  Waits in the kernels are bounded (about one second), so a
 * kernel never spins forever.  nonzero `clear` resets the word.  Reads device
 * memory, so it synchronises with the device; -1 if the read fails.
 */
SSM_API int ssm_device_error(int clear);

/*
 * ssm_state_update -- one token of recurrent (constant-memory) inference.
 *
 *   state   [batch][dim][dstate]  f32    h_{t-1} on entry, h_t on return
 *                                        (in place; 16-byte aligned)
 *   x       [batch][dim]          dtype  this token's u
 *   dt      [batch][dim]          dtype  this token's Delta_raw
 *   A       [dim][dstate]         f32    (16-byte aligned)
 *   B, C    [batch][dstate]       dtype  this token's B_t, C_t
 *   D       [dim]                 f32    NULL = 0
 *   z       [batch][dim]          dtype  NULL = no gate
 *   dt_bias [dim]                 f32    NULL = 0
 *   out     [batch][dim]          dtype  gated output y_t
 *   dt_softplus                          nonzero: Delta = softplus(dt + dt_bias)
 *
 * Applied L times from a zero state to the tokens of a sequence, it computes
 * the same recurrence as ssm_scan_fwd over that sequence.
 */
SSM_API ssm_status ssm_state_update(float* state, const void* x, const void* dt,
                            const float* A, const void* B, const void* C,
                            const float* D, const void* z, const float* dt_bias,
                            void* out, int64_t batch, int64_t dim, int64_t dstate,
                            int dt_softplus, int dtype, void* stream);

/*
 * ssm_state_update_grouped -- ssm_state_update with B and C per channel
 * group (as ssm_scan_fwd_grouped):
 *
 *   B, C    [batch][ngroups][dstate]  dtype   channel d reads [b][d / (dim / ngroups)]
 *
 * ngroups = 1 is exactly ssm_state_update; ngroups must divide dim
 * (SSM_ERR_SHAPE otherwise).
 */
SSM_API ssm_status ssm_state_update_grouped(float* state, const void* x, const void* dt, const float* A,
                                            const void* B, const void* C, const float* D, const void* z,
                                            const float* dt_bias, void* out, int64_t batch, int64_t dim,
                                            int64_t dstate, int64_t ngroups, int dt_softplus, int dtype,
                                            void* stream);

/*
 * ssm_scan_bwd -- backward of ssm_scan_fwd (from h = 0): the gradients of a
 * loss L with respect to every input, given dout = dL/d out, by the adjoint
 * recurrence lambda_t = C_t dy_t + exp(Delta_{t+1} A) lambda_{t+1},
 * dy_t = dout_t silu(z_t) (the training mode of the pages' "Efficient Scan").
 *
 *   inputs       as ssm_scan_fwd: u, delta, A, B, C, D, z, delta_bias, softplus_flag
 *   dout         [batch][seqlen][dim]     dtype
 *   du, ddelta   [batch][seqlen][dim]     dtype   (ddelta = dL/d delta_raw)
 *   dz           [batch][seqlen][dim]     dtype   NULL = not computed (ignored without z)
 *   dA           [dim][dstate]            f32
 *   dB, dC       [batch][dstate][seqlen]  f32     (summed over channels)
 *   dD           [dim]                    f32     NULL = not computed (ignored without D)
 *   ddelta_bias  [dim]                    f32     NULL = not computed (ignored without a bias)
 *   workspace    at least ssm_scan_bwd_workspace_bytes(...) bytes, 16-byte
 *                aligned, owned by the caller: the states entering every
 *                8-step chunk and the per-segment aggregates that carry the
 *                state forward and the adjoint backward across segments
 *
 * All gradients are overwritten (the float32 ones are zeroed on `stream` and
 * accumulated with atomics, so their summation order, and the last bits, may
 * vary from run to run).  Outputs must not overlap each other or any input
 * (SSM_ERR_ALIAS); a missing or short workspace is SSM_ERR_NULL /
 * SSM_ERR_SHAPE.
 */
SSM_API ssm_status ssm_scan_bwd(const void* u, const void* delta, const float* A, const void* B, const void* C,
                                const float* D, const void* z, const float* delta_bias, int softplus_flag,
                                const void* dout, void* du, void* ddelta, float* dA, float* dB, float* dC,
                                float* dD, void* dz, float* ddelta_bias, int64_t batch, int64_t dim,
                                int64_t seqlen, int64_t dstate, int dtype, void* workspace,
                                int64_t workspace_bytes, void* stream);

/*
 * ssm_scan_bwd_grouped -- ssm_scan_bwd with B and C per channel group (as
 * ssm_scan_fwd_grouped): B, C, dB and dC are [batch][ngroups][dstate][seqlen],
 * and dB, dC of a group sum over that group's channels only.  ngroups = 1 is
 * exactly ssm_scan_bwd; ngroups must divide dim (SSM_ERR_SHAPE otherwise).
 * The workspace is the same as ssm_scan_bwd's.
 */
SSM_API ssm_status ssm_scan_bwd_grouped(const void* u, const void* delta, const float* A, const void* B,
                                        const void* C, const float* D, const void* z, const float* delta_bias,
                                        int softplus_flag, const void* dout, void* du, void* ddelta, float* dA,
                                        float* dB, float* dC, float* dD, void* dz, float* ddelta_bias,
                                        int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                        int64_t ngroups, int dtype, void* workspace, int64_t workspace_bytes,
                                        void* stream);

/*
 * ssm_scan_bwd_from_state -- the backward of ssm_scan_fwd_from_state (and of
 * its grouped form) when the final state also enters the loss: the forward
 * starts from h_{-1} = initial_state, the adjoint starts from
 * lambda_{L-1} = C_{L-1} dy_{L-1} + dlast, and
 *
 *   initial_state   [batch][dim][dstate]  f32  NULL = zero
 *   dlast           [batch][dim][dstate]  f32  dL/d last_state; NULL = zero
 *   dinitial_state  [batch][dim][dstate]  f32  dL/d initial_state = exp(Delta_0 A) lambda_0;
 *                                              NULL = not computed
 *
 * all three 16-byte aligned (SSM_ERR_ALIGN).  A sequence processed in pieces
 * is differentiated piece by piece, last piece first: each piece's
 * dinitial_state is the dlast of the piece before it.  Every other argument
 * is as in ssm_scan_bwd_grouped (ngroups = 1 for shared B and C); the two
 * inputs may not overlap an output, and dinitial_state may not overlap an
 * input or another output (SSM_ERR_ALIAS).
 */
SSM_API ssm_status ssm_scan_bwd_from_state(const void* u, const void* delta, const float* A, const void* B,
                                           const void* C, const float* D, const void* z, const float* delta_bias,
                                           int softplus_flag, const float* initial_state, const void* dout,
                                           const float* dlast, void* du, void* ddelta, float* dA, float* dB,
                                           float* dC, float* dD, void* dz, float* ddelta_bias,
                                           float* dinitial_state, int64_t batch, int64_t dim, int64_t seqlen,
                                           int64_t dstate, int64_t ngroups, int dtype, void* workspace,
                                           int64_t workspace_bytes, void* stream);

/*
 * ssm_scan_bwd_workspace_bytes -- workspace ssm_scan_bwd needs.  The
 * sequence is cut into nch = ceil(seqlen / 8) chunks and those into
 * S = min(64, max(1, ceil(nch / 32))) segments; with r(x) = x rounded up to a
 * multiple of 256, the size is
 *     r(batch * nch * dim * dstate * 4)   the local state entering every chunk
 *   + r(batch * nch * dim * 4)            the sum of Delta before every chunk
 *   + 3 * r(batch * S * dim * dstate * 4) per segment: decay product, state, adjoint
 * bytes, at least 16; -1 for sizes or a dtype it would reject.
 */
SSM_API int64_t ssm_scan_bwd_workspace_bytes(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                             int dtype);

/*
 * ssm_conv1d_fwd -- depthwise causal convolution over time (+ SiLU): the step
 * that produces the scan input u in the Mamba block (width d_conv, the
 * "local convolution width" of the pages' usage examples).  Per channel d,
 *     y_t   = bias[d] + sum_{k=0}^{width-1} weight[d][k] * x_{t-(width-1)+k}
 *     out_t = silu(y_t) if silu_flag else y_t
 * where x_s for s < 0 is conv_state_in[b][d][(width-1)+s] (the width-1
 * inputs before the sequence, oldest first) or 0 when conv_state_in is NULL.
 *
 *   x, out          [batch][seqlen][dim]     dtype
 *   weight          [dim][width]             f32
 *   bias            [dim]                    f32   NULL = 0
 *   conv_state_in   [batch][dim][width-1]    f32   NULL = zeros
 *   conv_state_out  [batch][dim][width-1]    f32   NULL = not written; the
 *                   width-1 last inputs, oldest first (a later call's
 *                   conv_state_in, or ssm_conv1d_update's state)
 *
 * width 1..4 (SSM_ERR_UNSUPPORTED above).  conv_state_out may be
 * conv_state_in itself (in place); out and conv_state_out must not overlap any
 * other argument (SSM_ERR_ALIAS).  Pointers aligned to their element size;
 * rows of dim * sizeof(dtype) a multiple of 16 with 16-byte aligned x and out
 * take 16-byte vectors.  Enqueued on `stream`.
 */
SSM_API ssm_status ssm_conv1d_fwd(const void* x, const float* weight, const float* bias, int silu_flag,
                                  const float* conv_state_in, void* out, float* conv_state_out,
                                  int64_t batch, int64_t dim, int64_t seqlen, int64_t width, int dtype,
                                  void* stream);

/*
 * ssm_conv1d_update -- one decode step of the same convolution: the window is
 * conv_state (oldest first) followed by x; out = silu?(bias + weight . window);
 * conv_state then drops its oldest input and appends x (in place).
 *
 *   conv_state  [batch][dim][width-1]  f32    read and written (NULL only for width 1)
 *   x, out      [batch][dim]           dtype
 *   weight, bias as in ssm_conv1d_fwd
 */
SSM_API ssm_status ssm_conv1d_update(float* conv_state, const void* x, const float* weight, const float* bias,
                                     int silu_flag, void* out, int64_t batch, int64_t dim, int64_t width,
                                     int dtype, void* stream);

/* Static, human-readable name of a status code (never NULL). */
SSM_API const char* ssm_status_string(int status);

/*
 * ssm_scan_fwd_noalloc -- ssm_scan_fwd for callers that cannot allocate.
 *
 * The pages have no counterpart: this is a deployment variant of the scan.
 * Some callers cannot call cudaMalloc where they run the scan -- code inside
 * a framework whose allocator owns all device memory, allocation-free hot
 * loops, or plain C callers with no allocator to hand a workspace from.  This
 * entry point takes the same arguments as ssm_scan_fwd minus the workspace
 * and uses instead a scratch array that lives in the library: a file-scope
 * device array of ssm_scan_noalloc_max_workspace_bytes() bytes (32 MiB) that
 * every GPU loading the library holds until the process exits.  It performs
 * no allocation of any kind; the caller still passes every input and output.
 *
 * - Invalid arguments get the same codes as ssm_scan_fwd, checked first;
 *   valid sizes whose workspace (ssm_scan_workspace_bytes) exceeds the array
 *   are then rejected with SSM_ERR_SCRATCH.  Either way nothing is enqueued
 *   and the device is not touched.
 * - The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current) and caches it; make that
 *   first call before any stream capture.
 * - All calls on a device share the one array, and each call overwrites it
 *   (the parts that must start at zero are cleared by the call itself).
 *   Calls that overlap on the GPU -- on different streams, or from different
 *   host threads without ordering -- race on it: serialise them.
 */
SSM_API ssm_status ssm_scan_fwd_noalloc(const void* u, const void* delta, const float* A,
                                const void* B, const void* C, const float* D,
                                const void* z, const float* delta_bias, int softplus_flag,
                                void* out, float* last_state,
                                int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                int dtype, void* stream);

/* Size in bytes of ssm_scan_fwd_noalloc's fixed scratch array. */
SSM_API int64_t ssm_scan_noalloc_max_workspace_bytes(void);

/* The CUDA runtime's message for the calling thread's most recent
 * SSM_ERR_LAUNCH (a static string; "no launch error" if there was none). */
SSM_API const char* ssm_last_launch_error(void);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
SSM_API int ssm_version(void);

/* Scan kernels that ssm_force_scan_path can select. */
typedef enum ssm_scan_path {
    SSM_PATH_AUTO = 0,     /* the library's own choice (the default)                  */
    SSM_PATH_TMEM2 = 1,    /* tensor-memory kernel, two states per lane (bf16, N 16)  */
    SSM_PATH_WS = 2,       /* warp-specialised tensor-memory kernel, four states per
                              lane (bf16, N 16)                                        */
    SSM_PATH_SEG = 3,      /* segmented TMA kernel                                     */
    SSM_PATH_GENERIC = 4   /* generic kernel (no workspace, any alignment)            */
} ssm_scan_path;

/*
 * ssm_force_scan_path -- diagnostics for tests and benchmarks that compare
 * the scan kernels (no counterpart on the pages): every ssm_scan_fwd* call
 * that follows, in this process and on every device, runs the given kernel
 * instead of the library's own choice.  generic_layout selects one compiled
 * layout of the generic kernel (-1 = its planner's choice; ignored for the
 * other paths).  A forced kernel that cannot take a call's shape, alignment
 * or workspace makes that call return SSM_ERR_UNSUPPORTED before anything is
 * enqueued.  The setting is an atomic process-wide value read once per call;
 * SSM_PATH_AUTO restores the default.  Returns SSM_ERR_SHAPE for an unknown
 * path.  Production callers never need it.
 */
SSM_API ssm_status ssm_force_scan_path(int path, int generic_layout);

/*
 * ssm_debug_wait_test -- test hook for the kernels' bounded waits (no
 * counterpart on the pages).  Every wait in the library's kernels gives up
 * after a limit (1 s), sets a bit in the device error word, lets its CTA
 * drain its copies and free its tensor memory, and returns; this hook makes
 * that path run on purpose, without any fault:
 *   withhold_flag != 0: in the scans that follow, the first sequence segment
 *     of channel group 0 keeps its state hand-off flag unset, so the segment
 *     after it (when the call is cut into segments: more 32-channel groups
 *     than SMs, or 128/N-channel groups than warps for the segmented kernel)
 *     waits until the limit and gives up (bit 4), and the warps that wait on
 *     it give up in turn; in the decode steps that take the bulk-copy
 *     pipeline, block 0 never issues its first row's copies, so its consumers
 *     wait that stage out and give up (bit 1).  Those calls' outputs (and the
 *     decode step's state rows of block 0) are undefined.
 *   wait_limit_ns: the limit of every wait from now on (<= 0: the default).
 * ssm_debug_wait_test(0, 0) restores the defaults.  Writes a few words of
 * device memory on the current device (synchronous copies); call it only
 * while no scan or decode step runs.  Returns SSM_ERR_DEVICE if the copy fails.  Production
 * callers never need it.
 */
SSM_API ssm_status ssm_debug_wait_test(int withhold_flag, int64_t wait_limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* SSM_SCAN_H */
