/*
 * oracle.c -- plain, slow, sequential float64 reference of the Mamba selective
 * scan and of its single-token recurrent update.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker the CUDA library is
 * measured against.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load it; the library itself never does.  It shares no
 * code, header, table or helper with the CUDA path.
 *
 * What it computes, and where that comes from:
 *
 *  - "Mamba: Selective State Space Models" (eeshsaxena/mamba-ssm-implementation
 *    README), section "Mathematical Foundation / State Space Model": the
 *    continuous model h'(t) = A h(t) + B x(t), y(t) = C h(t) + D x(t).
 *  - same page, "Selective Mechanism": B, C and the timestep Delta depend on the
 *    input; Delta = tau_Delta(Parameter + Linear_Delta(x)).  Here the already
 *    projected Delta_raw is an input, "Parameter" is delta_bias, and tau_Delta
 *    is softplus (applied when softplus_flag is set).
 *  - same page, "Architecture": Delta drives a discretisation step; the page
 *    does not print the formula.  The reading adopted here is zero-order hold
 *    for A and the Euler rule for B:  dA = exp(Delta*A),  dB*u = Delta*B*u.
 *  - same page, "Efficient Scan", item 2 (sequential scan for inference): the
 *    recurrence h_t = dA_t * h_{t-1} + dB_t * u_t run one step at a time with a
 *    constant-size state, starting from h = 0 -- or, for a scan that continues
 *    an earlier one (a prompt processed in pieces, or a scan resumed after
 *    recurrent steps), from the state the earlier part left:
 *    oracle_scan_from takes that state as h_{-1}.
 *  - readout y_t = C_t . h_t + D * u_t (the y equation above, with h_t taken
 *    after the step-t update), then the Mamba block's gate
 *    ("Features": "Mamba block with gated residuals"): y_t *= silu(z_t).
 *
 * Everything is float64; every input arrives already widened exactly from its
 * stored type.  No exp2, no log2(e) prescale, no chunking, no reordering: loop
 * order is batch -> channel -> time -> state, exactly the definition.
 *
 * Layouts (row-major):
 *   u, delta, z, out : [batch][seqlen][dim]
 *   B, C             : [batch][dstate][seqlen], or [batch][ngroups][dstate][seqlen]
 *                      for the grouped entry points (channel d reads group
 *                      d / (dim / ngroups); one group is the plain layout)
 *   A                : [dim][dstate]
 *   D, delta_bias    : [dim]
 *   last_state       : [batch][dim][dstate]
 *   initial_state    : [batch][dim][dstate]  (oracle_scan_from only)
 * Decode step:
 *   state            : [batch][dim][dstate]  (updated in place)
 *   x, dt, z, out    : [batch][dim]
 *   B, C             : [batch][dstate], or [batch][ngroups][dstate] (grouped)
 *
 * Grouped B and C.  The pages give B and C as functions of the input shared by
 * every channel of a sequence.  The grouped entry points widen this the plain
 * way: the channels are cut into ngroups equal consecutive blocks and each
 * block has its own B_t and C_t; with one block this is the pages' model.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_MAX_DSTATE 256

/* softplus(x) = log(1 + e^x), written in the overflow-free form
 * max(x, 0) + log1p(exp(-|x|)). */
static double softplus(double x) {
    return (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x)));
}

/* silu(z) = z * sigmoid(z) = z / (1 + e^-z). */
static double silu(double zv) {
    return zv / (1.0 + exp(-zv));
}

/* Delta for one (time, channel): optional bias add, optional softplus. */
static double timestep(double delta_raw, const double* delta_bias, int d,
                       int softplus_flag) {
    double x = delta_raw + (delta_bias ? delta_bias[d] : 0.0);
    return softplus_flag ? softplus(x) : x;
}

/* One recurrence step for one (batch, channel): updates h[0..N) in place and
 * returns the gated output.  Bv / Cv give B and C of this step, read with a
 * stride so the same step serves the scan layout ([N][L]) and the decode
 * layout ([N]). */
static double one_step(double* h, const double* Arow, int N,
                       const double* Bv, const double* Cv, ptrdiff_t bc_stride,
                       double uv, double dlt, double Dd, const double* zp) {
    double y = 0.0;
    for (int n = 0; n < N; ++n) {
        double dA = exp(dlt * Arow[n]);                 /* zero-order hold */
        double dBu = (dlt * Bv[n * bc_stride]) * uv;    /* Euler:  (Delta B) u */
        h[n] = dA * h[n] + dBu;
        y += Cv[n * bc_stride] * h[n];
    }
    y += Dd * uv;
    if (zp) y *= silu(*zp);
    return y;
}

static int check_dims(int batch, int dim, int seqlen, int dstate) {
    if (batch <= 0 || dim <= 0 || seqlen <= 0 || dstate <= 0) return 1;
    if (dstate > ORACLE_MAX_DSTATE) return 1;
    return 0;
}

static int check_groups(int dim, int ngroups) {
    return (ngroups <= 0 || dim % ngroups != 0) ? 1 : 0;
}

/* Index of the B/C block that channel d of batch row b reads. */
static ptrdiff_t bc_block(ptrdiff_t b, ptrdiff_t d, ptrdiff_t dim, ptrdiff_t ngroups) {
    return b * ngroups + d / (dim / ngroups);
}

/* Full-sequence scan of every (batch, channel), independently, starting from
 * initial_state (h = 0 where it is NULL).  The OpenMP loop only distributes
 * whole independent channels across threads; each channel's arithmetic is the
 * sequential definition above.  last_state may be the same array as
 * initial_state (each channel reads its initial state before it writes). */
int oracle_scan_grouped(const double* u, const double* delta, const double* A,
                        const double* B, const double* C, const double* D,
                        const double* z, const double* delta_bias, int softplus_flag,
                        const double* initial_state, double* out, double* last_state,
                        int batch, int dim, int seqlen, int dstate, int ngroups) {
    if (!u || !delta || !A || !B || !C || !out) return 1;
    if (check_dims(batch, dim, seqlen, dstate) || check_groups(dim, ngroups)) return 2;
    const ptrdiff_t L = seqlen, Dm = dim, N = dstate;
    const long long total = (long long)batch * dim;
#pragma omp parallel for schedule(dynamic, 1)
    for (long long bd = 0; bd < total; ++bd) {
        const ptrdiff_t b = bd / Dm, d = bd % Dm;
        double h[ORACLE_MAX_DSTATE];
        for (ptrdiff_t n = 0; n < N; ++n)
            h[n] = initial_state ? initial_state[(b * Dm + d) * N + n] : 0.0;
        const ptrdiff_t blk = bc_block(b, d, Dm, ngroups);
        const double* Bb = B + blk * N * L;
        const double* Cb = C + blk * N * L;
        const double Dd = D ? D[d] : 0.0;
        for (ptrdiff_t t = 0; t < L; ++t) {
            const ptrdiff_t i = (b * L + t) * Dm + d;
            const double dlt = timestep(delta[i], delta_bias, (int)d, softplus_flag);
            out[i] = one_step(h, A + d * N, (int)N, Bb + t, Cb + t, L,
                              u[i], dlt, Dd, z ? z + i : NULL);
        }
        if (last_state)
            for (ptrdiff_t n = 0; n < N; ++n) last_state[(b * Dm + d) * N + n] = h[n];
    }
    return 0;
}

/* The scan from a given state, with B and C shared by all channels. */
int oracle_scan_from(const double* u, const double* delta, const double* A,
                     const double* B, const double* C, const double* D,
                     const double* z, const double* delta_bias, int softplus_flag,
                     const double* initial_state, double* out, double* last_state,
                     int batch, int dim, int seqlen, int dstate) {
    return oracle_scan_grouped(u, delta, A, B, C, D, z, delta_bias, softplus_flag, initial_state,
                               out, last_state, batch, dim, seqlen, dstate, 1);
}

/* The scan from h = 0. */
int oracle_scan(const double* u, const double* delta, const double* A,
                const double* B, const double* C, const double* D,
                const double* z, const double* delta_bias, int softplus_flag,
                double* out, double* last_state,
                int batch, int dim, int seqlen, int dstate) {
    return oracle_scan_from(u, delta, A, B, C, D, z, delta_bias, softplus_flag, NULL,
                            out, last_state, batch, dim, seqlen, dstate);
}

/* Single-token recurrent update ("Efficient Scan", item 2): the same step as
 * the scan's body, applied once to a caller-held state. */
int oracle_step_grouped(double* state, const double* x, const double* dt,
                        const double* A, const double* B, const double* C,
                        const double* D, const double* z, const double* dt_bias,
                        int dt_softplus, double* out, int batch, int dim, int dstate,
                        int ngroups) {
    if (!state || !x || !dt || !A || !B || !C || !out) return 1;
    if (check_dims(batch, dim, 1, dstate) || check_groups(dim, ngroups)) return 2;
    const ptrdiff_t Dm = dim, N = dstate;
    const long long total = (long long)batch * dim;
#pragma omp parallel for schedule(static)
    for (long long bd = 0; bd < total; ++bd) {
        const ptrdiff_t b = bd / Dm, d = bd % Dm;
        const ptrdiff_t i = b * Dm + d;
        const double dlt = timestep(dt[i], dt_bias, (int)d, dt_softplus);
        const ptrdiff_t blk = bc_block(b, d, Dm, ngroups);
        out[i] = one_step(state + i * N, A + d * N, (int)N, B + blk * N, C + blk * N, 1,
                          x[i], dlt, D ? D[d] : 0.0, z ? z + i : NULL);
    }
    return 0;
}

int oracle_step(double* state, const double* x, const double* dt,
                const double* A, const double* B, const double* C,
                const double* D, const double* z, const double* dt_bias,
                int dt_softplus, double* out, int batch, int dim, int dstate) {
    return oracle_step_grouped(state, x, dt, A, B, C, D, z, dt_bias, dt_softplus, out,
                               batch, dim, dstate, 1);
}

/* Backward of the full-sequence scan (from h = 0): given dout = dL/d out,
 * every input's gradient, by the adjoint of the recurrence above (the
 * gradients the "training" mode of the pages' "Efficient Scan" needs).  With
 *   x_t = delta_raw_t + bias,  Delta_t = softplus(x_t) (or x_t),
 *   a_t[n] = exp(Delta_t A[n]),  h_t = a_t h_{t-1} + Delta_t B_t u_t,
 *   y_t = C_t . h_t + D u_t,  out_t = y_t g_t,  g_t = silu(z_t) (or 1),
 * the adjoint state lambda_t = dL/dh_t runs backwards:
 *   dy_t = dout_t g_t,  lambda_t = C_t dy_t + a_{t+1} lambda_{t+1}  (lambda_L = 0),
 * and
 *   dC_t[n] += dy_t h_t[n]            dB_t[n] += lambda_t[n] Delta_t u_t
 *   du_t     = D dy_t + sum_n lambda_t[n] Delta_t B_t[n]
 *   dDelta_t = sum_n lambda_t[n] (A[n] a_t[n] h_{t-1}[n] + B_t[n] u_t)
 *   dA[n]   += lambda_t[n] Delta_t a_t[n] h_{t-1}[n]
 *   dD      += dy_t u_t,   dz_t = dout_t y_t silu'(z_t)
 *   ddelta_raw_t = dDelta_t softplus'(x_t) (= dDelta_t without softplus),
 *   dbias  += ddelta_raw_t.
 * B and C are shared by all channels (of a group, in the grouped form), so dB
 * and dC sum over those channels.  Every
 * output array is overwritten; dz, dD and dbias may be NULL when z, D or the
 * bias is absent.  Sequential (no threads): each output sums over channels.
 *
 * oracle_scan_bwd_from is the backward of the scan from a given state
 * (oracle_scan_from) whose final state also enters the loss: with h_{-1} =
 * initial_state (0 when NULL) and dlast = dL/d last_state (0 when NULL), the
 * adjoint starts from lambda_{L-1} = C_{L-1} dy_{L-1} + dlast, and
 *   dinitial = dL/dh_{-1} = a_0 lambda_0
 * is written when dinitial is not NULL.  A sequence cut in two pieces is
 * differentiated piece by piece: the second piece's dinitial is the first
 * piece's dlast. */
static double sigmoid(double v) { return 1.0 / (1.0 + exp(-v)); }

int oracle_scan_bwd_from(const double* u, const double* delta, const double* A,
                         const double* B, const double* C, const double* D,
                         const double* z, const double* delta_bias, int softplus_flag,
                         const double* initial_state, const double* dout, const double* dlast,
                         double* du, double* ddelta, double* dA, double* dB, double* dC,
                         double* dD, double* dz, double* dbias, double* dinitial,
                         int batch, int dim, int seqlen, int dstate, int ngroups) {
    if (!u || !delta || !A || !B || !C || !dout || !du || !ddelta || !dA || !dB || !dC) return 1;
    if (check_dims(batch, dim, seqlen, dstate) || check_groups(dim, ngroups)) return 2;
    const ptrdiff_t L = seqlen, Dm = dim, N = dstate;
    for (ptrdiff_t i = 0; i < Dm * N; ++i) dA[i] = 0.0;
    for (ptrdiff_t i = 0; i < (ptrdiff_t)batch * ngroups * N * L; ++i) dB[i] = dC[i] = 0.0;
    if (dD) for (ptrdiff_t d = 0; d < Dm; ++d) dD[d] = 0.0;
    if (dbias) for (ptrdiff_t d = 0; d < Dm; ++d) dbias[d] = 0.0;
    double* hs = (double*)malloc((size_t)(L + 1) * N * sizeof(double));   /* h_{-1} .. h_{L-1} */
    double* dls = (double*)malloc((size_t)L * sizeof(double));
    double* ys = (double*)malloc((size_t)L * sizeof(double));
    if (!hs || !dls || !ys) { free(hs); free(dls); free(ys); return 3; }
    for (ptrdiff_t b = 0; b < batch; ++b)
        for (ptrdiff_t d = 0; d < Dm; ++d) {
            const double* Ar = A + d * N;
            const ptrdiff_t blk = bc_block(b, d, Dm, ngroups);
            const double* Bb = B + blk * N * L;
            const double* Cb = C + blk * N * L;
            const double Dd = D ? D[d] : 0.0;
            const ptrdiff_t sbase = (b * Dm + d) * N;
            /* forward from h_{-1}, keeping every state */
            for (ptrdiff_t n = 0; n < N; ++n) hs[n] = initial_state ? initial_state[sbase + n] : 0.0;
            for (ptrdiff_t t = 0; t < L; ++t) {
                const ptrdiff_t i = (b * L + t) * Dm + d;
                const double dlt = timestep(delta[i], delta_bias, (int)d, softplus_flag);
                dls[t] = dlt;
                double y = 0.0;
                for (ptrdiff_t n = 0; n < N; ++n) {
                    const double h = exp(dlt * Ar[n]) * hs[t * N + n] + (dlt * Bb[n * L + t]) * u[i];
                    hs[(t + 1) * N + n] = h;
                    y += Cb[n * L + t] * h;
                }
                ys[t] = y + Dd * u[i];
            }
            /* backward */
            /* lambda "after" the last step is dlast, carried into step L-1 with weight 1 */
            double lam[ORACLE_MAX_DSTATE], anext[ORACLE_MAX_DSTATE];
            for (ptrdiff_t n = 0; n < N; ++n) {
                lam[n] = dlast ? dlast[sbase + n] : 0.0;
                anext[n] = 1.0;
            }
            for (ptrdiff_t t = L - 1; t >= 0; --t) {
                const ptrdiff_t i = (b * L + t) * Dm + d;
                const double dlt = dls[t];
                const double g = z ? silu(z[i]) : 1.0;
                const double dy = dout[i] * g;
                if (z && dz) {
                    const double sg = sigmoid(z[i]);
                    dz[i] = dout[i] * ys[t] * sg * (1.0 + z[i] * (1.0 - sg));
                }
                double dut = Dd * dy, ddl = 0.0;
                for (ptrdiff_t n = 0; n < N; ++n) {
                    const double a = exp(dlt * Ar[n]);
                    const double hprev = hs[t * N + n], h = hs[(t + 1) * N + n];
                    lam[n] = Cb[n * L + t] * dy + anext[n] * lam[n];
                    dC[(blk * N + n) * L + t] += dy * h;
                    dB[(blk * N + n) * L + t] += lam[n] * dlt * u[i];
                    dut += lam[n] * dlt * Bb[n * L + t];
                    ddl += lam[n] * (Ar[n] * a * hprev + Bb[n * L + t] * u[i]);
                    dA[d * N + n] += lam[n] * dlt * a * hprev;
                    anext[n] = a;
                }
                du[i] = dut;
                if (dD) dD[d] += dy * u[i];
                const double xr = delta[i] + (delta_bias ? delta_bias[d] : 0.0);
                const double dx = softplus_flag ? ddl * sigmoid(xr) : ddl;
                ddelta[i] = dx;
                if (dbias) dbias[d] += dx;
            }
            /* h_0 = a_0 h_{-1} + ...: the adjoint of the initial state */
            if (dinitial)
                for (ptrdiff_t n = 0; n < N; ++n) dinitial[sbase + n] = anext[n] * lam[n];
        }
    free(hs);
    free(dls);
    free(ys);
    return 0;
}

int oracle_scan_bwd_grouped(const double* u, const double* delta, const double* A,
                            const double* B, const double* C, const double* D,
                            const double* z, const double* delta_bias, int softplus_flag,
                            const double* dout, double* du, double* ddelta, double* dA,
                            double* dB, double* dC, double* dD, double* dz, double* dbias,
                            int batch, int dim, int seqlen, int dstate, int ngroups) {
    return oracle_scan_bwd_from(u, delta, A, B, C, D, z, delta_bias, softplus_flag, NULL, dout, NULL,
                                du, ddelta, dA, dB, dC, dD, dz, dbias, NULL, batch, dim, seqlen, dstate,
                                ngroups);
}

int oracle_scan_bwd(const double* u, const double* delta, const double* A,
                    const double* B, const double* C, const double* D,
                    const double* z, const double* delta_bias, int softplus_flag,
                    const double* dout, double* du, double* ddelta, double* dA,
                    double* dB, double* dC, double* dD, double* dz, double* dbias,
                    int batch, int dim, int seqlen, int dstate) {
    return oracle_scan_bwd_grouped(u, delta, A, B, C, D, z, delta_bias, softplus_flag, dout, du,
                                   ddelta, dA, dB, dC, dD, dz, dbias, batch, dim, seqlen, dstate, 1);
}

/* Depthwise causal convolution over time, per channel, width W, then the
 * optional SiLU: the local convolution that produces the scan input u in the
 * Mamba block ("d_conv: local convolution width" in the pages' usage examples).
 * Reading adopted (the pages give only the width): PyTorch Conv1d's
 * cross-correlation with W-1 steps of left padding, truncated to L outputs,
 *     y_t = bias[d] + sum_{k=0}^{W-1} w[d][k] * x_{t-(W-1)+k},
 * where x_s for s < 0 is the carried state state_in[b][d][(W-1)+s] (the W-1
 * inputs before this sequence, oldest first), or 0 without one.  state_out
 * (nullable) receives the W-1 last inputs, oldest first.  x, out:
 * [batch][seqlen][dim]; w: [dim][W]; state: [batch][dim][W-1]. */
static double conv_input(const double* x, const double* state_in, ptrdiff_t b, ptrdiff_t d,
                         ptrdiff_t s, ptrdiff_t L, ptrdiff_t Dm, int W) {
    if (s >= 0) return x[(b * L + s) * Dm + d];
    return state_in ? state_in[(b * Dm + d) * (W - 1) + (W - 1) + s] : 0.0;
}

int oracle_conv1d(const double* x, const double* w, const double* bias, int silu_flag,
                  const double* state_in, double* out, double* state_out,
                  int batch, int dim, int seqlen, int width) {
    if (!x || !w || !out) return 1;
    if (batch <= 0 || dim <= 0 || seqlen <= 0 || width < 1) return 2;
    const ptrdiff_t L = seqlen, Dm = dim;
    const int W = width;
    const long long total = (long long)batch * dim;
#pragma omp parallel for schedule(dynamic, 1)
    for (long long bd = 0; bd < total; ++bd) {
        const ptrdiff_t b = bd / Dm, d = bd % Dm;
        for (ptrdiff_t t = 0; t < L; ++t) {
            double acc = bias ? bias[d] : 0.0;
            for (int k = 0; k < W; ++k)
                acc += w[d * W + k] * conv_input(x, state_in, b, d, t - (W - 1) + k, L, Dm, W);
            out[(b * L + t) * Dm + d] = silu_flag ? silu(acc) : acc;
        }
    }
    if (state_out) {
        /* gather every channel's last inputs first: state_out may be state_in */
        const long long n = total * (W - 1);
        double* tmp = (double*)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
        if (!tmp) return 3;
        for (long long bd = 0; bd < total; ++bd)
            for (int k = 0; k < W - 1; ++k)
                tmp[bd * (W - 1) + k] = conv_input(x, state_in, bd / Dm, bd % Dm, L - (W - 1) + k, L, Dm, W);
        for (long long i = 0; i < n; ++i) state_out[i] = tmp[i];
        free(tmp);
    }
    return 0;
}

/* One decode step of the convolution: the window is the carried state
 * (oldest first) followed by the new input; the state then drops its oldest
 * entry and appends the new input. */
int oracle_conv1d_update(double* state, const double* x, const double* w, const double* bias,
                         int silu_flag, double* out, int batch, int dim, int width) {
    if (!state || !x || !w || !out) return 1;
    if (batch <= 0 || dim <= 0 || width < 1) return 2;
    const int W = width;
    for (long long bd = 0; bd < (long long)batch * dim; ++bd) {
        const ptrdiff_t d = bd % dim;
        double* st = state + bd * (W - 1);
        double acc = bias ? bias[d] : 0.0;
        for (int k = 0; k < W - 1; ++k) acc += w[d * W + k] * st[k];
        acc += w[d * W + W - 1] * x[bd];
        out[bd] = silu_flag ? silu(acc) : acc;
        for (int k = 0; k + 1 < W - 1; ++k) st[k] = st[k + 1];
        if (W > 1) st[W - 2] = x[bd];
    }
    return 0;
}

/* Scalar helpers exposed so the pins can test them against closed forms. */
double oracle_softplus(double x) { return softplus(x); }
double oracle_silu(double x) { return silu(x); }

void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
