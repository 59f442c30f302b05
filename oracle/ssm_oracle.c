/*
 * ssm_oracle.c -- float64 CPU oracle for the selective state-space scan and
 * its single-token decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * definition that the CUDA library is checked against.  Only the test suite,
 * the package smoke check and the benchmark's CPU-baseline leg may load it.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (sources are the pages on Mamba / selective SSMs):
 *   - "Mamba と状態空間モデル(SSM)" (ta-paperlens), section "Mamba: 状態を
 *     「選択的」にする", pseudocode: dt = softplus(x W_d + bias), A stays a
 *     learned parameter, the state update and y_t = C_t h.
 *   - "State Space Models (SSM)" (ultralytics glossary), section "SSMの仕組み",
 *     code listing: zero-order hold  A_bar = exp(delta*A),
 *     B_bar = (A_bar - 1)/A * B,  h = A_bar*h + B_bar*x_t,  y_t = C h,
 *     starting from h = 0.
 *   - news.han.ihouse.idv.tw article 1304, output equation y = C h + D x
 *     (the skip term D).
 *   - agenticai-flow Mamba guide, block diagram: the S6 output is multiplied
 *     element-wise by SiLU(z).
 *
 * Per batch b, channel d, step t, state n (sequential in t, h starts at 0):
 *   dt      = softplus(delta[b,t,d] + dt_bias[d])
 *   Abar    = exp(dt * A[d,n])
 *   Bbar    = (exp(dt*A[d,n]) - 1) / A[d,n] * B[b,t,n]     (expm1 form; the
 *             limit dt*B[b,t,n] when A[d,n] == 0)
 *   h[n]    = Abar * h[n] + Bbar * u[b,t,d]
 *   y[b,t,d]= (sum_n C[b,t,n] * h[n] + Dskip[d] * u[b,t,d]) * silu(z[b,t,d])
 *   h_last[b,d,n] = h[n] after the last step.
 *
 * Layouts (row-major): u, delta, z, y: [B, L, D];  B, C: [B, L, N];
 * A: [D, N];  dt_bias, Dskip: [D];  h_last / state: [B, D, N].
 * dtype 0: u, delta, z, B, C are float32; dtype 1: they are bfloat16, decoded
 * exactly (bf16 is the top half of a float32).  dt_bias, A, Dskip are float32.
 * Optional inputs: dt_bias == NULL means 0, Dskip == NULL means 0,
 * z == NULL means no gate.  h_last == NULL means it is not written.
 *
 * Every function here is pinned by tests/test_oracle_pins.py against values
 * fixed by the pages and by mathematics (the convolution form, brute-force
 * unrolling, a continuous-time ODE solve, closed forms, library routines).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Read element i of an input tensor of the given dtype, as a double. */
static double load_elem(const void *p, int64_t i, int dtype)
{
    if (dtype == 0)
        return (double)((const float *)p)[i];
    /* bfloat16: the 16 stored bits are the high half of a float32. */
    uint16_t bits16 = ((const uint16_t *)p)[i];
    uint32_t bits32 = (uint32_t)bits16 << 16;
    float f;
    memcpy(&f, &bits32, sizeof f);
    return (double)f;
}

/* softplus(x) = log(1 + exp(x)), written in the overflow-free form. */
static double softplus(double x)
{
    return fmax(x, 0.0) + log1p(exp(-fabs(x)));
}

/* SiLU(z) = z * sigmoid(z) = z / (1 + exp(-z)). */
static double silu(double z)
{
    return z / (1.0 + exp(-z));
}

/*
 * Zero-order-hold pair for one (dt, a):  *abar = exp(dt a) and
 * *bcoef = Bbar / B = (exp(dt a) - 1) / a, whose limit at a == 0 is dt.
 */
static void zoh(double dt, double a, double *abar, double *bcoef)
{
    *abar = exp(dt * a);
    *bcoef = (a == 0.0) ? dt : expm1(dt * a) / a;
}

/*
 * One selective-scan channel (b, d): runs the recurrence over all L steps.
 * Writes y for that channel into y[(b*L + t)*D + d] and, if h_last is not
 * NULL, the final state into h_last[(b*D + d)*N + n].  h is N doubles of
 * scratch.
 */
static void scan_channel(const void *u, const void *delta, const float *dt_bias,
                         const float *A, const void *B, const void *C,
                         const float *Dskip, const void *z, double *y,
                         double *h_last, int64_t b, int64_t d, int64_t L,
                         int64_t D, int64_t N, int dtype, double *h)
{
    for (int64_t n = 0; n < N; n++)
        h[n] = 0.0;
    double bias = dt_bias ? (double)dt_bias[d] : 0.0;
    double dsk = Dskip ? (double)Dskip[d] : 0.0;
    for (int64_t t = 0; t < L; t++) {
        int64_t i_btd = (b * L + t) * D + d;
        double ut = load_elem(u, i_btd, dtype);
        double dt = softplus(load_elem(delta, i_btd, dtype) + bias);
        double acc = 0.0;
        for (int64_t n = 0; n < N; n++) {
            double abar, bcoef;
            zoh(dt, (double)A[d * N + n], &abar, &bcoef);
            double bt = load_elem(B, (b * L + t) * N + n, dtype);
            double ct = load_elem(C, (b * L + t) * N + n, dtype);
            h[n] = abar * h[n] + bcoef * bt * ut;
            acc += ct * h[n];
        }
        acc += dsk * ut;
        if (z)
            acc *= silu(load_elem(z, i_btd, dtype));
        y[i_btd] = acc;
    }
    if (h_last)
        for (int64_t n = 0; n < N; n++)
            h_last[(b * D + d) * N + n] = h[n];
}

/*
 * Selective scan over channels d in [d_begin, d_end) of every batch entry.
 * Returns 0, or -1 for a bad argument, -2 when scratch cannot be allocated.
 * Callers may split the channel range across threads; channels are
 * independent and each is computed exactly as above.
 */
int oracle_scan_fwd(const void *u, const void *delta, const float *dt_bias,
                    const float *A, const void *B, const void *C,
                    const float *Dskip, const void *z, double *y,
                    double *h_last, int64_t batch, int64_t L, int64_t D,
                    int64_t N, int dtype, int64_t d_begin, int64_t d_end)
{
    if (!u || !delta || !A || !B || !C || !y)
        return -1;
    if (batch < 0 || L < 0 || D < 0 || N < 1 || (dtype != 0 && dtype != 1))
        return -1;
    if (d_begin < 0 || d_end > D || d_begin > d_end)
        return -1;
    double *h = (double *)malloc(sizeof(double) * (size_t)N);
    if (!h)
        return -2;
    for (int64_t b = 0; b < batch; b++)
        for (int64_t d = d_begin; d < d_end; d++)
            scan_channel(u, delta, dt_bias, A, B, C, Dskip, z, y, h_last, b, d,
                         L, D, N, dtype, h);
    free(h);
    return 0;
}

/*
 * Single-token decode step: the same per-token update as one step of the
 * scan, applied to a stored state.  state: [B, D, N] float64, updated in
 * place; u, delta, z, y: [B, D]; B, C: [B, N].
 */
int oracle_step(double *state, const void *u, const void *delta,
                const float *dt_bias, const float *A, const void *B,
                const void *C, const float *Dskip, const void *z, double *y,
                int64_t batch, int64_t D, int64_t N, int dtype)
{
    if (!state || !u || !delta || !A || !B || !C || !y)
        return -1;
    if (batch < 0 || D < 0 || N < 1 || (dtype != 0 && dtype != 1))
        return -1;
    for (int64_t b = 0; b < batch; b++) {
        for (int64_t d = 0; d < D; d++) {
            int64_t i_bd = b * D + d;
            double ut = load_elem(u, i_bd, dtype);
            double bias = dt_bias ? (double)dt_bias[d] : 0.0;
            double dt = softplus(load_elem(delta, i_bd, dtype) + bias);
            double acc = 0.0;
            for (int64_t n = 0; n < N; n++) {
                double abar, bcoef;
                zoh(dt, (double)A[d * N + n], &abar, &bcoef);
                double bt = load_elem(B, b * N + n, dtype);
                double ct = load_elem(C, b * N + n, dtype);
                double *hp = &state[i_bd * N + n];
                *hp = abar * *hp + bcoef * bt * ut;
                acc += ct * *hp;
            }
            acc += (Dskip ? (double)Dskip[d] : 0.0) * ut;
            if (z)
                acc *= silu(load_elem(z, i_bd, dtype));
            y[i_bd] = acc;
        }
    }
    return 0;
}

/*
 * Discretisation variants of the input term (the decay Abar = exp(dt A) is
 * the same in all three):
 *   disc 0, zero-order hold (ultralytics "SSMの仕組み"):
 *       h_t = Abar h_{t-1} + (Abar - 1)/A B_t u_t
 *   disc 1, Euler (ta-paperlens, the selective-state pseudocode of
 *       "Mamba: 状態を「選択的」にする"; the method news.han.ihouse.idv.tw article
 *       1304 attributes to Mamba-2, error O(dt^2) per step):
 *       h_t = Abar h_{t-1} + dt B_t u_t
 *   disc 2, trapezoidal (news.han.ihouse.idv.tw article 1304, "より正確な
 *       離散化：台形法則": both ends of the step, error O(dt^3) per step; the
 *       page's data-dependent convex weight is not specified, read here as
 *       the plain trapezoid, weight 1/2):
 *       h_t = Abar h_{t-1} + dt/2 (B_t u_t + Abar B_{t-1} u_{t-1}),
 *       with B_{-1} u_{-1} = 0.
 * The readout, skip and gate are those of oracle_scan_fwd.  q is N doubles of
 * scratch holding B_{t-1} u_{t-1}.
 */
static void scan_channel_disc(const void *u, const void *delta, const float *dt_bias,
                              const float *A, const void *B, const void *C,
                              const float *Dskip, const void *z, double *y,
                              double *h_last, int64_t b, int64_t d, int64_t L,
                              int64_t D, int64_t N, int dtype, int disc, double *h,
                              double *q)
{
    for (int64_t n = 0; n < N; n++) {
        h[n] = 0.0;
        q[n] = 0.0;
    }
    const double bias_d = dt_bias ? (double)dt_bias[d] : 0.0;
    const double skip_d = Dskip ? (double)Dskip[d] : 0.0;
    for (int64_t t = 0; t < L; t++) {
        int64_t i_btd = (b * L + t) * D + d;
        double ut = load_elem(u, i_btd, dtype);
        double dt = softplus(load_elem(delta, i_btd, dtype) + bias_d);
        double acc = 0.0;
        for (int64_t n = 0; n < N; n++) {
            double a = (double)A[d * N + n];
            double abar = exp(dt * a);
            double qt = load_elem(B, (b * L + t) * N + n, dtype) * ut;
            double ct = load_elem(C, (b * L + t) * N + n, dtype);
            if (disc == 0)
                h[n] = abar * h[n] + (a != 0.0 ? expm1(dt * a) / a : dt) * qt;
            else if (disc == 1)
                h[n] = abar * h[n] + dt * qt;
            else
                h[n] = abar * h[n] + 0.5 * dt * (qt + abar * q[n]);
            q[n] = qt;
            acc += ct * h[n];
        }
        double out = acc + skip_d * ut;
        if (z)
            out *= silu(load_elem(z, i_btd, dtype));
        y[i_btd] = out;
    }
    if (h_last) {
        double *hl = h_last + (b * D + d) * N;
        for (int64_t n = 0; n < N; n++)
            hl[n] = h[n];
    }
}

/* oracle_scan_fwd with a discretisation variant (disc 0, 1 or 2, above). */
int oracle_scan_fwd_disc(const void *u, const void *delta, const float *dt_bias,
                         const float *A, const void *B, const void *C,
                         const float *Dskip, const void *z, double *y,
                         double *h_last, int64_t batch, int64_t L, int64_t D,
                         int64_t N, int dtype, int disc, int64_t d_begin, int64_t d_end)
{
    if (!u || !delta || !A || !B || !C || !y)
        return -1;
    if (batch < 0 || L < 0 || D < 0 || N < 1 || (dtype != 0 && dtype != 1))
        return -1;
    if (disc < 0 || disc > 2 || d_begin < 0 || d_end > D || d_begin > d_end)
        return -1;
    double *h = (double *)malloc(sizeof(double) * (size_t)N * 2);
    if (!h)
        return -2;
    for (int64_t b = 0; b < batch; b++)
        for (int64_t d = d_begin; d < d_end; d++)
            scan_channel_disc(u, delta, dt_bias, A, B, C, Dskip, z, y, h_last, b, d,
                              L, D, N, dtype, disc, h, h + N);
    free(h);
    return 0;
}

/*
 * The short causal convolution before the SSM (ta-paperlens, "現場ではこう
 * 使う": d_conv, a short 1-D convolution in front of the SSM; agenticai-flow,
 * d_conv=4 with the causal-conv1d package), read as depthwise (one filter per
 * channel), width 4, zero history before t = 0:
 *     v_t = conv_b[d] + sum_{k=0}^{3} conv_w[d, k] x[t - 3 + k]
 *     u_t = v_t                      (act 0)
 *     u_t = v_t / (1 + exp(-v_t))    (act 1, SiLU as in the usual Mamba block)
 * then the zero-order-hold scan of oracle_scan_fwd on u (in float64, u is not
 * rounded to the input dtype).  x has the layout and dtype of u.
 */
static void conv_scan_channel(const void *x, const float *conv_w, const float *conv_b, int act,
                              const void *delta, const float *dt_bias, const float *A,
                              const void *B, const void *C, const float *Dskip,
                              const void *z, double *y, double *h_last, int64_t b,
                              int64_t d, int64_t L, int64_t D, int64_t N, int dtype,
                              double *h)
{
    memset(h, 0, sizeof(double) * (size_t)N);
    const double bias_d = dt_bias ? (double)dt_bias[d] : 0.0;
    const double skip_d = Dskip ? (double)Dskip[d] : 0.0;
    const double cb = conv_b ? (double)conv_b[d] : 0.0;
    for (int64_t t = 0; t < L; t++) {
        int64_t i_btd = (b * L + t) * D + d;
        double v = cb;
        for (int k = 0; k < 4; k++) {
            int64_t ts = t - 3 + k;
            if (ts >= 0)
                v += (double)conv_w[d * 4 + k] * load_elem(x, (b * L + ts) * D + d, dtype);
        }
        const double ut = act ? v / (1.0 + exp(-v)) : v;
        double dt = softplus(load_elem(delta, i_btd, dtype) + bias_d);
        double acc = 0.0;
        for (int64_t n = 0; n < N; n++) {
            double a = (double)A[d * N + n];
            double abar = exp(dt * a);
            double coef = a != 0.0 ? expm1(dt * a) / a : dt;
            h[n] = abar * h[n] + coef * load_elem(B, (b * L + t) * N + n, dtype) * ut;
            acc += load_elem(C, (b * L + t) * N + n, dtype) * h[n];
        }
        double out = acc + skip_d * ut;
        if (z)
            out *= silu(load_elem(z, i_btd, dtype));
        y[i_btd] = out;
    }
    if (h_last) {
        double *hl = h_last + (b * D + d) * N;
        for (int64_t n = 0; n < N; n++)
            hl[n] = h[n];
    }
}

/* Convolution (conv_w [D, 4], conv_b [D] or NULL, act 0/1) then the scan. */
int oracle_conv_scan_fwd(const void *x, const float *conv_w, const float *conv_b, int act,
                         const void *delta, const float *dt_bias, const float *A,
                         const void *B, const void *C, const float *Dskip, const void *z,
                         double *y, double *h_last, int64_t batch, int64_t L, int64_t D,
                         int64_t N, int dtype, int64_t d_begin, int64_t d_end)
{
    if (!x || !conv_w || !delta || !A || !B || !C || !y)
        return -1;
    if (batch < 0 || L < 0 || D < 0 || N < 1 || (dtype != 0 && dtype != 1) ||
        (act != 0 && act != 1))
        return -1;
    if (d_begin < 0 || d_end > D || d_begin > d_end)
        return -1;
    double *h = (double *)malloc(sizeof(double) * (size_t)N);
    if (!h)
        return -2;
    for (int64_t b = 0; b < batch; b++)
        for (int64_t d = d_begin; d < d_end; d++)
            conv_scan_channel(x, conv_w, conv_b, act, delta, dt_bias, A, B, C, Dskip, z, y,
                              h_last, b, d, L, D, N, dtype, h);
    free(h);
    return 0;
}

/*
 * Backward pass of the zero-order-hold scan: the reverse-mode derivative
 * (adjoint) of oracle_scan_fwd for a loss whose derivative is dy with
 * respect to y and dh_last (NULL means 0) with respect to h_last.  The
 * backward half of the layer is what the fused kernel on the ta-paperlens
 * page recomputes states for instead of storing them ("代償と、それを払う方法
 * （並列スキャン）"); this oracle simply keeps every state of the channel.
 *
 * With s_t = sum_n C_t[n] h_t[n] + Dskip u_t, y_t = s_t g_t, g = silu(z)
 * (g = 1 without z), q[n] = (Abar[n] - 1)/a[n] and lam[n] the derivative of
 * the loss with respect to h_t[n], walking t from L-1 down to 0:
 *   ds_t     = dy_t g_t
 *   dz_t     = dy_t s_t silu'(z_t),   silu'(z) = sig(z) (1 + z (1 - sig(z)))
 *   lam[n]  += ds_t C_t[n]                      (h_t is read out at step t)
 *   dC_t[n] += ds_t h_t[n]
 *   dB_t[n] += lam[n] q[n] u_t
 *   du_t     = ds_t Dskip + sum_n lam[n] q[n] B_t[n]
 *   ddt      = sum_n lam[n] Abar[n] (a[n] h_{t-1}[n] + B_t[n] u_t)
 *              (d Abar/d dt = a Abar, d q/d dt = Abar)
 *   dA[n]   += lam[n] (dt Abar[n] h_{t-1}[n] + q'[n] B_t[n] u_t),
 *              q' = d q/d a = dt^2 (x e^x - (e^x - 1)) / x^2 with x = dt a,
 *              dt^2/2 at a == 0
 *   ddelta_t = ddt sig(delta_t + bias)          (softplus' = sigmoid)
 *   ddt_bias += ddelta_t;  dDskip += ds_t u_t
 *   lam[n]   = Abar[n] lam[n]                   (h_{t-1} feeds h_t)
 * starting from lam = dh_last and h_{-1} = 0.
 * Outputs (float64): du, ddelta, dz [B, L, D] (dz may be NULL, and is
 * ignored without z); dA [D, N], ddt_bias [D], dDskip [D] are written for the
 * channels in [d_begin, d_end) (sums over batch and steps); dB, dC [B, L, N]
 * are ADDED to (sums over channels: the caller zeroes them, and gives each
 * thread its own pair when it splits the channel range).
 */
static double sigmoid_of(double v) { return 1.0 / (1.0 + exp(-v)); }

/* d/da of (exp(dt a) - 1)/a. */
static double dq_da(double dt, double a)
{
    double x = dt * a;
    if (fabs(x) < 1e-3) /* Taylor series of (x e^x - e^x + 1)/x^2 */
        return dt * dt * (0.5 + x * (1.0 / 3.0 + x * (1.0 / 8.0 + x * (1.0 / 30.0))));
    return dt * dt * (x * exp(x) - expm1(x)) / (x * x);
}

static void bwd_channel(const void *u, const void *delta, const float *dt_bias, const float *A,
                        const void *B, const void *C, const float *Dskip, const void *z,
                        const void *dy, const float *dh_last, double *du, double *ddelta,
                        double *ddt_bias, double *dA, double *dB, double *dC, double *dDskip,
                        double *dz, int64_t b, int64_t d, int64_t L, int64_t D, int64_t N,
                        int dtype, double *traj, double *lam)
{
    const double bias_v = dt_bias ? (double)dt_bias[d] : 0.0;
    const double skip_v = Dskip ? (double)Dskip[d] : 0.0;
    /* forward: every state h_t, kept in traj[t * N + n] */
    for (int64_t t = 0; t < L; t++) {
        const int64_t e = (b * L + t) * D + d;
        const double ut = load_elem(u, e, dtype);
        const double dt = softplus(load_elem(delta, e, dtype) + bias_v);
        for (int64_t n = 0; n < N; n++) {
            double abar, q;
            zoh(dt, (double)A[d * N + n], &abar, &q);
            const double prev = t > 0 ? traj[(t - 1) * N + n] : 0.0;
            traj[t * N + n] = abar * prev + q * load_elem(B, (b * L + t) * N + n, dtype) * ut;
        }
    }
    for (int64_t n = 0; n < N; n++)
        lam[n] = dh_last ? (double)dh_last[(b * D + d) * N + n] : 0.0;
    /* backward */
    for (int64_t t = L - 1; t >= 0; t--) {
        const int64_t e = (b * L + t) * D + d;
        const double ut = load_elem(u, e, dtype);
        const double pre = load_elem(delta, e, dtype) + bias_v;
        const double dt = softplus(pre);
        const double dyt = load_elem(dy, e, dtype);
        double s = skip_v * ut;
        for (int64_t n = 0; n < N; n++)
            s += load_elem(C, (b * L + t) * N + n, dtype) * traj[t * N + n];
        double g = 1.0, ds = dyt;
        if (z) {
            const double zt = load_elem(z, e, dtype);
            const double sg = sigmoid_of(zt);
            g = zt * sg;
            ds = dyt * g;
            if (dz)
                dz[e] = dyt * s * sg * (1.0 + zt * (1.0 - sg));
        }
        double du_t = ds * skip_v, ddt = 0.0;
        for (int64_t n = 0; n < N; n++) {
            const int64_t r = (b * L + t) * N + n;
            const double a = (double)A[d * N + n];
            const double bt = load_elem(B, r, dtype);
            const double ht = traj[t * N + n];
            const double hp = t > 0 ? traj[(t - 1) * N + n] : 0.0;
            double abar, q;
            zoh(dt, a, &abar, &q);
            lam[n] += ds * load_elem(C, r, dtype);
            dC[r] += ds * ht;
            dB[r] += lam[n] * q * ut;
            du_t += lam[n] * q * bt;
            ddt += lam[n] * abar * (a * hp + bt * ut);
            dA[d * N + n] += lam[n] * (dt * abar * hp + dq_da(dt, a) * bt * ut);
            lam[n] *= abar;
        }
        du[e] = du_t;
        const double dd = ddt * sigmoid_of(pre);
        ddelta[e] = dd;
        if (ddt_bias)
            ddt_bias[d] += dd;
        if (dDskip)
            dDskip[d] += ds * ut;
    }
}

int oracle_scan_bwd(const void *u, const void *delta, const float *dt_bias, const float *A,
                    const void *B, const void *C, const float *Dskip, const void *z,
                    const void *dy, const float *dh_last, double *du, double *ddelta,
                    double *ddt_bias, double *dA, double *dB, double *dC, double *dDskip,
                    double *dz, int64_t batch, int64_t L, int64_t D, int64_t N, int dtype,
                    int64_t d_begin, int64_t d_end)
{
    if (!u || !delta || !A || !B || !C || !dy || !du || !ddelta || !dA || !dB || !dC)
        return -1;
    if (batch < 0 || L < 0 || D < 0 || N < 1 || (dtype != 0 && dtype != 1))
        return -1;
    if (d_begin < 0 || d_end > D || d_begin > d_end)
        return -1;
    double *traj = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * (size_t)N);
    double *lam = (double *)malloc(sizeof(double) * (size_t)N);
    if (!traj || !lam) {
        free(traj);
        free(lam);
        return -2;
    }
    for (int64_t d = d_begin; d < d_end; d++) {
        for (int64_t n = 0; n < N; n++)
            dA[d * N + n] = 0.0;
        if (ddt_bias)
            ddt_bias[d] = 0.0;
        if (dDskip)
            dDskip[d] = 0.0;
        for (int64_t b = 0; b < batch; b++)
            bwd_channel(u, delta, dt_bias, A, B, C, Dskip, z, dy, dh_last, du, ddelta, ddt_bias,
                        dA, dB, dC, dDskip, dz, b, d, L, D, N, dtype, traj, lam);
    }
    free(traj);
    free(lam);
    return 0;
}

/* ABI probe used by the Python wrapper to refuse a stale build. */
int oracle_abi_version(void) { return 4; }
