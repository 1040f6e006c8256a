/*
 * Selective-scan oracle: plain, sequential, fp64 CPU restatement of the
 * Mamba selective state-space recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes, and where each step comes from:
 *
 *   - The discrete linear recurrence  h_t = Abar h_{t-1} + Bbar x_t,
 *     y_t = C h_t  ("Mamba", elemedex.maurosantelli.com.ar, section
 *     "How it works"; "State Spaces, Selectively - Mamba", papermap
 *     interactive paper explainer, Chapter 02 "The Discretized View").
 *   - Zero-order-hold discretisation with step size Delta: Abar = exp(Delta A)
 *     ("Mamba remembers by forgetting, read closely", interactiveml.org,
 *     the scalar recurrence h_t = exp(-Delta_t) h_{t-1} + ...), and one of
 *     two input terms, chosen by the caller:
 *       Bbar x = Delta B x (the first-order form, the library's default; the
 *       pages say only that Abar and Bbar are derived from (Delta, A, B)), or
 *       Bbar x = (exp(Delta A) - 1) / A * B x, the exact zero-order hold of
 *       a diagonal A (with the limit Delta B x at A = 0).  For A = -1, B = 1
 *       this is the interactiveml.org scalar update
 *       h_t = exp(-Delta_t) h_{t-1} + (1 - exp(-Delta_t)) x_t.
 *   - Selection: Delta, B and C are given per token ("How it works",
 *     elemedex; "The Discretized View", papermap).  A is diagonal: one real
 *     decay per (channel, state) pair.
 *   - The state starts at zero (the interactiveml.org listing starts its
 *     state at 0).
 *   - Options that the pages do not spell out and that follow the usual
 *     Mamba layer interface: Delta = softplus(delta + delta_bias) when
 *     requested, a per-channel skip term D x_t, and an output gate
 *     y_t *= silu(z_t) ("output gate" in "Simplifications and limits" of the
 *     sghael.github.io Mamba page; "multiplicative gate" in the elemedex
 *     entry).  The gate multiplies the whole output, skip term included.
 *
 * The recurrence is exact, so the oracle is the definition itself, written
 * as loops in the order the pages state the steps; no blocking, fusion or
 * reordering.  Inputs are read from the same host arrays the GPU receives
 * (fp32 widened, bf16 decoded exactly) or from fp64 arrays.
 *
 * Parity status: pinned (see the oracle pin tests).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* element type codes for the array arguments */
enum { OR_F32 = 0, OR_BF16 = 1, OR_F64 = 2 };

/* Read element i of an array of the given type, widened to double.  bf16 is
 * the top half of an IEEE fp32, so shifting it up decodes it exactly. */
static double load(int type, const void* p, int64_t i) {
    if (type == OR_F64) return ((const double*)p)[i];
    if (type == OR_F32) return (double)((const float*)p)[i];
    uint32_t bits = (uint32_t)((const uint16_t*)p)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* softplus(v) = log(1 + e^v), written so that neither branch overflows. */
static double softplus(double v) {
    if (v > 0.0) return v + log1p(exp(-v));
    return log1p(exp(v));
}

/* silu(z) = z * sigmoid(z) = z / (1 + e^-z). */
static double silu(double z) { return z / (1.0 + exp(-z)); }

/* The factor that multiplies B x in the state update: Delta for the
 * first-order input term, (exp(Delta A) - 1) / A for the exact zero-order
 * hold, whose limit at A = 0 is Delta (expm1 keeps it accurate when
 * Delta A is small). */
static double input_weight(int zoh, double dt, double a) {
    if (!zoh) return dt;
    return a != 0.0 ? expm1(dt * a) / a : dt;
}

/* The weight's derivatives, for the backward pass.  d w / d Delta: 1, or
 * exp(Delta A) for the exact hold.  d w / d A: 0, or for the exact hold
 * (Delta e^x - (e^x - 1) / A) / A with x = Delta A, which is Delta^2 psi(x),
 * psi(x) = (x e^x - e^x + 1) / x^2 = sum_{k>=0} (k + 1) x^k / (k + 2)!; the
 * series (to k = 29, far below double rounding for |x| < 1/2) stands in for
 * the closed form where it would cancel, and gives Delta^2 / 2 at A = 0. */
static double input_weight_ddt(int zoh, double dt, double a) { return zoh ? exp(dt * a) : 1.0; }
static double input_weight_da(int zoh, double dt, double a) {
    if (!zoh) return 0.0;
    const double x = dt * a;
    if (fabs(x) < 0.5) {
        double sum = 0.0, xp = 1.0, fact = 2.0;   /* x^k, (k + 2)! */
        for (int k = 0; k < 30; k++) {
            sum += (k + 1) * xp / fact;
            xp *= x;
            fact *= (double)(k + 3);
        }
        return dt * dt * sum;
    }
    return (dt * exp(x) - expm1(x) / a) / a;
}

typedef struct {
    int64_t batch, dim, dstate, seqlen;
    int io, pio; /* element types: io for u/delta/B/C/z, pio for A/D/bias */
    const void *u, *delta, *A, *B, *C, *D, *z, *bias;
    int softplus_on;
    int zoh;             /* 0: Bbar = Delta B; 1: Bbar = (exp(Delta A) - 1) / A B */
    const int64_t* chan; /* flat channel ids b*dim + d, or NULL for all */
    int64_t nchan;
    double* y;          /* nchan x seqlen */
    double* last_state; /* nchan x dstate, or NULL */
    const double* h0;   /* nchan x dstate initial state, or NULL for zero */
    int64_t next;       /* work counter, guarded by mu */
    pthread_mutex_t mu;
} scan_job;

/* One channel (b, d): the recurrence over t = 0 .. L-1. */
static void scan_channel(const scan_job* j, int64_t k, double* h) {
    const int64_t L = j->seqlen, N = j->dstate;
    const int64_t c = j->chan ? j->chan[k] : k;
    const int64_t b = c / j->dim, d = c % j->dim;
    const int64_t row = c * L;            /* u, delta, z: (batch, dim, L) */
    const int64_t bc_row = b * L * N;     /* B, C: (batch, L, N) */
    const double bias = j->bias ? load(j->pio, j->bias, d) : 0.0;
    const double Dskip = j->D ? load(j->pio, j->D, d) : 0.0;
    for (int64_t n = 0; n < N; n++) h[n] = j->h0 ? j->h0[k * N + n] : 0.0;
    for (int64_t t = 0; t < L; t++) {
        const double v = load(j->io, j->delta, row + t) + bias;
        const double dt = j->softplus_on ? softplus(v) : v;
        const double x = load(j->io, j->u, row + t);
        double yv = 0.0;
        for (int64_t n = 0; n < N; n++) {
            const double a = load(j->pio, j->A, d * N + n);
            const double Bv = load(j->io, j->B, bc_row + t * N + n);
            h[n] = exp(dt * a) * h[n] + input_weight(j->zoh, dt, a) * Bv * x;
        }
        for (int64_t n = 0; n < N; n++)
            yv += load(j->io, j->C, bc_row + t * N + n) * h[n];
        yv += Dskip * x;
        if (j->z) yv *= silu(load(j->io, j->z, row + t));
        j->y[k * L + t] = yv;
    }
    if (j->last_state)
        for (int64_t n = 0; n < N; n++) j->last_state[k * N + n] = h[n];
}

static void* scan_worker(void* arg) {
    scan_job* j = (scan_job*)arg;
    double* h = (double*)malloc(sizeof(double) * (size_t)j->dstate);
    if (!h) return NULL;
    for (;;) {
        pthread_mutex_lock(&j->mu);
        const int64_t k = j->next++;
        pthread_mutex_unlock(&j->mu);
        if (k >= j->nchan) break;
        scan_channel(j, k, h);
    }
    free(h);
    return NULL;
}

/*
 * Forward selective scan over the channels listed in `chan` (flat ids
 * b*dim + d; NULL means every channel in order, and then nchan must equal
 * batch*dim).  Outputs are compact: y is nchan x seqlen, last_state is
 * nchan x dstate.  h0 (nchan x dstate, fp64) is an optional initial state;
 * NULL means zero.  zoh selects the input term (0: Delta B x, 1: the exact
 * zero-order hold (exp(Delta A) - 1) / A B x).  Channels are independent, so
 * they are spread over `nthreads` POSIX threads; each channel's loop is
 * sequential.  Returns 0, or -1 on a bad argument.
 */
int oracle_scan_fwd(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, int io, int pio,
                    const void* u, const void* delta, const void* A, const void* B,
                    const void* C, const void* D, const void* z, const void* delta_bias,
                    int delta_softplus, int zoh, const int64_t* chan, int64_t nchan,
                    const double* h0, double* y, double* last_state, int nthreads) {
    if (batch <= 0 || dim <= 0 || dstate <= 0 || seqlen < 0 || nchan < 0) return -1;
    if (!u || !delta || !A || !B || !C || !y) return -1;
    if (io < OR_F32 || io > OR_F64 || (pio != OR_F32 && pio != OR_F64)) return -1;
    if (!chan && nchan != batch * dim) return -1;
    if (chan)
        for (int64_t k = 0; k < nchan; k++)
            if (chan[k] < 0 || chan[k] >= batch * dim) return -1;
    scan_job j;
    memset(&j, 0, sizeof j);
    j.batch = batch; j.dim = dim; j.dstate = dstate; j.seqlen = seqlen;
    j.io = io; j.pio = pio;
    j.u = u; j.delta = delta; j.A = A; j.B = B; j.C = C; j.D = D; j.z = z;
    j.bias = delta_bias; j.softplus_on = delta_softplus; j.zoh = zoh != 0;
    j.chan = chan; j.nchan = nchan; j.y = y; j.last_state = last_state; j.h0 = h0;
    j.next = 0;
    pthread_mutex_init(&j.mu, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    int started = 0;
    for (int i = 1; i < nthreads; i++)
        if (pthread_create(&th[started], NULL, scan_worker, &j) == 0) started++;
    scan_worker(&j);
    for (int i = 0; i < started; i++) pthread_join(th[i], NULL);
    pthread_mutex_destroy(&j.mu);
    return 0;
}

/*
 * One token of recurrent (generation) mode: the same update with L = 1,
 * starting from the given state, which is updated in place.  Recurrent mode
 * costs the same for every token ("Training without stepping token by
 * token", sghael.github.io Mamba page).
 * Shapes: state (batch, dim, dstate) fp64; x, delta, z, y (batch, dim);
 * B, C (batch, dstate); A (dim, dstate); D, delta_bias (dim).
 */
int oracle_state_step(int64_t batch, int64_t dim, int64_t dstate, int io, int pio,
                      double* state, const void* x, const void* delta, const void* A,
                      const void* B, const void* C, const void* D, const void* z,
                      const void* delta_bias, int delta_softplus, double* y) {
    if (batch <= 0 || dim <= 0 || dstate <= 0) return -1;
    if (!state || !x || !delta || !A || !B || !C || !y) return -1;
    if (io < OR_F32 || io > OR_F64 || (pio != OR_F32 && pio != OR_F64)) return -1;
    for (int64_t b = 0; b < batch; b++) {
        for (int64_t d = 0; d < dim; d++) {
            const int64_t c = b * dim + d;
            const double bias = delta_bias ? load(pio, delta_bias, d) : 0.0;
            const double v = load(io, delta, c) + bias;
            const double dt = delta_softplus ? softplus(v) : v;
            const double xv = load(io, x, c);
            double* h = state + c * dstate;
            double yv = 0.0;
            for (int64_t n = 0; n < dstate; n++) {
                const double a = load(pio, A, d * dstate + n);
                h[n] = exp(dt * a) * h[n] + dt * load(io, B, b * dstate + n) * xv;
            }
            for (int64_t n = 0; n < dstate; n++) yv += load(io, C, b * dstate + n) * h[n];
            yv += (D ? load(pio, D, d) : 0.0) * xv;
            if (z) yv *= silu(load(io, z, c));
            y[c] = yv;
        }
    }
    return 0;
}

/*
 * Backward pass of the forward scan above (gradients for training): given
 * dy = dLoss/dy (and optionally dlast = dLoss/dlast_state), the gradients of
 * the loss with respect to every input.  The pages describe the backward
 * pass only as the forward recomputed in on-chip memory instead of storing
 * the expanded state ("State Spaces, Selectively - Mamba", papermap,
 * "The hardware-aware scan"); this oracle states what that pass must
 * produce: the reverse-mode derivative of the recurrence, written out
 * step by step in reverse token order.
 *
 * For one channel (b, d), with x_t = u_t, v_t = delta_t + bias,
 * Delta_t = softplus(v_t) (or v_t), a_tn = exp(Delta_t A_n),
 * h_tn = a_tn h_(t-1)n + Delta_t B_tn x_t, s_t = sum_n C_tn h_tn + D x_t and
 * y_t = s_t silu(z_t) (or s_t), let g_n be the adjoint of h_tn.  The forward
 * starts from h_(-1) = h0 (zero when no initial state is given); its input
 * term is w_tn B_tn x_t with w = Delta (first order) or (exp(Delta A) - 1) / A
 * (exact hold), w' = dw/dDelta, w_A = dw/dA (input_weight_ddt, _da).  Going
 * from t = L-1 down to 0, starting from g = dlast:
 *
 *   ds_t   = dy_t silu(z_t)           dz_t = dy_t s_t silu'(z_t)
 *   dD    += ds_t x_t                 dx_t = ds_t D
 *   g_n   += ds_t C_tn                dC_tn = ds_t h_tn
 *   dDelta_t = sum_n g_n (A_n a_tn h_(t-1)n + w'_tn B_tn x_t)
 *   dx_t  += sum_n g_n w_tn B_tn      dB_tn = g_n w_tn x_t
 *   dA_n  += g_n (Delta_t a_tn h_(t-1)n + w_A,tn B_tn x_t)
 *   g_n    = g_n a_tn                 (the adjoint of h_(t-1)n)
 *   ddelta_t = dDelta_t sigmoid(v_t) (softplus' = sigmoid) or dDelta_t
 *   dbias += ddelta_t
 *
 * The forward states h_t are recomputed first and kept for the channel
 * (L x N doubles), then the loop above runs.  Per-channel outputs: du,
 * ddelta, dz (nchan x L), dA (nchan x N), dD, dbias (nchan), and the
 * channel's terms of dB, dC (nchan x L x N; the caller sums them over the
 * channels of a batch row) and dh0 = g after t = 0 (nchan x N).
 */
typedef struct {
    int64_t batch, dim, dstate, seqlen;
    int io, pio;
    const void *u, *delta, *A, *B, *C, *D, *z, *bias;
    int softplus_on;
    const double *dy, *dlast;   /* (batch, dim, L), (batch, dim, N) (dlast may be NULL) */
    const double* h0;           /* (batch, dim, N) initial state, or NULL for zero */
    int zoh;                    /* input term: 0 first order, 1 exact zero-order hold */
    double *du, *ddelta, *dz, *dA, *dD, *dbias, *dBc, *dCc, *dh0;
    const int64_t* chan;        /* flat channel ids, or NULL for all */
    int64_t nchan, next;
    pthread_mutex_t mu;
} bwd_job;

static double sigmoid(double v) { return 1.0 / (1.0 + exp(-v)); }

/* channel c = chan[k] (or k); its outputs go to row k of the compact arrays,
 * dy and dlast are read at row c of the full arrays */
static void bwd_channel(const bwd_job* j, int64_t k, double* hs, double* g) {
    const int64_t L = j->seqlen, N = j->dstate;
    const int64_t c = j->chan ? j->chan[k] : k;
    const int64_t b = c / j->dim, d = c % j->dim;
    const int64_t row = c * L, bc_row = b * L * N;
    const double bias = j->bias ? load(j->pio, j->bias, d) : 0.0;
    const double Dskip = j->D ? load(j->pio, j->D, d) : 0.0;
    /* forward: hs[(t + 1) * N + n] = h_tn, hs[n] = h_(-1)n = h0 (or 0) */
    for (int64_t n = 0; n < N; n++) hs[n] = j->h0 ? j->h0[c * N + n] : 0.0;
    for (int64_t t = 0; t < L; t++) {
        const double v = load(j->io, j->delta, row + t) + bias;
        const double dt = j->softplus_on ? softplus(v) : v;
        const double x = load(j->io, j->u, row + t);
        for (int64_t n = 0; n < N; n++) {
            const double An = load(j->pio, j->A, d * N + n);
            const double a = exp(dt * An);
            hs[(t + 1) * N + n] = a * hs[t * N + n] +
                                  input_weight(j->zoh, dt, An) * load(j->io, j->B, bc_row + t * N + n) * x;
        }
    }
    /* reverse */
    for (int64_t n = 0; n < N; n++) {
        g[n] = j->dlast ? j->dlast[c * N + n] : 0.0;
        j->dA[k * N + n] = 0.0;
    }
    double dD = 0.0, dbias = 0.0;
    for (int64_t t = L - 1; t >= 0; t--) {
        const double v = load(j->io, j->delta, row + t) + bias;
        const double dt = j->softplus_on ? softplus(v) : v;
        const double x = load(j->io, j->u, row + t);
        const double* h = hs + (t + 1) * N;
        const double* hp = hs + t * N;
        double s = Dskip * x;
        for (int64_t n = 0; n < N; n++) s += load(j->io, j->C, bc_row + t * N + n) * h[n];
        const double dyv = j->dy[c * L + t];
        double ds = dyv;
        if (j->z) {
            const double zv = load(j->io, j->z, row + t);
            const double sg = sigmoid(zv);
            ds = dyv * zv * sg;
            j->dz[k * L + t] = dyv * s * sg * (1.0 + zv * (1.0 - sg));
        } else if (j->dz) {
            j->dz[k * L + t] = 0.0;
        }
        dD += ds * x;
        double dx = ds * Dskip, ddt = 0.0;
        for (int64_t n = 0; n < N; n++) {
            const double Cv = load(j->io, j->C, bc_row + t * N + n);
            const double Bv = load(j->io, j->B, bc_row + t * N + n);
            const double An = load(j->pio, j->A, d * N + n);
            const double a = exp(dt * An);
            const double w = input_weight(j->zoh, dt, An);
            g[n] += ds * Cv;
            j->dCc[(k * L + t) * N + n] = ds * h[n];
            ddt += g[n] * (An * a * hp[n] + input_weight_ddt(j->zoh, dt, An) * Bv * x);
            dx += g[n] * w * Bv;
            j->dBc[(k * L + t) * N + n] = g[n] * w * x;
            j->dA[k * N + n] += g[n] * (dt * a * hp[n] + input_weight_da(j->zoh, dt, An) * Bv * x);
            g[n] *= a;
        }
        const double dv = j->softplus_on ? ddt * sigmoid(v) : ddt;
        j->ddelta[k * L + t] = dv;
        j->du[k * L + t] = dx;
        dbias += dv;
    }
    j->dD[k] = dD;
    j->dbias[k] = dbias;
    if (j->dh0)
        for (int64_t n = 0; n < N; n++) j->dh0[k * N + n] = g[n];
}

static void* bwd_worker(void* arg) {
    bwd_job* j = (bwd_job*)arg;
    double* hs = (double*)malloc(sizeof(double) * (size_t)((j->seqlen + 1) * j->dstate));
    double* g = (double*)malloc(sizeof(double) * (size_t)j->dstate);
    if (!hs || !g) {
        free(hs);
        free(g);
        return NULL;
    }
    for (;;) {
        pthread_mutex_lock(&j->mu);
        const int64_t k = j->next++;
        pthread_mutex_unlock(&j->mu);
        if (k >= j->nchan) break;
        bwd_channel(j, k, hs, g);
    }
    free(hs);
    free(g);
    return NULL;
}

/*
 * Backward selective scan over the channels listed in `chan` (flat ids
 * b*dim + d; NULL means every channel in order, and then nchan must equal
 * batch*dim); see the comment above.  Inputs as for oracle_scan_fwd; dy is
 * (batch, dim, L) fp64, dlast (batch, dim, N) fp64 or NULL and h0, the
 * forward's initial state, (batch, dim, N) fp64 or NULL, all full; zoh
 * selects the input term as for oracle_scan_fwd.
 * Outputs (fp64, compact, one row per listed channel): du, ddelta, dz
 * (nchan x L; dz may be NULL when z is), dA (nchan x N: the channel's
 * share, summed over the batch by the caller), dD, dbias (nchan), dBc, dCc
 * (nchan x L x N: per-channel terms) and dh0 (nchan x N) or NULL.
 * Returns 0, or -1 on a bad argument.
 */
int oracle_scan_bwd(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, int io, int pio,
                    const void* u, const void* delta, const void* A, const void* B,
                    const void* C, const void* D, const void* z, const void* delta_bias,
                    int delta_softplus, const double* dy, const double* dlast, const double* h0,
                    int zoh, const int64_t* chan, int64_t nchan, double* du, double* ddelta, double* dz,
                    double* dA, double* dD, double* dbias, double* dBc, double* dCc, double* dh0,
                    int nthreads) {
    if (batch <= 0 || dim <= 0 || dstate <= 0 || seqlen < 0) return -1;
    if (!u || !delta || !A || !B || !C || !dy || !du || !ddelta || !dA || !dD || !dbias || !dBc ||
        !dCc)
        return -1;
    if (z && !dz) return -1;
    if (io < OR_F32 || io > OR_F64 || (pio != OR_F32 && pio != OR_F64)) return -1;
    if (!chan && nchan != batch * dim) return -1;
    if (chan)
        for (int64_t k = 0; k < nchan; k++)
            if (chan[k] < 0 || chan[k] >= batch * dim) return -1;
    bwd_job j;
    memset(&j, 0, sizeof j);
    j.batch = batch; j.dim = dim; j.dstate = dstate; j.seqlen = seqlen;
    j.io = io; j.pio = pio;
    j.u = u; j.delta = delta; j.A = A; j.B = B; j.C = C; j.D = D; j.z = z;
    j.bias = delta_bias; j.softplus_on = delta_softplus;
    j.dy = dy; j.dlast = dlast; j.h0 = h0; j.zoh = zoh;
    j.du = du; j.ddelta = ddelta; j.dz = dz; j.dA = dA; j.dD = dD; j.dbias = dbias;
    j.dBc = dBc; j.dCc = dCc; j.dh0 = dh0;
    j.chan = chan;
    j.nchan = nchan;
    j.next = 0;
    pthread_mutex_init(&j.mu, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    int started = 0;
    for (int i = 1; i < nthreads; i++)
        if (pthread_create(&th[started], NULL, bwd_worker, &j) == 0) started++;
    bwd_worker(&j);
    for (int i = 0; i < started; i++) pthread_join(th[i], NULL);
    pthread_mutex_destroy(&j.mu);
    return 0;
}

/*
 * The block's short convolution, which produces the scan's input u from the
 * block input x ("Mamba", elemedex entry, section "How it works": the block
 * is a linear projection, a short convolution, the selective SSM and a
 * multiplicative gate; "Simplifications and limits" of the sghael.github.io
 * Mamba page: a short convolution).  The pages give no more detail; the
 * reading taken (the usual Mamba layer) is a causal depthwise convolution of
 * width K (each channel filtered by its own K taps, output t seeing inputs
 * t-K+1 .. t), a per-channel bias, and the SiLU activation:
 *
 *   u[b,d,t] = silu( sum_{k=0}^{K-1} w[d,k] * x[b,d,t-(K-1)+k] + cbias[d] )
 *
 * Inputs before token 0 are the K-1 values of `state` (batch, dim, K-1),
 * oldest first, or zero when state is NULL.  x and state have the element
 * type io (fp32, bf16 bits or fp64); w (dim, K) and cbias (dim) have type
 * pio.  u is fp64 (batch, dim, L).  Returns 0, or -1 on a bad argument.
 */
int oracle_conv_silu(int64_t batch, int64_t dim, int64_t seqlen, int64_t K, int io, int pio,
                     const void* x, const void* w, const void* cbias, const void* state,
                     double* u) {
    if (batch <= 0 || dim <= 0 || seqlen < 0 || K < 1 || !x || !w || !u) return -1;
    if (io < OR_F32 || io > OR_F64 || (pio != OR_F32 && pio != OR_F64)) return -1;
    for (int64_t b = 0; b < batch; b++) {
        for (int64_t d = 0; d < dim; d++) {
            const int64_t c = b * dim + d;
            for (int64_t t = 0; t < seqlen; t++) {
                double acc = cbias ? load(pio, cbias, d) : 0.0;
                for (int64_t k = 0; k < K; k++) {
                    const int64_t src = t - (K - 1) + k;   /* the input this tap sees */
                    double xv = 0.0;
                    if (src >= 0)
                        xv = load(io, x, c * seqlen + src);
                    else if (state)
                        xv = load(io, state, c * (K - 1) + (K - 1) + src);
                    acc += load(pio, w, d * K + k) * xv;
                }
                u[c * seqlen + t] = silu(acc);
            }
        }
    }
    return 0;
}
