/*
 * oracle.c -- plain, slow fp64 CPU oracle for Mamba's selective scan.
 *
 * TEST INFRASTRUCTURE ONLY. This file exists so that the tests, the smoke
 * check and the CPU-baseline leg of the benchmark can compare the CUDA path
 * against an obviously correct restatement of the method. Nothing on the
 * product path may link, load or call it, and it shares no code, header,
 * table or helper with the CUDA library.
 *
 * What it computes (source: "Mamba: Selective State Space Models",
 * youngju.dev, section 3.3 "Hardware-Aware algorithm", the simplified
 * selective_scan listing; the discrete recurrence of section 2.2; shapes as
 * in booiljung.github.io "3.1 LTI ... Input-Dependent parameters",
 * section 0.4.2):
 *
 *   x, delta : (Bsz, L, D)      A : (D, N)      B, C : (Bsz, L, N)
 *   for every batch b and channel d, with h[0..N) = h0[b,d,:] (zeros if absent):
 *     for t = 0 .. L-1:
 *       dl = delta[b,t,d]              (softplus(dl) = log(1 + e^dl) when asked)
 *       for n: h[n] = exp(dl * A[d,n]) * h[n] + (dl * B[b,t,n]) * x[b,t,d]
 *       y[b,t,d] = sum_n h[n] * C[b,t,n]          (read-out after the update)
 *     hT[b,d,:] = h
 *
 * deltaB is the simplified dl * B of the listing. The *_gated entry points
 * take a zoh flag for the zero-order-hold form of section 2.2 instead,
 * Bbar = (dA)^-1 (exp(dA) - I) dB, which for a diagonal A is, per state,
 *   Bbar[n] = dl * B[n] * phi(dl * A[d,n]),   phi(w) = (e^w - 1) / w, phi(0) = 1.
 *
 * Optionally (the *_gated entry points) the output of the block around the
 * scan, as the MambaBlock listing of section 3.4 on the same page has it:
 *   y[b,t,d] = (sum_n h[n] * C[b,t,n] + Dskip[d] * x[b,t,d]) * silu(z[b,t,d])
 * with silu(z) = z / (1 + e^-z). The listing shows the gate and defines the
 * per-channel parameter D (Dskip here) but elides where D enters; the skip is
 * taken before the gate. Either term may be absent.
 *
 * The decode step (the O(1)-state recurrent mode of section 6 on the same
 * page) is one iteration of the t-loop with L = 1, applied in place to a
 * caller-held state, with delta taken as given (no softplus).
 *
 * Inputs are float (exactly the values the GPU sees: fp32 values or
 * bf16 values widened to fp32) except the optional initial state h0, which
 * is double so that a state handed over from an earlier call loses nothing;
 * every operation is done in double.
 * Chains (b, d) are independent, so a pool of POSIX threads splits them;
 * each chain runs the loop above unchanged, so the thread count does not
 * change any result bit.
 *
 * Also here, each with its own comment below: the backward pass of the scan
 * (oracle_selscan_bwd, a plain reverse sweep over each chain's stored
 * states) and of the block's skip and gate (oracle_selscan_bwd_gated), the
 * causal conv1d before the scan (oracle_conv1d), and the Mamba-2 SSD
 * forward (oracle_ssd_fwd).
 *
 * Pins (tests/test_oracle_pins.py): brute-force unrolled sum, A = 0 running
 * sum, N = 1 scalar recurrence, L = 1 closed form, LTI convolution kernel,
 * geometric closed form, delta -> 0 persistence, delta -> inf reset,
 * chunked associative composition, step == forward, linearity; for the
 * backward, central differences of the forward, autograd of an unrolled
 * forward and homogeneity identities; for SSD, its dual quadratic form, a
 * chunked form and the selective scan at headdim 1.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* softplus(u) = log(1 + e^u)   (booiljung.github.io, section 0.4.2).
 * Written as max(u, 0) + log1p(e^-|u|), which is the same function without
 * overflow for large |u|. */
double oracle_softplus(double u)
{
    double a = fabs(u);
    return (u > 0.0 ? u : 0.0) + log1p(exp(-a));
}

/* The block's output around the scan's read-out y for element (b, t, d) at
 * flat index btd: the skip term Dskip[d] * x, then the gate silu(z)
 * = z / (1 + e^-z) (section 3.4). Dskip NULL: no skip; z NULL: no gate. */
static double gate(double y, const float *Dskip, const float *z, int64_t d,
                   int64_t btd, double xv)
{
    if (Dskip)
        y += (double)Dskip[d] * xv;
    if (z) {
        double zv = (double)z[btd];
        y *= zv / (1.0 + exp(-zv));
    }
    return y;
}

/* phi(w) = (e^w - 1) / w, the zero-order-hold factor of section 2.2 for a
 * diagonal A (its limit 1 at w = 0, where dA is not invertible). */
static double zoh_factor(double w)
{
    return w == 0.0 ? 1.0 : expm1(w) / w;
}

/* One (b, d) chain of the forward scan.
 * y_out[t * y_stride] receives y[b,t,d]; h_out[n] receives the final state. */
static void scan_chain(const float *x, const float *delta, const float *A,
                       const float *B, const float *C, const double *h0,
                       const float *Dskip, const float *z, int zoh,
                       int64_t b, int64_t d, int64_t L, int64_t D, int64_t N,
                       int delta_softplus, double *y_out, int64_t y_stride,
                       double *h_out, double *h)
{
    for (int64_t n = 0; n < N; ++n)
        h[n] = h0 ? h0[(b * D + d) * N + n] : 0.0;
    for (int64_t t = 0; t < L; ++t) {
        int64_t bt = b * L + t;
        double dl = (double)delta[bt * D + d];
        if (delta_softplus)
            dl = oracle_softplus(dl);
        double xv = (double)x[bt * D + d];
        double acc = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            double dA = exp(dl * (double)A[d * N + n]);   /* deltaA */
            double dB = dl * (double)B[bt * N + n];        /* deltaB */
            if (zoh)
                dB *= zoh_factor(dl * (double)A[d * N + n]);
            h[n] = dA * h[n] + dB * xv;
        }
        for (int64_t n = 0; n < N; ++n)
            acc += h[n] * (double)C[bt * N + n];
        if (y_out)
            y_out[t * y_stride] = gate(acc, Dskip, z, d, bt * D + d, xv);
    }
    if (h_out)
        for (int64_t n = 0; n < N; ++n)
            h_out[n] = h[n];
}

/* ---- a small thread pool over chain indices -------------------------- */

typedef struct {
    const float *x, *delta, *A, *B, *C;
    const float *Dskip, *z;   /* optional block output (NULL: absent) */
    int zoh;                  /* zero-order-hold Bbar instead of dl * B */
    const double *h0;
    int64_t Bsz, L, D, N;
    int delta_softplus;
    const int64_t *chains; /* NULL: all chains, index c = b * D + d */
    int64_t nchains;
    double *y, *hT;        /* full layout when chains == NULL, else packed */
    int64_t next;          /* next chain to take (under lock) */
    pthread_mutex_t lock;
    int failed;
} fwd_job;

static void *fwd_worker(void *arg)
{
    fwd_job *j = (fwd_job *)arg;
    double *h = (double *)malloc(sizeof(double) * (size_t)(j->N > 0 ? j->N : 1));
    if (!h) {
        pthread_mutex_lock(&j->lock);
        j->failed = 1;
        pthread_mutex_unlock(&j->lock);
        return NULL;
    }
    for (;;) {
        int64_t i;
        pthread_mutex_lock(&j->lock);
        i = j->next++;
        pthread_mutex_unlock(&j->lock);
        if (i >= j->nchains)
            break;
        int64_t c = j->chains ? j->chains[i] : i;
        int64_t b = c / j->D, d = c % j->D;
        double *y_out, *h_out;
        int64_t y_stride;
        if (j->chains) { /* packed: y (nchains, L), hT (nchains, N) */
            y_out = j->y ? j->y + i * j->L : NULL;
            y_stride = 1;
            h_out = j->hT ? j->hT + i * j->N : NULL;
        } else {         /* full: y (Bsz, L, D), hT (Bsz, D, N) */
            y_out = j->y ? j->y + b * j->L * j->D + d : NULL;
            y_stride = j->D;
            h_out = j->hT ? j->hT + c * j->N : NULL;
        }
        scan_chain(j->x, j->delta, j->A, j->B, j->C, j->h0, j->Dskip, j->z, j->zoh, b, d,
                   j->L, j->D, j->N, j->delta_softplus, y_out, y_stride, h_out, h);
    }
    free(h);
    return NULL;
}

static int pick_threads(int nthreads, int64_t work)
{
    if (nthreads <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = n > 0 ? (int)n : 1;
    }
    if (nthreads > 256)
        nthreads = 256;
    if ((int64_t)nthreads > work)
        nthreads = work > 0 ? (int)work : 1;
    return nthreads;
}

static int run_fwd(fwd_job *j, int nthreads)
{
    pthread_t tid[256];
    int started = 0;
    nthreads = pick_threads(nthreads, j->nchains);
    pthread_mutex_init(&j->lock, NULL);
    j->next = 0;
    j->failed = 0;
    for (int i = 1; i < nthreads; ++i)
        if (pthread_create(&tid[started], NULL, fwd_worker, j) == 0)
            ++started;
    fwd_worker(j); /* the calling thread works too */
    for (int i = 0; i < started; ++i)
        pthread_join(tid[i], NULL);
    pthread_mutex_destroy(&j->lock);
    return j->failed ? -1 : 0;
}

/* Full forward scan over every chain.
 * y: (Bsz, L, D) double, may be NULL; hT: (Bsz, D, N) double, may be NULL;
 * h0: (Bsz, D, N) double or NULL for zeros. nthreads <= 0 uses every online
 * CPU. Returns 0, or -1 on bad arguments / allocation failure. */
int oracle_selscan_fwd_gated(const float *x, const float *delta, const float *A,
                             const float *B, const float *C, const float *Dskip,
                             const float *z, const double *h0, double *y, double *hT,
                             int64_t Bsz, int64_t L, int64_t D, int64_t N,
                             int delta_softplus, int zoh, int nthreads);

int oracle_selscan_fwd(const float *x, const float *delta, const float *A,
                       const float *B, const float *C, const double *h0,
                       double *y, double *hT, int64_t Bsz, int64_t L,
                       int64_t D, int64_t N, int delta_softplus, int nthreads)
{
    return oracle_selscan_fwd_gated(x, delta, A, B, C, NULL, NULL, h0, y, hT,
                                    Bsz, L, D, N, delta_softplus, 0, nthreads);
}

/* The forward scan with the block's skip and gate (either may be NULL):
 * Dskip (D), z (Bsz, L, D); zoh selects the zero-order-hold Bbar. */
int oracle_selscan_fwd_gated(const float *x, const float *delta, const float *A,
                             const float *B, const float *C, const float *Dskip,
                             const float *z, const double *h0, double *y, double *hT,
                             int64_t Bsz, int64_t L, int64_t D, int64_t N,
                             int delta_softplus, int zoh, int nthreads)
{
    if (Bsz < 0 || L < 0 || D < 0 || N < 0)
        return -1;
    if (L > 0 && (!x || !delta || !B || !C))
        return -1;
    if (N > 0 && !A)
        return -1;
    fwd_job j;
    memset(&j, 0, sizeof j);
    j.x = x; j.delta = delta; j.A = A; j.B = B; j.C = C; j.h0 = h0;
    j.Dskip = Dskip; j.z = z; j.zoh = zoh;
    j.Bsz = Bsz; j.L = L; j.D = D; j.N = N;
    j.delta_softplus = delta_softplus;
    j.chains = NULL;
    j.nchains = Bsz * D;
    j.y = y; j.hT = hT;
    return run_fwd(&j, nthreads);
}

/* Forward scan for a chosen set of chains only (chain c = b * D + d), for
 * sampled checks of sizes the full oracle would take too long on.
 * y_out: (nchains, L), hT_out: (nchains, N); either may be NULL. */
int oracle_selscan_fwd_chains_gated(const float *x, const float *delta,
                                    const float *A, const float *B, const float *C,
                                    const float *Dskip, const float *z,
                                    const double *h0, const int64_t *chains,
                                    int64_t nchains, double *y_out, double *hT_out,
                                    int64_t Bsz, int64_t L, int64_t D, int64_t N,
                                    int delta_softplus, int zoh, int nthreads);

int oracle_selscan_fwd_chains(const float *x, const float *delta,
                              const float *A, const float *B, const float *C,
                              const double *h0, const int64_t *chains,
                              int64_t nchains, double *y_out, double *hT_out,
                              int64_t Bsz, int64_t L, int64_t D, int64_t N,
                              int delta_softplus, int nthreads)
{
    return oracle_selscan_fwd_chains_gated(x, delta, A, B, C, NULL, NULL, h0, chains,
                                           nchains, y_out, hT_out, Bsz, L, D, N,
                                           delta_softplus, 0, nthreads);
}

/* oracle_selscan_fwd_chains with the block's skip and gate, and zoh. */
int oracle_selscan_fwd_chains_gated(const float *x, const float *delta,
                                    const float *A, const float *B, const float *C,
                                    const float *Dskip, const float *z,
                                    const double *h0, const int64_t *chains,
                                    int64_t nchains, double *y_out, double *hT_out,
                                    int64_t Bsz, int64_t L, int64_t D, int64_t N,
                                    int delta_softplus, int zoh, int nthreads)
{
    if (Bsz < 0 || L < 0 || D < 0 || N < 0 || nchains < 0 || (nchains && !chains))
        return -1;
    for (int64_t i = 0; i < nchains; ++i)
        if (chains[i] < 0 || chains[i] >= Bsz * D)
            return -1;
    fwd_job j;
    memset(&j, 0, sizeof j);
    j.x = x; j.delta = delta; j.A = A; j.B = B; j.C = C; j.h0 = h0;
    j.Dskip = Dskip; j.z = z; j.zoh = zoh;
    j.Bsz = Bsz; j.L = L; j.D = D; j.N = N;
    j.delta_softplus = delta_softplus;
    j.chains = chains;
    j.nchains = nchains;
    j.y = y_out; j.hT = hT_out;
    return run_fwd(&j, nthreads);
}

/* Decode step: one iteration of the loop above, state updated in place.
 *   state : (Bsz, D, N) double, in/out        x, delta : (Bsz, D) float
 *   A : (D, N)        B, C : (Bsz, N)          y : (Bsz, D) double
 * delta is used as given. When chains != NULL only those chains are
 * updated, with state packed as (nchains, N) and y as (nchains). */
int oracle_selscan_step_gated(double *state, const float *x, const float *delta,
                              const float *A, const float *B, const float *C,
                              const float *Dskip, const float *z, double *y,
                              const int64_t *chains, int64_t nchains,
                              int64_t Bsz, int64_t D, int64_t N, int zoh);

int oracle_selscan_step(double *state, const float *x, const float *delta,
                        const float *A, const float *B, const float *C,
                        double *y, const int64_t *chains, int64_t nchains,
                        int64_t Bsz, int64_t D, int64_t N)
{
    return oracle_selscan_step_gated(state, x, delta, A, B, C, NULL, NULL, y,
                                     chains, nchains, Bsz, D, N, 0);
}

/* oracle_selscan_step with the block's skip and gate: Dskip (D), z (Bsz, D);
 * zoh selects the zero-order-hold Bbar. */
int oracle_selscan_step_gated(double *state, const float *x, const float *delta,
                              const float *A, const float *B, const float *C,
                              const float *Dskip, const float *z, double *y,
                              const int64_t *chains, int64_t nchains,
                              int64_t Bsz, int64_t D, int64_t N, int zoh)
{
    if (!state || !x || !delta || !A || !B || !C || Bsz < 0 || D < 0 || N < 0)
        return -1;
    int64_t count = chains ? nchains : Bsz * D;
    for (int64_t i = 0; i < count; ++i) {
        int64_t c = chains ? chains[i] : i;
        if (c < 0 || c >= Bsz * D)
            return -1;
        int64_t b = c / D, d = c % D;
        double *h = state + (chains ? i : c) * N;
        double dl = (double)delta[b * D + d];
        double xv = (double)x[b * D + d];
        double acc = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            double dA = exp(dl * (double)A[d * N + n]);
            double dB = dl * (double)B[b * N + n];
            if (zoh)
                dB *= zoh_factor(dl * (double)A[d * N + n]);
            h[n] = dA * h[n] + dB * xv;
        }
        for (int64_t n = 0; n < N; ++n)
            acc += h[n] * (double)C[b * N + n];
        if (y)
            y[i] = gate(acc, Dskip, z, d, b * D + d, xv);
    }
    return 0;
}

/* ---- the causal depthwise convolution before the scan ------------------
 * youngju.dev "Mamba: Selective State Space Models", section 3.4, the
 * MambaBlock listing: a Conv1d over the sequence with one filter of d_conv
 * taps per channel (groups = channels), padded by d_conv - 1 in front and cut
 * back to L outputs, then SiLU:
 *   out[b,t,d] = silu(bias[d] + sum_{k<K} w[d,k] * x[b, t-K+1+k, d])
 * Inputs before t = 0 come from state_in (Bsz, D, K-1), the previous K-1
 * inputs of each channel, oldest first (zeros when NULL); state_out
 * receives the last K-1 inputs in the same layout. bias may be NULL
 * (zero); silu = 0 leaves the sum as it is. out: (Bsz, L, D) double.
 * The decode step is the same with L = 1 and the state updated in place. */
int oracle_conv1d(const float *x, const float *w, const float *bias,
                  const float *state_in, double *out, float *state_out,
                  int64_t Bsz, int64_t L, int64_t D, int64_t K, int silu)
{
    if (Bsz < 0 || L < 0 || D < 0 || K < 1 || (L > 0 && !x) || !w)
        return -1;
    for (int64_t b = 0; b < Bsz; ++b) {
        for (int64_t d = 0; d < D; ++d) {
            /* the value of x at time tau (tau < 0: from the carried state) */
            for (int64_t t = 0; t < L; ++t) {
                double acc = bias ? (double)bias[d] : 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    int64_t tau = t - (K - 1) + k;
                    double v;
                    if (tau >= 0)
                        v = (double)x[(b * L + tau) * D + d];
                    else
                        v = state_in ? (double)state_in[(b * D + d) * (K - 1) + (K - 1 + tau)] : 0.0;
                    acc += (double)w[d * K + k] * v;
                }
                if (silu)
                    acc = acc / (1.0 + exp(-acc));
                if (out)
                    out[(b * L + t) * D + d] = acc;
            }
            if (state_out) {
                for (int64_t j = 0; j < K - 1; ++j) {
                    int64_t tau = L - (K - 1) + j;   /* the last K-1 inputs, oldest first */
                    float v;
                    if (tau >= 0)
                        v = x[(b * L + tau) * D + d];
                    else
                        v = state_in ? state_in[(b * D + d) * (K - 1) + (K - 1 + tau)] : 0.0f;
                    state_out[(b * D + d) * (K - 1) + j] = v;
                }
            }
        }
    }
    return 0;
}

/* ---- backward pass of the scan --------------------------------------------
 * Gradients of a scalar loss through the forward scan above (dl * B form,
 * optional softplus), given the loss's gradients gy (Bsz, L, D) with respect
 * to y and, optionally, ghT (Bsz, D, N) with respect to hT. The pages give
 * the backward pass only as part of the hardware-aware design, whose states
 * are recomputed rather than stored (booiljung.github.io "3.1 LTI ...
 * Input-Dependent parameters", section 3.1.5.3); they print no gradient
 * formulas, so these are the chain rule applied to the recurrence. This is
 * the plain reverse sweep, keeping each chain's states:
 *   forward   h_t = a_t h_{t-1} + b_t,  a_t = exp(dl_t A),  b_t = dl_t B_t x_t,
 *             y_t = sum_n h_t C_t
 *   backward  g_t = gy_t C_t + a_{t+1} g_{t+1}   (g_{L-1} also takes ghT)
 *             dC_t += gy_t h_t,  da_t = g_t h_{t-1},  db_t = g_t
 *             d dl_t = sum_n (da_t a_t A + db_t B_t x_t),  dA += da_t a_t dl_t,
 *             dB_t += db_t dl_t x_t,  dx_t = sum_n db_t dl_t B_t,
 *             d delta_t = d dl_t * sigmoid(delta_t) when softplus is applied,
 *             dh0 = a_0 g_0.
 * Outputs (all double, zeroed here): dx, ddelta (Bsz, L, D); dA (D, N);
 * dB, dC (Bsz, L, N); dh0 (Bsz, D, N) or NULL. Single-threaded. */
int oracle_selscan_bwd(const float *x, const float *delta, const float *A,
                       const float *B, const float *C, const double *h0,
                       const double *gy, const double *ghT,
                       double *dx, double *ddelta, double *dA, double *dB,
                       double *dC, double *dh0, int64_t Bsz, int64_t L,
                       int64_t D, int64_t N, int delta_softplus)
{
    if (Bsz < 0 || L < 0 || D < 0 || N < 1 || !A || !gy || !dx || !ddelta || !dA || !dB || !dC)
        return -1;
    if (L > 0 && (!x || !delta || !B || !C))
        return -1;
    memset(dx, 0, sizeof(double) * (size_t)(Bsz * L * D));
    memset(ddelta, 0, sizeof(double) * (size_t)(Bsz * L * D));
    memset(dA, 0, sizeof(double) * (size_t)(D * N));
    memset(dB, 0, sizeof(double) * (size_t)(Bsz * L * N));
    memset(dC, 0, sizeof(double) * (size_t)(Bsz * L * N));
    if (dh0)
        memset(dh0, 0, sizeof(double) * (size_t)(Bsz * D * N));
    /* hs[(t + 1) * N + n] = h after step t; hs[n] = the initial state */
    double *hs = (double *)malloc(sizeof(double) * (size_t)((L + 1) * N));
    double *g = (double *)malloc(sizeof(double) * (size_t)N);
    double *dls = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
    if (!hs || !g || !dls) {
        free(hs); free(g); free(dls);
        return -1;
    }
    for (int64_t b = 0; b < Bsz; ++b) {
        for (int64_t d = 0; d < D; ++d) {
            for (int64_t n = 0; n < N; ++n)
                hs[n] = h0 ? h0[(b * D + d) * N + n] : 0.0;
            for (int64_t t = 0; t < L; ++t) {   /* forward, keeping the states */
                int64_t bt = b * L + t;
                double dl = (double)delta[bt * D + d];
                if (delta_softplus)
                    dl = oracle_softplus(dl);
                dls[t] = dl;
                double xv = (double)x[bt * D + d];
                for (int64_t n = 0; n < N; ++n)
                    hs[(t + 1) * N + n] = exp(dl * (double)A[d * N + n]) * hs[t * N + n]
                                          + dl * (double)B[bt * N + n] * xv;
            }
            for (int64_t n = 0; n < N; ++n)
                g[n] = ghT ? ghT[(b * D + d) * N + n] : 0.0;
            for (int64_t t = L - 1; t >= 0; --t) {   /* reverse sweep */
                int64_t bt = b * L + t;
                double dl = dls[t];
                double xv = (double)x[bt * D + d];
                double gyv = gy[bt * D + d];
                double gdl = 0.0, gx = 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    double an = (double)A[d * N + n];
                    double a = exp(dl * an);
                    double Bn = (double)B[bt * N + n];
                    g[n] += gyv * (double)C[bt * N + n];           /* y_t reads h_t */
                    dC[bt * N + n] += gyv * hs[(t + 1) * N + n];
                    double da = g[n] * hs[t * N + n];
                    gdl += da * a * an + g[n] * Bn * xv;
                    dA[d * N + n] += da * a * dl;
                    dB[bt * N + n] += g[n] * dl * xv;
                    gx += g[n] * dl * Bn;
                    g[n] *= a;                                      /* into h_{t-1} */
                }
                dx[bt * D + d] = gx;
                if (delta_softplus) {
                    double u = (double)delta[bt * D + d];
                    gdl *= 1.0 / (1.0 + exp(-u));                   /* softplus' = sigmoid */
                }
                ddelta[bt * D + d] = gdl;
            }
            if (dh0)
                for (int64_t n = 0; n < N; ++n)
                    dh0[(b * D + d) * N + n] = g[n];
        }
    }
    free(hs); free(g); free(dls);
    return 0;
}

/* ---- Mamba-2 SSD -------------------------------------------------------
 * The state-space-dual model of youngju.dev "Mamba: Selective State Space
 * Models", section 4.1 (recurrence h_t = A_t h_{t-1} + B_t x_t, y_t = C_t h_t)
 * with the multi-head layout of section 5.2 (heads of headdim P, state size
 * N). A_t is a scalar per head, exp(dt * A[hd]) (the structured form whose
 * dual matrix M is semiseparable), and the input term takes dt * B as in the
 * simplified selective_scan listing of section 3.3. B and C are shared by
 * all heads.
 *
 *   x : (Bsz, L, H, P)   dt : (Bsz, L, H)   A : (H)   B, C : (Bsz, L, N)
 *   h0, hT : (Bsz, H, N, P) double (h0 NULL: zeros)   y : (Bsz, L, H, P) double
 *   for every batch b and head hd, from h[n][p] = h0:
 *     for t: dl = dt[b,t,hd] (softplus(dl) when asked), a = exp(dl * A[hd])
 *            h[n][p] = a * h[n][p] + (dl * B[b,t,n]) * x[b,t,hd,p]
 *            y[b,t,hd,p] = sum_n C[b,t,n] * h[n][p]
 * Single-threaded. */
int oracle_ssd_fwd(const float *x, const float *dt, const float *A, const float *B,
                   const float *C, const double *h0, double *y, double *hT,
                   int64_t Bsz, int64_t L, int64_t H, int64_t P, int64_t N,
                   int dt_softplus)
{
    if (Bsz < 0 || L < 0 || H < 0 || P < 1 || N < 1 || !y || !hT || (H > 0 && !A))
        return -1;
    if (L > 0 && (!x || !dt || !B || !C))
        return -1;
    double *h = (double *)malloc(sizeof(double) * (size_t)(N * P));
    if (!h)
        return -1;
    for (int64_t b = 0; b < Bsz; ++b) {
        for (int64_t hd = 0; hd < H; ++hd) {
            const int64_t s0 = (b * H + hd) * N * P;
            for (int64_t i = 0; i < N * P; ++i)
                h[i] = h0 ? h0[s0 + i] : 0.0;
            for (int64_t t = 0; t < L; ++t) {
                const int64_t bt = b * L + t;
                double dl = (double)dt[bt * H + hd];
                if (dt_softplus)
                    dl = oracle_softplus(dl);
                const double a = exp(dl * (double)A[hd]);
                const float *xv = x + (bt * H + hd) * P;
                for (int64_t n = 0; n < N; ++n) {
                    const double db = dl * (double)B[bt * N + n];
                    for (int64_t p = 0; p < P; ++p)
                        h[n * P + p] = a * h[n * P + p] + db * (double)xv[p];
                }
                double *yv = y + (bt * H + hd) * P;
                for (int64_t p = 0; p < P; ++p) {
                    double acc = 0.0;
                    for (int64_t n = 0; n < N; ++n)
                        acc += (double)C[bt * N + n] * h[n * P + p];
                    yv[p] = acc;
                }
            }
            for (int64_t i = 0; i < N * P; ++i)
                hT[s0 + i] = h[i];
        }
    }
    free(h);
    return 0;
}

/* Backward of the block's output around the scan (youngju.dev "Mamba:
 * Selective State Space Models", section 3.4, the MambaBlock listing):
 * out = (y + Dskip[d] x) * silu(z) with y the scan's read-out, given dout =
 * dLoss/dout (Bsz, L, D) and dLoss/dhT. With s = sigmoid(z), silu(z) = z s
 * and silu'(z) = s (1 + z (1 - s)):
 *   the scan's backward (oracle_selscan_bwd) takes gy = dout * silu(z);
 *   dz      = dout * (y + Dskip x) * silu'(z)            (Bsz, L, D)
 *   dDskip  = sum_{b,t} dout * silu(z) * x               (D)
 *   dx     += dout * silu(z) * Dskip.
 * Either term may be absent (Dskip NULL: no skip, dDskip untouched; z NULL:
 * no gate, dz untouched). Outputs as oracle_selscan_bwd, plus dDskip and dz
 * (double, zeroed here when their term is present). */
int oracle_selscan_bwd_gated(const float *x, const float *delta, const float *A,
                             const float *B, const float *C, const float *Dskip,
                             const float *z, const double *h0, const double *dout,
                             const double *ghT, double *dx, double *ddelta, double *dA,
                             double *dB, double *dC, double *dh0, double *dDskip, double *dz,
                             int64_t Bsz, int64_t L, int64_t D, int64_t N, int delta_softplus)
{
    if (Bsz < 0 || L < 0 || D < 0 || N < 1 || !dout || (Dskip && !dDskip) || (z && !dz))
        return -1;
    const size_t E = (size_t)(Bsz * L * D);
    double *y = (double *)malloc(sizeof(double) * (E > 0 ? E : 1));
    double *gy = (double *)malloc(sizeof(double) * (E > 0 ? E : 1));
    if (!y || !gy) {
        free(y); free(gy);
        return -1;
    }
    int rc = oracle_selscan_fwd_gated(x, delta, A, B, C, NULL, NULL, h0, y, NULL, Bsz, L, D, N,
                                      delta_softplus, 0, 1);
    if (rc == 0) {
        for (size_t i = 0; i < E; ++i) {
            double g = dout[i];
            if (z) {
                const double zv = (double)z[i];
                g *= zv / (1.0 + exp(-zv));
            }
            gy[i] = g;
        }
        rc = oracle_selscan_bwd(x, delta, A, B, C, h0, gy, ghT, dx, ddelta, dA, dB, dC, dh0,
                                Bsz, L, D, N, delta_softplus);
    }
    if (rc == 0) {
        if (Dskip)
            memset(dDskip, 0, sizeof(double) * (size_t)D);
        for (size_t i = 0; i < E; ++i) {
            const int64_t d = (int64_t)(i % (size_t)D);
            const double xv = (double)x[i];
            if (Dskip) {
                dDskip[d] += gy[i] * xv;
                dx[i] += gy[i] * (double)Dskip[d];
            }
            if (z) {
                const double zv = (double)z[i];
                const double s = 1.0 / (1.0 + exp(-zv));
                const double pre = y[i] + (Dskip ? (double)Dskip[d] * xv : 0.0);
                dz[i] = dout[i] * pre * s * (1.0 + zv * (1.0 - s));
            }
        }
    }
    free(y); free(gy);
    return rc;
}
