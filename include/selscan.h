/*
 * selscan.h -- C ABI of libselscan, Mamba's selective scan on one NVIDIA
 * B300 (sm_103a).
 *
 * The operation (youngju.dev, "Mamba: Selective State Space Models",
 * section 3.3, the simplified selective_scan listing; the recurrence of
 * section 2.2; the (B, L, D) / (B, L, N) shapes of booiljung.github.io
 * "3.1 LTI systems and input-dependent parameters", section 0.4.2):
 *
 *   for every batch b and channel d, starting from h[n] = h0[b,d,n] (or 0):
 *     for t = 0 .. L-1:
 *       dl = delta[b,t,d], or softplus(dl) = log(1 + e^dl) when delta_softplus
 *       h[n] = exp(dl * A[d,n]) * h[n] + (dl * B[b,t,n]) * x[b,t,d]   (n < N)
 *       y[b,t,d] = sum_n h[n] * C[b,t,n]
 *     hT[b,d,n] = h[n]
 *
 * deltaB is the simplified dl * B of that listing; selscan_fwd_ex offers
 * the zero-order-hold form of section 2.2 instead, and selscan_fwd_gated /
 * selscan_fwd_ex the block's skip and gate around the scan (section 3.4).
 * The hidden state h never goes to device memory:
 * it lives in registers; long sequences are cut into chunks whose carries
 * are composed as associative (decay, offset) pairs (booiljung.github.io
 * section 3.1.5.2, the parallel scan).
 *
 * Conventions shared by every entry point
 *  - Every tensor argument is a DEVICE pointer (memory the current CUDA
 *    device can read), except in selscan_fwd_host, whose tensors are all in
 *    host memory; always row-major and contiguous, last axis fastest. The
 *    caller owns all of them; the library keeps no pointer after a call
 *    returns.
 *  - dtype selects the element type of x, delta, B, C and y:
 *    SELSCAN_F32 (IEEE fp32) or SELSCAN_BF16 (bfloat16). A, h0, hT and the
 *    decode state are always fp32; all arithmetic is fp32. bf16 outputs are
 *    rounded to nearest even.
 *  - stream is a cudaStream_t (NULL = the legacy default stream). Work is
 *    enqueued on it and the call returns without waiting: results are ready
 *    once the stream reaches that point. Faults inside kernels surface, as
 *    with any CUDA library, at the caller's next synchronisation (see
 *    selscan_check_device_error).
 *  - Return value: SELSCAN_OK (0) or a selscan_status code. Argument checks
 *    run before any CUDA call: on SELSCAN_ERR_INVALID_ARG or
 *    SELSCAN_ERR_UNSUPPORTED nothing was launched and no output was
 *    touched. selscan_last_error() then describes the failure.
 *  - Thread safety: calls may be made concurrently from several host
 *    threads on different streams. A kernel that gives up waiting records
 *    the failure in a fault word of the stream it ran on, and only
 *    selscan_check_device_error on that stream reports it (up to 64
 *    streams per device have words of their own; beyond that, streams
 *    share one).
 */
#ifndef SELSCAN_H
#define SELSCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SELSCAN_F32 = 0,
    SELSCAN_BF16 = 1
} selscan_dtype;

typedef enum {
    SELSCAN_OK = 0,
    SELSCAN_ERR_INVALID_ARG = 1,  /* null pointer, negative size, bad dtype, overlapping buffers */
    SELSCAN_ERR_UNSUPPORTED = 2,  /* valid request the library does not implement (N > 64) */
    SELSCAN_ERR_CUDA = 3,         /* a CUDA runtime call or kernel launch failed */
    SELSCAN_ERR_NO_MEMORY = 4,    /* the chunk-carry workspace could not be allocated */
    SELSCAN_ERR_TIMEOUT = 5       /* a kernel gave up waiting for an input tile or a chunk carry
                                     (reported by selscan_check_device_error; the kernel's outputs
                                     are invalid) */
} selscan_status;

/* Largest state size N the kernels implement. */
#define SELSCAN_MAX_N 64

/* Flags of selscan_fwd_ex and selscan_step_ex. */
#define SELSCAN_FLAG_SOFTPLUS 1   /* delta is the pre-activation: dl = softplus(delta) */
#define SELSCAN_FLAG_ZOH 2        /* zero-order-hold Bbar instead of dl * B (see selscan_fwd_ex) */

/*
 * selscan_fwd -- the forward selective scan over a whole sequence.
 * (youngju.dev "Mamba: Selective State Space Models", section 3.3;
 *  softplus from booiljung.github.io section 0.4.2.)
 *
 *   x, delta : (Bsz, L, D), dtype        delta is the step size, or its raw
 *                                        pre-activation when delta_softplus != 0
 *   A        : (D, N) fp32               the diagonal state matrix per channel
 *   B, C     : (Bsz, L, N), dtype        input / output matrices per token
 *   y        : (Bsz, L, D), dtype        written
 *   h0       : (Bsz, D, N) fp32 or NULL  initial state (NULL = zeros)
 *   hT       : (Bsz, D, N) fp32 or NULL  final state, written when non-NULL
 *
 * Sizes: Bsz >= 0, L >= 0, D >= 0, 1 <= N <= SELSCAN_MAX_N. Bsz == 0 or
 * D == 0 is an empty problem (OK, nothing written). L == 0 writes only hT
 * (= h0, or zeros). x, delta, B, C and y must be non-NULL when L > 0 and
 * Bsz * D > 0; A must be non-NULL when Bsz * D > 0.
 *
 * Aliasing: y may equal x or delta exactly (in-place output); h0 may equal
 * hT exactly (resume in place). Any other overlap between y or hT and
 * another argument is SELSCAN_ERR_INVALID_ARG. When the sequence is cut
 * into chunks, output in place over delta takes the plain-load kernels
 * (whose chunk reductions finish before any output is written; the fused
 * kernel's correction pass reads delta after the first pass wrote y), and
 * in-place resume writes the final state to the workspace first and copies
 * it to hT after the scan.
 *
 * Memory: chunked plans use a library-owned workspace: the chunk carries
 * (ceil(L / chunk) * Bsz * D * (N + 1) fp32), a ticket and two flags per
 * channel group, with bf16 output on the fused path the bf16 rounding
 * residual of the first pass (Bsz * L * D bf16), and Bsz * D * N fp32 for
 * in-place resume. selscan_fwd_plan reports its size. It is taken from a
 * private stream-ordered pool on `stream` and returned to it before the
 * call's work completes; selscan_release_workspace() gives the pool's
 * memory back to the device. SELSCAN_ERR_NO_MEMORY if it cannot be had.
 */
int selscan_fwd(const void *x, const void *delta, const float *A, const void *B,
                const void *C, void *y, int64_t Bsz, int64_t L, int64_t D,
                int64_t N, int dtype, int delta_softplus, const float *h0,
                float *hT, void *stream);

/*
 * selscan_fwd_gated -- selscan_fwd with the block's output around the scan
 * fused into the read-out (youngju.dev "Mamba: Selective State Space
 * Models", section 3.4, the MambaBlock listing):
 *
 *   y[b,t,d] = (sum_n h[n] * C[b,t,n] + Dskip[d] * x[b,t,d]) * silu(z[b,t,d])
 *   silu(z)  = z / (1 + e^-z)
 *
 *   Dskip : (D) fp32 or NULL    the per-channel skip parameter (D in the
 *                               listing); NULL = no skip term
 *   z     : (Bsz, L, D), dtype  the gate input; NULL = no gate
 *
 * The listing shows the gate and defines the skip parameter but elides where
 * it is applied; the skip is added before the gate. The final state hT does
 * not see either term. Everything else (shapes, sizes, aliasing, memory,
 * errors) is as for selscan_fwd; y may also equal z exactly, and neither
 * may partially overlap y or hT. With both NULL this is selscan_fwd.
 * The fused kernel applies them in its read-out when the rows are 16-byte
 * aligned and delta_softplus is set; other cases take the plain-load
 * kernels, with the same results.
 */
int selscan_fwd_gated(const void *x, const void *delta, const float *A, const void *B,
                      const void *C, const float *Dskip, const void *z, void *y,
                      int64_t Bsz, int64_t L, int64_t D, int64_t N, int dtype,
                      int delta_softplus, const float *h0, float *hT, void *stream);

/*
 * selscan_fwd_ex -- selscan_fwd_gated with a flags word in place of
 * delta_softplus: SELSCAN_FLAG_SOFTPLUS as delta_softplus != 0, and
 * SELSCAN_FLAG_ZOH for the zero-order-hold discretisation of youngju.dev
 * section 2.2, Bbar = (dl A)^-1 (exp(dl A) - I) dl B, which for the diagonal
 * A is, per state,
 *
 *   Bbar[n] = dl * B[n] * phi(dl * A[d,n]),   phi(w) = (e^w - 1) / w,  phi(0) = 1
 *
 * in place of the simplified dl * B[n] (the decay exp(dl A) is the same).
 * phi is evaluated from the decay, or from its series where |w| < 1/16, so
 * A == 0 gives the limit dl * B. The zero-order-hold form runs in the
 * fused TMA kernel for N <= 16 with 16-byte rows and SELSCAN_FLAG_SOFTPLUS
 * set, and on the plain-load kernels otherwise. Unknown flag bits are
 * SELSCAN_ERR_INVALID_ARG.
 */
int selscan_fwd_ex(const void *x, const void *delta, const float *A, const void *B,
                   const void *C, const float *Dskip, const void *z, void *y,
                   int64_t Bsz, int64_t L, int64_t D, int64_t N, int dtype, int flags,
                   const float *h0, float *hT, void *stream);

/*
 * selscan_step -- one decode step of the recurrent mode, O(1) state per
 * token (youngju.dev section 6: inference O(1) per token with a fixed
 * state; the same update as selscan_fwd with L = 1).
 *
 *   state : (Bsz, D, N) fp32, read and updated in place
 *   x     : (Bsz, D) fp32      delta : (Bsz, D) fp32, used as given (already
 *                                      positive; no softplus is applied)
 *   A     : (D, N) fp32        B, C  : (Bsz, N) fp32
 *   y     : (Bsz, D) fp32, written:  y[b,d] = sum_n state'[b,d,n] * C[b,n]
 *   where state'[b,d,n] = exp(delta[b,d] * A[d,n]) * state[b,d,n]
 *                         + delta[b,d] * B[b,n] * x[b,d]
 *
 * Sizes as for selscan_fwd (Bsz, D >= 0; 1 <= N <= SELSCAN_MAX_N). y must
 * not overlap state or any input; state must not overlap an input.
 */
int selscan_step(float *state, const float *x, const float *delta, const float *A,
                 const float *B, const float *C, float *y, int64_t Bsz, int64_t D,
                 int64_t N, void *stream);

/* selscan_step with the block's skip and gate on the step's output, as in
 * selscan_fwd_gated: y = (sum_n state'[n] * C[n] + Dskip[d] * x) * silu(z).
 * Dskip (D) and z (Bsz, D) are fp32 device pointers or NULL; the state does
 * not see either term. Neither may overlap y or state. */
int selscan_step_gated(float *state, const float *x, const float *delta, const float *A,
                       const float *B, const float *C, const float *Dskip, const float *z,
                       float *y, int64_t Bsz, int64_t D, int64_t N, void *stream);

/* selscan_step_gated with a flags word: SELSCAN_FLAG_ZOH selects the
 * zero-order-hold Bbar as in selscan_fwd_ex (the step takes no softplus;
 * any other bit is SELSCAN_ERR_INVALID_ARG). */
int selscan_step_ex(float *state, const float *x, const float *delta, const float *A,
                    const float *B, const float *C, const float *Dskip, const float *z,
                    float *y, int64_t Bsz, int64_t D, int64_t N, int flags, void *stream);

/*
 * selscan_fwd_noalloc -- selscan_fwd for callers that cannot allocate device
 * memory. The pages describe no counterpart: this is a deployment variant of
 * selscan_fwd, not part of the method.
 *
 * Who needs it: code that runs where another allocator owns every byte of
 * device memory (a framework's caching allocator, or a server that reserves
 * the whole GPU at start-up, so cudaMalloc would fail or fragment its pool);
 * code on a latency budget that cannot afford cudaMalloc/cudaFree, which can
 * synchronise the device and take milliseconds; and plugins whose host
 * program forbids them to allocate. selscan_fwd takes a small workspace from
 * a pool for long sequences; this entry point takes it from a fixed array
 * compiled into the library instead, and makes no allocation of any kind.
 *
 * Arguments, results, alias rules and error codes are those of selscan_fwd,
 * and it splits the work the same way. The scratch array holds
 * SELSCAN_NOALLOC_SCRATCH_BYTES (8 MiB); every GPU that loads the library
 * holds it until the process exits. A call whose plan needs more scratch
 * (the workspace_bytes that selscan_fwd_plan reports: see selscan_fwd's
 * "Memory"; chunked bf16 plans include Bsz * L * D * 2 bytes for the
 * rounding residual) returns SELSCAN_ERR_UNSUPPORTED
 * before anything is launched; run such a problem through selscan_fwd, or in
 * pieces along L, handing hT of one piece to h0 of the next.
 *
 * The first call on each device looks up the array's device address; make
 * that first call before any stream capture. Every call on a device shares
 * the one array, and it keeps whatever the last call left in it: calls that
 * can overlap on the GPU (on streams not ordered with each other) race on it
 * and produce wrong results, so order them on one stream or synchronise
 * between them. Nothing in the array has to start at zero: each call writes
 * every scratch element before it reads it.
 */
#define SELSCAN_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)

int selscan_fwd_noalloc(const void *x, const void *delta, const float *A, const void *B,
                        const void *C, void *y, int64_t Bsz, int64_t L, int64_t D,
                        int64_t N, int dtype, int delta_softplus, const float *h0,
                        float *hT, void *stream);

/*
 * selscan_fwd_plan -- how selscan_fwd would run a problem of this size on
 * the current device, without running it (for tests and benchmarks).
 *   chunks          : number of chunks the sequence is cut into (1 = one pass)
 *   chunk_len       : timesteps per chunk
 *   launches        : kernels one selscan_fwd call enqueues
 *   workspace_bytes : chunk-carry workspace the call uses (0 for one chunk)
 * Any output pointer may be NULL. The figures assume 16-byte aligned
 * tensors (alignment decides between the TMA-staged and the plain
 * kernels). Same size checks as selscan_fwd; needs a CUDA device (it reads
 * the SM count). The plan depends only on the sizes,
 * dtype and device, plus the tuning variables SELSCAN_CHUNK and
 * SELSCAN_TARGET_WARPS when set.
 */
int selscan_fwd_plan(int64_t Bsz, int64_t L, int64_t D, int64_t N, int dtype,
                     int *chunks, int64_t *chunk_len, int *launches,
                     int64_t *workspace_bytes);

/*
 * selscan_fwd_host -- selscan_fwd with every tensor in HOST memory.
 * (No counterpart on the pages: this is the library's host-to-device path.)
 *
 * Same arguments, shapes, sizes, aliasing rules and results as selscan_fwd,
 * except that x, delta, A, B, C, y, h0 and hT are host pointers. They need
 * not be page-locked, but only page-locked (pinned) buffers let the copies
 * run asynchronously and overlap the scan.
 *
 * The sequence is cut into pieces along L (about 32 MB of input each, and at
 * least two when L >= 128). Inputs go in on two copy streams. While
 * piece p is scanned on the current device, piece p+1's inputs are copied
 * in and piece p-1's output is copied out, on library-owned streams;
 * each piece starts from the device-resident final state of the one before,
 * so the pieces compose exactly like the chunks of one call. Device staging
 * (two pieces' inputs and outputs, A and the state) comes from the same
 * stream-ordered pool as the chunk workspace.
 *
 * Blocking: returns once y (and hT) are in host memory. Work already
 * enqueued on `stream` is waited for first. Calls on one device are
 * serialised by the library; calls on different devices may run together.
 */
int selscan_fwd_host(const void *x, const void *delta, const float *A, const void *B,
                     const void *C, void *y, int64_t Bsz, int64_t L, int64_t D, int64_t N,
                     int dtype, int delta_softplus, const float *h0, float *hT, void *stream);

/*
 * selscan_fwd_host_ex -- selscan_fwd_ex (the block's skip and gate, the
 * flags word) with every tensor in HOST memory, pipelined like
 * selscan_fwd_host. Dskip (D fp32) and z (Bsz, L, D, like x) are host
 * pointers or NULL, as in selscan_fwd_ex; z travels with the other
 * per-step inputs of each piece. Arguments, aliasing rules, blocking and
 * errors as for selscan_fwd_ex and selscan_fwd_host.
 */
int selscan_fwd_host_ex(const void *x, const void *delta, const float *A, const void *B,
                        const void *C, const float *Dskip, const void *z, void *y, int64_t Bsz,
                        int64_t L, int64_t D, int64_t N, int dtype, int flags, const float *h0,
                        float *hT, void *stream);

/*
 * selscan_conv1d -- the causal depthwise convolution and SiLU in front of
 * the scan (youngju.dev "Mamba: Selective State Space Models", section 3.4,
 * the MambaBlock listing: Conv1d with one filter of K taps per channel,
 * padded by K - 1 in front and cut back to L outputs, then SiLU):
 *
 *   out[b,t,d] = silu(bias[d] + sum_{k<K} w[d,k] * x[b, t-K+1+k, d])
 *
 *   x, out    : (Bsz, L, D), dtype     w : (D, K) fp32    bias : (D) fp32 or NULL
 *   state_in  : (Bsz, D, K-1) fp32 or NULL   the K-1 inputs before t = 0 of
 *               every channel, oldest first (NULL = zeros: a fresh sequence)
 *   state_out : (Bsz, D, K-1) fp32 or NULL   receives the last K-1 inputs, for
 *               the next piece of the sequence or for selscan_conv1d_step
 *   silu      : 0 leaves the sum without the SiLU
 *
 * Sizes: Bsz, L, D >= 0 (Bsz <= 65535, L <= 65535 * 64); 1 <= K <= 8
 * (K = 1 carries no state). out must not overlap any input; state_out must
 * not overlap out or any input (state_in included: pass another buffer).
 * L == 0 copies state_in (or zeros) to state_out. Errors as for selscan_fwd.
 * Bound by HBM bandwidth: x is read once and out written once.
 */
int selscan_conv1d(const void *x, const float *w, const float *bias, void *out, int64_t Bsz,
                   int64_t L, int64_t D, int64_t K, int dtype, int silu, const float *state_in,
                   float *state_out, void *stream);

/* One decode step of selscan_conv1d, fp32: out (Bsz, D) from the carried
 * conv_state (Bsz, D, K-1, oldest first) and this token's x (Bsz, D); the
 * state then shifts by one and takes x, in place. conv_state may be NULL
 * when K == 1. out must not overlap conv_state or an input. */
int selscan_conv1d_step(float *conv_state, const float *x, const float *w, const float *bias,
                        float *out, int64_t Bsz, int64_t D, int64_t K, int silu, void *stream);

/*
 * selscan_bwd -- the backward pass of selscan_fwd (fp32, dl * B form, no
 * skip or gate): the gradients of a scalar loss with respect to every input,
 * given its gradients with respect to y and hT. The hardware-aware design of
 * booiljung.github.io "3.1 LTI systems and input-dependent parameters",
 * section 3.1.5.3, recomputes the states in the backward pass instead of
 * storing them; so does this call. With g_t = dLoss/dh_t, carried backwards
 * as g_t = gy_t C_t + exp(dl_{t+1} A) g_{t+1} from g_{L-1} = gy C + dhT:
 *
 *   dC[b,t,n]  = sum_d gy[b,t,d] h_t[n]     dB[b,t,n] = sum_d g_t[n] dl x[b,t,d]
 *   dx[b,t,d]  = sum_n g_t[n] dl B[b,t,n]   dA[d,n]   = sum_{b,t} g_t h_{t-1} a_t dl
 *   ddelta[b,t,d] = sum_n (g_t h_{t-1} a_t A[d,n] + g_t B x), times
 *                   sigmoid(delta) when delta_softplus (d softplus / du)
 *   dh0[b,d,n] = exp(dl_0 A) g_0
 *
 *   x, delta, dy, dx, ddelta : (Bsz, L, D) fp32   A, dA : (D, N) fp32
 *   B, C, dB, dC             : (Bsz, L, N) fp32
 *   h0, dhT, dh0             : (Bsz, D, N) fp32 or NULL (h0 NULL = zeros,
 *                              dhT NULL = no loss on hT, dh0 NULL = not wanted)
 *
 * Sizes: Bsz, L, D >= 0 with Bsz <= 65535; 1 <= N <= 32. Every output is
 * overwritten; no output may overlap an input or another output. Pointers
 * 4-byte aligned. L == 0 gives dA = 0 and dh0 = dhT (or zeros).
 * Workspace, from the same stream-ordered pool as selscan_fwd's: the local
 * state and the running sum of dl at the start of every 16-step chunk,
 * Bsz * ceil(L / 16) * D * (Np + 1) floats with Np the smallest of 4, 8, 16
 * and 32 that is >= N; and per segment (L is cut into K segments of whole
 * chunks, K at most the number of blocks that fill the GPU once) two
 * Bsz * K * D * Np arrays and one of Bsz * K * D floats.
 * dA, dB and dC are sums formed with atomic additions, so their last bits
 * may differ from run to run; dx, ddelta and dh0 are reproducible.
 * Errors as for selscan_fwd.
 */
int selscan_bwd(const float *x, const float *delta, const float *A, const float *B,
                const float *C, const float *h0, const float *dy, const float *dhT,
                float *dx, float *ddelta, float *dA, float *dB, float *dC, float *dh0,
                int64_t Bsz, int64_t L, int64_t D, int64_t N, int delta_softplus,
                void *stream);

/*
 * selscan_bwd_gated -- selscan_bwd for the block's output with its skip and
 * gate (the MambaBlock listing of youngju.dev "Mamba: Selective State Space
 * Models", section 3.4: y = (scan + Dskip * x) * silu(z), as selscan_fwd_gated
 * computes it), dy being dLoss/dy of that output. With s the scan's read-out
 * and silu'(z) = sigmoid(z) (1 + z (1 - sigmoid(z))):
 *
 *   the scan's upstream gradient  gs = dy * silu(z)   (dy without a gate)
 *   dz[b,t,d]  = dy (s + Dskip x) silu'(z)
 *   dDskip[d]  = sum_{b,t} gs x                dx += gs Dskip
 *
 * and every other gradient as selscan_bwd with gs in place of dy.
 *
 *   Dskip, dDskip : (D) fp32, both or neither     z, dz : (Bsz, L, D) fp32, both or neither
 *
 * Everything else as selscan_bwd (with both NULL it is selscan_bwd). dDskip
 * is a sum formed with atomic additions, like dA; dz is reproducible.
 */
int selscan_bwd_gated(const float *x, const float *delta, const float *A, const float *B,
                      const float *C, const float *Dskip, const float *z, const float *h0,
                      const float *dy, const float *dhT, float *dx, float *ddelta, float *dA,
                      float *dB, float *dC, float *dDskip, float *dz, float *dh0, int64_t Bsz,
                      int64_t L, int64_t D, int64_t N, int delta_softplus, void *stream);

/*
 * selscan_ssd_fwd -- the Mamba-2 state space duality (SSD) forward
 * (youngju.dev "Mamba: Selective State Space Models", section 4.1: the
 * recurrence h_t = A_t h_{t-1} + B_t x_t, y_t = C_t h_t and its dual form
 * Y = (T o M) X; section 5.2: heads of headdim P with a state of size N).
 * Per batch row b and head hd, with dl = dt[b,t,hd] (softplus(dt) when
 * dt_softplus), a scalar decay per step and B, C shared by all heads:
 *
 *   h[n][p] = exp(dl * A[hd]) * h[n][p] + (dl * B[b,t,n]) * x[b,t,hd,p]
 *   y[b,t,hd,p] = sum_n C[b,t,n] * h[n][p]
 *
 *   x, y  : (Bsz, L, H, P), dtype    dt : (Bsz, L, H) fp32    A : (H) fp32
 *   B, C  : (Bsz, L, N), dtype
 *   h0    : (Bsz, H, N, P) fp32 or NULL (zeros)
 *   hT    : (Bsz, H, N, P) fp32 or NULL (not written)
 *
 * Sizes: N = 64 or 128, P = 32, 64 or 128, Bsz and H at most 65535, any
 * L >= 0 (L == 0 writes only hT). The products run on the tensor cores
 * (tcgen05) with fp16 operands and fp32 accumulators, in chunks of 64 steps
 * (the dual form inside a chunk, the states carried across chunks), so
 * results agree with an exact evaluation to about 1e-3 relative for either
 * dtype. Pointers: x, B, C, y, h0 and hT 16-byte aligned, dt and A
 * 4-byte aligned. y and hT must not overlap any input or each other.
 * Workspace, from the same stream-ordered pool as selscan_fwd's, with
 * nch = ceil(L / 64): 4 * Bsz * H * nch * N * P bytes (each chunk's own state
 * and the state entering it, fp16), 2 * Bsz * nch * 64 * (64 + N) bytes
 * (C B^T and C of each chunk, fp16) and 4 * Bsz * H * nch bytes (the chunk
 * decays). Errors as for selscan_fwd.
 */
int selscan_ssd_fwd(const void *x, const float *dt, const float *A, const void *B,
                    const void *C, void *y, const float *h0, float *hT, int64_t Bsz,
                    int64_t L, int64_t H, int64_t P, int64_t N, int dtype, int dt_softplus,
                    void *stream);

/* Message describing the last non-OK status returned on this host thread
 * (empty string if none). The pointer stays valid until the next call on
 * the same thread. */
const char *selscan_last_error(void);

/* Waits for `stream` and reports whether work enqueued on it failed:
 * SELSCAN_OK; SELSCAN_ERR_CUDA with the CUDA error in selscan_last_error();
 * or SELSCAN_ERR_TIMEOUT when a kernel stopped waiting for an input tile
 * (fault code 1), for the carry of an earlier chunk (fault code 2) or for a
 * tensor-core product (fault code 3) that never came. Every wait inside the kernels is bounded (2 s of GPU time,
 * which keeps counting while the context is time-sliced out on a shared
 * GPU), so a broken pipeline ends with this status instead of a hang, and
 * the context stays usable. A call that timed out left its outputs
 * invalid. Each stream has its own fault word (see "Thread safety"); this
 * call reads and clears the word of `stream` only. */
int selscan_check_device_error(void *stream);

/* Test hook for the timeout path: makes a wait run out without any fault.
 * With withhold_carries = 1, later chunked forward calls in this process
 * never announce their composed chunk carries, so every correction pass of
 * a later chunk waits for a flag that nothing sets; wait_limit_ms (1..2000)
 * shortens that wait (0 = the default 2 s). Such calls end early with
 * invalid outputs, and selscan_check_device_error on their stream returns
 * SELSCAN_ERR_TIMEOUT (fault code 2). selscan_test_fault_injection(0, 0)
 * restores normal operation. Off by default; nothing in the environment can
 * turn it on. SELSCAN_ERR_INVALID_ARG for arguments out of range. */
int selscan_test_fault_injection(int withhold_carries, int wait_limit_ms);

/* Page-locked host memory for the host-buffer entry points: `bytes` rounded
 * up to 2 MB, 2 MB aligned, from an anonymous mapping (transparent huge
 * pages requested) registered with the CUDA driver for every device. On
 * the B300 hosts measured, copies from such buffers ran at 52-55 GB/s,
 * while buffers from cudaHostAlloc ran anywhere from 11 to 55 GB/s (and any
 * pinned buffer whose lines were still dirty in the CPU cache at 15-17
 * GB/s). Returns NULL on failure (selscan_last_error says why). Free with
 * selscan_host_free, which returns SELSCAN_ERR_INVALID_ARG for a pointer
 * this call did not return; NULL is ignored. Thread-safe. */
void *selscan_host_alloc(size_t bytes);
int selscan_host_free(void *ptr);

/* Returns the memory held by the chunk-carry workspace pools of every
 * device this process used to the device. Safe to call at any time; work
 * already enqueued keeps its memory until it completes. */
void selscan_release_workspace(void);

/* Library version string, e.g. "libselscan 0.1.0 (sm_103a)". */
const char *selscan_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SELSCAN_H */
