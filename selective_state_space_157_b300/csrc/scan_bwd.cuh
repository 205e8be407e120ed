// scan_bwd.cuh -- the backward pass of the selective scan (fp32).
//
// The hardware-aware design of booiljung.github.io "3.1 LTI systems and
// input-dependent parameters", section 3.1.5.3, trains through the scan by
// recomputing the states in the backward pass instead of storing them. The
// pages give no gradient formulas; these are the chain rule applied to the
// recurrence h_t = a_t h_{t-1} + dl_t B_t x_t, a_t = exp(dl_t A), y_t =
// sum_n h_t C_t. With g_t = dLoss/dh_t (the adjoint, carried backwards as
// g_t = gy_t C_t + a_{t+1} g_{t+1}, starting from dLoss/dhT):
//   dC_t += gy_t h_t                dB_t += g_t dl_t x_t
//   dx_t  = sum_n g_t dl_t B_t      dA   += g_t h_{t-1} a_t dl_t
//   d dl_t = sum_n (g_t h_{t-1} a_t A + g_t B_t x_t),  times sigmoid(u)
//            when dl = softplus(u)
//   dh0   = a_0 g_0.
// a_t h_{t-1} is taken as h_t - dl_t x_t B_t, so the adjoint needs the
// recomputed states but not the decays of the step before.
//
// The block's skip and gate (GATE kernels): with y = (s + Dskip x) silu(z),
// s the scan's read-out, the scan's upstream gradient is gs = gy silu(z)
// (gy where there is no gate), and
//   dz_t = gy_t (s_t + Dskip x_t) silu'(z_t),  silu'(z) = sigmoid(z) (1 + z (1 - sigmoid(z)))
//   dx_t += gs_t Dskip,   dDskip = sum_{b,t} gs_t x_t.
//
// Layout of the work. A thread owns kBwdS = 4 states of one chain (b, d),
// P threads a chain (P = the power of two >= N / 4, at most 8); a block is
// kBwdThreads threads = CPB = kBwdThreads / P chains of one batch row. Sums
// over n are a thread's own four states, then shuffles over its P lanes;
// sums over d (dB, dC) are a reduce-scatter over the chains of a warp, then
// over the warps in shared memory, then one atomic per block, step and state.
//
// The sequence is cut into K segments of whole chunks (kBwdT steps), so that
// K * (channel tiles) * Bsz blocks fill the GPU. Segments are independent
// until their carries are composed, the associative pairs of
// booiljung.github.io "3.1 ...", section 3.1.5.2, in both directions:
//   1. bwd_local_kernel: per segment, the forward recurrence from a zero
//      state, writing the local state and the running sum of dl at every
//      chunk start (the checkpoints), the end state and the segment's sum of
//      dl; in the same pass, what the segment alone sends into the state
//      before it (the adjoint from zero at its end, summed in closed form).
//   2. bwd_main_kernel: per segment, first the carries: the true state
//      entering the segment (h_in(k+1) = exp(A S_k) h_in(k) + hl(k), from
//      h0) and the adjoint entering it from the right (g_out(k-1) =
//      exp(A S_k) g_out(k) + gl(k), from dLoss/dhT), each thread composing
//      the pairs of the segments before and after its own; then chunks last
//      to first: the chunk's start state is its local checkpoint plus
//      exp(A S) h_in, its states are recomputed into registers, and the
//      adjoint runs back through them from g_out, producing every gradient.
// Steps past L are staged as zeros with dl = 0, so they leave h and g as
// they are and contribute nothing; only their stores are skipped.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "device_math.cuh"

namespace selscan {

constexpr int kBwdThreads = 128;
constexpr int kBwdWarps = kBwdThreads / 32;
constexpr int kBwdT = 16;      // timesteps per chunk: states of a chunk live in registers
constexpr int kBwdS = 4;       // states per thread

struct BwdArgs {
    const float *x, *delta, *A, *B, *C, *h0, *gy, *ghT;
    const float *Dskip, *z;    // the block's skip (D) and gate (Bsz, L, D), or null (GATE kernels)
    float *dx, *ddelta, *dA, *dB, *dC, *dh0;
    float *dDskip, *dz;        // their gradients, written when Dskip / z are given
    float *ckpt;               // (Bsz, nch, D, NP) local state at each chunk start
    float *spre;               // (Bsz, nch, D) sum of dl from the segment start to the chunk start
    float *hl, *gl;            // (Bsz, K, D, NP) segment end state from zero; adjoint out of the segment from zero
    float *sdl;                // (Bsz, K, D) the segment's sum of dl
    int64_t Bsz, L, D, N;
    int64_t nch;               // chunks of kBwdT steps
    int64_t cps;               // chunks per segment
    int K;                     // segments
    int softplus;
};

// sigmoid(u) = d softplus(u) / du. ex2 of a large argument gives +inf and
// the quotient 0, the limit.
__device__ __forceinline__ float bwd_sigmoid(float u)
{
    return __fdividef(1.0f, 1.0f + ex2(-u * kLog2e));
}

// Shared memory of the main kernel, in bytes: two buffers of a chunk's raw
// inputs as they arrive (delta, x, gy per step and chain; B and C rows; each
// thread's checkpoint and its chain's sum of dl), the cooked chunk (dl, x,
// gy, sigmoid) per step and chain, dx and d delta per step and chain, and
// the per-warp sums of the dB and dC terms.
// GATE kernels also stage z, and keep gy silu'(z) and dz per step and chain.
__host__ __device__ constexpr int bwd_main_smem(int P, bool gate = false)
{
    return (2 * (gate ? 4 : 3) * kBwdT * (kBwdThreads / P) + 2 * 2 * kBwdT * 4 * P + 2 * 4 * kBwdThreads +
            2 * (kBwdThreads / P) + kBwdT * (kBwdThreads / P) * 4 + (gate ? 4 : 2) * kBwdT * (kBwdThreads / P) +
            kBwdT * kBwdWarps * 2 * 4 * P) * 4;
}
// Steps a stage of the local kernel stages: whole chunks, as many as keep the
// values a thread loads ahead (at most 16 per array) in registers; at
// P = 4 and 8 that leaves at most a 12-byte spill, at P = 1 and 2 (N <= 8,
// more chains per block) the kernel spills more but those shapes are small.
__host__ __device__ constexpr int bwd_local_tt(int P)
{
    return P >= 4 ? 32 : 16;
}
__host__ __device__ constexpr int bwd_local_smem(int P)
{
    return (bwd_local_tt(P) * (kBwdThreads / P) * 4 + 2 * bwd_local_tt(P) * 4 * P) * 4;
}

// The raw inputs of one chunk that this thread stages: loaded into registers
// one chunk ahead, so the loads are in flight while the block works on the
// current chunk. Element j = threadIdx.x + q * kBwdThreads of the chunk's
// (step, chain) rows and (step, state) rows.
template <int P, int TT> struct BwdRegs {
    static constexpr int CPB = kBwdThreads / P, NP = kBwdS * P;
    static constexpr int RX = (TT * CPB + kBwdThreads - 1) / kBwdThreads;
    static constexpr int RB = (TT * NP + kBwdThreads - 1) / kBwdThreads;
    float u[RX], x[RX], gy[RX], z[RX], B[RB], C[RB];
};

// Loads steps t0 .. t0 + TT (zeros from step lim on, and past D and N).
// WZ: also the gate z (when the call has one).
template <int P, int TT, bool WX, bool WGY, bool WB, bool WC, bool WZ = false>
__device__ __forceinline__ void bwd_load(const BwdArgs &a, int64_t b, int64_t d0, int64_t t0, int64_t lim,
                                         BwdRegs<P, TT> &r)
{
    using R = BwdRegs<P, TT>;
#pragma unroll
    for (int q = 0; q < R::RX; ++q) {
        const int j = threadIdx.x + q * kBwdThreads;
        const int i = j / R::CPB, c = j % R::CPB;
        const bool ok = j < TT * R::CPB && t0 + i < lim && d0 + c < a.D;
        const int64_t idx = (b * a.L + t0 + i) * a.D + d0 + c;
        r.u[q] = ok ? __ldg(a.delta + idx) : 0.0f;
        if (WX) r.x[q] = ok ? __ldg(a.x + idx) : 0.0f;
        if (WGY) r.gy[q] = ok ? __ldg(a.gy + idx) : 0.0f;
        if (WZ) r.z[q] = (ok && a.z) ? __ldg(a.z + idx) : 0.0f;
    }
#pragma unroll
    for (int q = 0; q < R::RB; ++q) {
        const int j = threadIdx.x + q * kBwdThreads;
        const int i = j / R::NP, m = j % R::NP;
        const bool ok = j < TT * R::NP && t0 + i < lim && m < a.N;
        const int64_t idx = (b * a.L + t0 + i) * a.N + m;
        if (WB) r.B[q] = ok ? __ldg(a.B + idx) : 0.0f;
        if (WC) r.C[q] = ok ? __ldg(a.C + idx) : 0.0f;
    }
}

// Writes the loaded steps to shared memory: (dl, x, gy, sigmoid(u)) per step
// and chain (dl = 0 from step lim on), B and C rows. WZ: gy is taken times
// silu(z), the scan's share of it, when the call has a gate.
template <int P, int TT, bool WX, bool WGY, bool WB, bool WC, bool WZ = false>
__device__ __forceinline__ void bwd_put(const BwdArgs &a, const BwdRegs<P, TT> &r, int64_t d0, int64_t t0,
                                        int64_t lim, float4 *s_in, float *s_B, float *s_C)
{
    using R = BwdRegs<P, TT>;
#pragma unroll
    for (int q = 0; q < R::RX; ++q) {
        const int j = threadIdx.x + q * kBwdThreads;
        if (j < TT * R::CPB) {
            const int i = j / R::CPB, c = j % R::CPB;
            const bool ok = t0 + i < lim && d0 + c < a.D;
            const float dl = !ok ? 0.0f : (a.softplus ? softplus(r.u[q]) : r.u[q]);
            const float sg = (ok && a.softplus && WX && WGY) ? bwd_sigmoid(r.u[q]) : 1.0f;
            float gv = WGY ? r.gy[q] : 0.0f;
            if (WZ && a.z)
                gv *= silu(r.z[q]);
            s_in[j] = make_float4(dl, WX ? r.x[q] : 0.0f, gv, sg);
        }
    }
#pragma unroll
    for (int q = 0; q < R::RB; ++q) {
        const int j = threadIdx.x + q * kBwdThreads;
        if (j < TT * R::NP) {
            if (WB) s_B[j] = r.B[q];
            if (WC) s_C[j] = r.C[q];
        }
    }
}

__device__ __forceinline__ float2 f2(float v) { return make_float2(v, v); }

// Programmatic dependent launch: the kernels may start while the kernel
// before them is finishing; they call bwd_dep_wait() before they touch
// anything it uses (the wait returns once that whole grid has completed and
// its writes are visible). bwd_dep_trigger() lets the next kernel start
// early.
__device__ __forceinline__ void bwd_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void bwd_dep_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Asynchronous copies global -> shared (cp.async): 4 or 16 bytes, zeros
// instead when !ok (no byte is read then).
__device__ __forceinline__ void cp_async4(void *dst, const void *src, bool ok)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src), "r"(ok ? 4 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async16(void *dst, const void *src, bool ok)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src), "r"(ok ? 16 : 0)
                 : "memory");
}
// A shared-memory load the compiler must issue where it stands: the adjoint
// reads its step's inputs afresh, so that the recomputation's decays are not
// kept alive in registers across the chunk.
__device__ __forceinline__ float4 lds4_fresh(const float4 *p)
{
    float4 v;
    asm volatile("ld.volatile.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"((uint32_t)__cvta_generic_to_shared(p)));
    return v;
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ float2 ex2v(float2 v) { return make_float2(ex2(v.x), ex2(v.y)); }

// Reduce-scatter of v[0 .. 8) over the chains of a warp (lanes that differ in
// bits O, O/2, .., P of the lane index; recursive halving while more than
// one value is left, plain sums after). A lane ends with the sums of
// max(1, 8 P / 32) consecutive entries, starting at the entry its lane bits
// select (bwd_rs_first).
template <int O, int P, int M> struct ChainReduceScatter {
    __device__ __forceinline__ static void run(float (&v)[8], int lane)
    {
        if constexpr (O >= P) {
            if constexpr (M > 1) {
                const bool up = (lane & O) != 0;
#pragma unroll
                for (int j = 0; j < M / 2; ++j) {
                    const float keep = up ? v[j + M / 2] : v[j];
                    const float send = up ? v[j] : v[j + M / 2];
                    v[j] = keep + __shfl_xor_sync(0xffffffffu, send, O);
                }
                ChainReduceScatter<O / 2, P, M / 2>::run(v, lane);
            } else {
                v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
                ChainReduceScatter<O / 2, P, 1>::run(v, lane);
            }
        }
    }
};

template <int P> __device__ __forceinline__ int bwd_rs_first(int lane)
{
    int f = (lane & 16) ? 4 : 0;
    if (P <= 8 && (lane & 8)) f += 2;
    if (P <= 4 && (lane & 4)) f += 1;
    return f;
}
// Lanes that hold a copy of another lane's sums after the plain levels.
template <int P> __device__ __forceinline__ bool bwd_rs_writer(int lane)
{
    return (lane & (3 & ~(P - 1))) == 0;
}

// ---------------------------------------------------------------- kernel 1
// grid (ceil(D / CPB), Bsz, K), kBwdThreads threads, bwd_local_smem(P) bytes.
// One pass over the segment from its start, in stages of TL =
// bwd_local_tt(P) steps (whole chunks; zeros past the segment's end, which
// belong to the next segment), loaded into registers one stage ahead. It
// runs the forward recurrence from a zero state (checkpoints, end state, sum
// of dl) and, in the same pass, forms what the segment alone sends into the
// state before it: the adjoint from zero at the segment's end, which
// unrolls to gl = sum_t exp(A S_t) gy_t C_t with S_t the sum of dl from the
// segment's start through step t.
template <int P, bool GATE>
__global__ void __launch_bounds__(kBwdThreads, 4) bwd_local_kernel(const BwdArgs a)
{
    constexpr int CPB = kBwdThreads / P, NP = kBwdS * P;
    constexpr int TL = bwd_local_tt(P), CH = TL / kBwdT;
    extern __shared__ float4 bwd_smem4[];
    float4 *s_in = bwd_smem4;
    float *s_B = reinterpret_cast<float *>(s_in + TL * CPB);
    float *s_C = s_B + TL * NP;

    const int tid = threadIdx.x, j = tid % P, c = tid / P;
    const int64_t b = blockIdx.y, k = blockIdx.z;
    const int64_t d0 = (int64_t)blockIdx.x * CPB, d = d0 + c;
    const bool chain = d < a.D;
    const int64_t L = a.L, D = a.D, N = a.N, nch = a.nch;
    float2 A2[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int n0 = kBwdS * j + 2 * e;
        A2[e].x = (chain && n0 < N) ? __ldg(a.A + d * N + n0) * kLog2e : 0.0f;
        A2[e].y = (chain && n0 + 1 < N) ? __ldg(a.A + d * N + n0 + 1) * kLog2e : 0.0f;
    }
    const int64_t ci0 = k * a.cps, ci1 = min(ci0 + a.cps, nch);
    const int64_t s0 = ci0 * kBwdT, s1 = min(ci1 * kBwdT, L);   // the segment's steps
    const int nst = (int)((s1 - s0 + TL - 1) / TL);
    const int64_t pair = ((b * a.K + k) * D + d) * NP + kBwdS * j;

    // Launched as a programmatic dependent of the kernel before it (the
    // previous call's main kernel, typically, which may still be adding into
    // the outputs zeroed below): nothing is touched before it has completed.
    bwd_dep_wait();
    // The main kernel adds dA, dB and dC up atomically: zero them here, over
    // the whole grid.
    {
        const int64_t nthr = (int64_t)gridDim.x * gridDim.y * gridDim.z * kBwdThreads;
        const int64_t gt = (((int64_t)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x) * kBwdThreads + tid;
        for (int64_t i = gt; i < a.Bsz * L * N; i += nthr) {
            a.dB[i] = 0.0f;
            a.dC[i] = 0.0f;
        }
        for (int64_t i = gt; i < D * N; i += nthr)
            a.dA[i] = 0.0f;
        if (GATE && a.dDskip)
            for (int64_t i = gt; i < D; i += nthr)
                a.dDskip[i] = 0.0f;
    }

    float2 h[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    float2 gl[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    // exp(A S_t), S_t the sum of dl from the segment's start through step t:
    // the running product of the steps' decays.
    float2 ep[2] = {make_float2(1.f, 1.f), make_float2(1.f, 1.f)};
    float S = 0.0f, Sc = 0.0f;   // compensated sum of dl through the last chunk
    BwdRegs<P, TL> r;
    bwd_load<P, TL, true, true, true, true, GATE>(a, b, d0, s0, s1, r);
    for (int st = 0; st < nst; ++st) {
        const int64_t t0 = s0 + (int64_t)st * TL;
        __syncthreads();
        bwd_put<P, TL, true, true, true, true, GATE>(a, r, d0, t0, s1, s_in, s_B, s_C);
        if (st + 1 < nst)
            bwd_load<P, TL, true, true, true, true, GATE>(a, b, d0, t0 + TL, s1, r);
        __syncthreads();
#pragma unroll 1
        for (int q = 0; q < CH; ++q) {
            const int64_t ci = ci0 + (int64_t)st * CH + q;
            if (chain && ci < ci1) {
                const int64_t o = (b * nch + ci) * D + d;
                *reinterpret_cast<float4 *>(a.ckpt + o * NP + kBwdS * j) =
                    make_float4(h[0].x, h[0].y, h[1].x, h[1].y);
                if (j == 0)
                    a.spre[o] = S;
            }
            float sc = 0.0f;
#pragma unroll
            for (int i = q * kBwdT; i < (q + 1) * kBwdT; ++i) {
                const float4 in = s_in[i * CPB + c];
                const float4 B4 = *reinterpret_cast<const float4 *>(s_B + i * NP + kBwdS * j);
                const float4 C4 = *reinterpret_cast<const float4 *>(s_C + i * NP + kBwdS * j);
                const float dl = in.x, u = dl * in.y;
                const float2 dl2 = f2(dl), u2 = f2(u), gy2 = f2(in.z);
                const float2 a0 = ex2v(__fmul2_rn(dl2, A2[0])), a1 = ex2v(__fmul2_rn(dl2, A2[1]));
                h[0] = __ffma2_rn(a0, h[0], __fmul2_rn(u2, make_float2(B4.x, B4.y)));
                h[1] = __ffma2_rn(a1, h[1], __fmul2_rn(u2, make_float2(B4.z, B4.w)));
                sc += dl;
                ep[0] = __fmul2_rn(ep[0], a0);
                ep[1] = __fmul2_rn(ep[1], a1);
                gl[0] = __ffma2_rn(ep[0], __fmul2_rn(gy2, make_float2(C4.x, C4.y)), gl[0]);
                gl[1] = __ffma2_rn(ep[1], __fmul2_rn(gy2, make_float2(C4.z, C4.w)), gl[1]);
            }
            const float yk = sc - Sc, tk = S + yk;   // S += sc, compensated
            Sc = (tk - S) - yk;
            S = tk;
        }
    }
    bwd_dep_trigger();
    if (chain) {
        *reinterpret_cast<float4 *>(a.hl + pair) = make_float4(h[0].x, h[0].y, h[1].x, h[1].y);
        if (j == 0)
            a.sdl[(b * a.K + k) * D + d] = S;
        if (k > 0)   // nothing lies before the first segment
            *reinterpret_cast<float4 *>(a.gl + pair) = make_float4(gl[0].x, gl[0].y, gl[1].x, gl[1].y);
    }
}

constexpr int kBwdFold = 8;   // segments whose pairs the main kernel loads at once

// ---------------------------------------------------------------- kernel 2
// grid (ceil(D / CPB), Bsz, K), kBwdThreads threads, bwd_main_smem(P) bytes.
// dA, dB and dC are accumulated atomically (the local kernel zeroed them).
// Chunk inputs arrive by cp.async into one of two raw buffers while the
// block works on the other, so no register holds a chunk in flight.
template <int P, bool GATE>
__global__ void __launch_bounds__(kBwdThreads, 4) bwd_main_kernel(const BwdArgs a)
{
    constexpr int CPB = kBwdThreads / P, NP = kBwdS * P;
    constexpr int TC = kBwdT * CPB, TN = kBwdT * NP;
    constexpr int RS = (8 * P / 32) > 1 ? 8 * P / 32 : 1;   // reduce-scatter values left per lane
    extern __shared__ float4 bwd_smem4[];
    float4 *s_ck = bwd_smem4;                       // [2][kBwdThreads] checkpoints
    constexpr int NRAW = GATE ? 4 : 3;
    float4 *s_in = s_ck + 2 * kBwdThreads;          // [T][CPB] (dl, x, gy, sigmoid); gy times silu(z) if gated
    float *s_raw = reinterpret_cast<float *>(s_in + TC);   // [2][NRAW][T][CPB] delta, x, gy (, z)
    float *s_rB = s_raw + 2 * NRAW * TC;            // [2][T][NP]
    float *s_rC = s_rB + 2 * TN;
    float *s_sp = s_rC + 2 * TN;                    // [2][CPB]
    float *s_dx = s_sp + 2 * CPB;                   // [T][CPB]
    float *s_dd = s_dx + TC;
    float *s_part = s_dd + TC;                      // [T][warps][2][NP]
    float *s_zf = s_part + kBwdT * kBwdWarps * 2 * NP;   // GATE: [T][CPB] gy silu'(z)
    float *s_dz = s_zf + TC;                        // GATE: [T][CPB] dz

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, j = tid % P, c = tid / P;
    const int64_t b = blockIdx.y, k = blockIdx.z;
    const int64_t d0 = (int64_t)blockIdx.x * CPB, d = d0 + c;
    const bool chain = d < a.D;
    const int64_t L = a.L, D = a.D, N = a.N, nch = a.nch;
    float2 A2[2], An[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int n0 = kBwdS * j + 2 * e;
        An[e].x = (chain && n0 < N) ? __ldg(a.A + d * N + n0) : 0.0f;
        An[e].y = (chain && n0 + 1 < N) ? __ldg(a.A + d * N + n0 + 1) : 0.0f;
        A2[e] = __fmul2_rn(An[e], f2(kLog2e));
    }
    const int64_t ci0 = k * a.cps, ci1 = min(ci0 + a.cps, nch);
    bwd_dep_wait();   // the local kernel's checkpoints and segment pairs
    float2 hin[2], g[2], dA[2];
    dA[0] = dA[1] = make_float2(0.f, 0.f);
    const bool has_z = GATE && a.z != nullptr, has_sk = GATE && a.Dskip != nullptr;
    const float dsk = (has_sk && chain) ? __ldg(a.Dskip + d) : 0.0f;
    float ddsk = 0.0f;   // dDskip of this chain, summed over the segment (lane j == 0)

    // Issues the copies of chunk ci into raw buffer s.
    auto stage = [&](int64_t ci, int sb) {
        const int64_t t0 = ci * kBwdT;
        float *ru = s_raw + (sb * NRAW) * TC, *rx = ru + TC, *rg = rx + TC;
        for (int e = tid; e < TC; e += kBwdThreads) {
            const int i = e / CPB, cc = e % CPB;
            const bool ok = t0 + i < L && d0 + cc < D;
            const int64_t idx = ok ? (b * L + t0 + i) * D + d0 + cc : 0;
            cp_async4(ru + e, a.delta + idx, ok);
            cp_async4(rx + e, a.x + idx, ok);
            cp_async4(rg + e, a.gy + idx, ok);
            if (GATE)
                cp_async4(rg + TC + e, a.z + (has_z ? idx : 0), ok && has_z);
        }
        for (int e = tid; e < TN; e += kBwdThreads) {
            const int i = e / NP, m = e % NP;
            const bool ok = t0 + i < L && m < N;
            const int64_t idx = ok ? (b * L + t0 + i) * N + m : 0;
            cp_async4(s_rB + sb * TN + e, a.B + idx, ok);
            cp_async4(s_rC + sb * TN + e, a.C + idx, ok);
        }
        const int64_t o = (b * nch + ci) * D + d;
        cp_async16(s_ck + sb * kBwdThreads + tid, a.ckpt + (chain ? o * NP + kBwdS * j : 0), chain);
        if (j == 0)
            cp_async4(s_sp + sb * CPB + c, a.spre + (chain ? o : 0), chain);
        cp_async_commit();
    };

    stage(ci1 - 1, (int)((ci1 - 1) & 1));
    // While the first chunk arrives: the state entering this segment, h0
    // carried through segments 0 .. k-1 (h_in(k'+1) = exp(A S_k') h_in(k') +
    // hl(k')), and the adjoint entering it from the right, dLoss/dhT carried
    // back through segments K-1 .. k+1 (g(k'-1) = exp(A S_k') g(k') + gl(k')):
    // the associative pairs of booiljung.github.io "3.1 ...", section 3.1.5.2,
    // composed in both directions. Up to kBwdFold segments' pairs are loaded
    // before their dependent arithmetic.
    {
        float hv[kBwdS], gv[kBwdS];
#pragma unroll
        for (int e = 0; e < kBwdS; ++e) {
            const int64_t n = kBwdS * j + e;
            const bool st = chain && n < N;
            hv[e] = (st && a.h0) ? __ldg(a.h0 + (b * D + d) * N + n) : 0.0f;
            gv[e] = (st && a.ghT) ? __ldg(a.ghT + (b * D + d) * N + n) : 0.0f;
        }
        hin[0] = make_float2(hv[0], hv[1]);
        hin[1] = make_float2(hv[2], hv[3]);
        g[0] = make_float2(gv[0], gv[1]);
        g[1] = make_float2(gv[2], gv[3]);
        const int64_t seg0 = b * a.K * D + d;   // segment kk of this chain: seg0 + kk * D
        for (int64_t k0 = 0; k0 < k; k0 += kBwdFold) {
            float dec[kBwdFold];
            float4 lv[kBwdFold];
#pragma unroll
            for (int q = 0; q < kBwdFold; ++q) {
                const bool ok = chain && k0 + q < k;
                const int64_t sg = seg0 + (k0 + q) * D;
                dec[q] = ok ? a.sdl[sg] : 0.0f;
                lv[q] = ok ? *reinterpret_cast<const float4 *>(a.hl + sg * NP + kBwdS * j) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int q = 0; q < kBwdFold; ++q) {
                if (k0 + q < k) {
                    const float2 d2 = f2(dec[q]);
                    hin[0] = __ffma2_rn(ex2v(__fmul2_rn(d2, A2[0])), hin[0], make_float2(lv[q].x, lv[q].y));
                    hin[1] = __ffma2_rn(ex2v(__fmul2_rn(d2, A2[1])), hin[1], make_float2(lv[q].z, lv[q].w));
                }
            }
        }
        for (int64_t k0 = a.K - 1; k0 > k; k0 -= kBwdFold) {
            float dec[kBwdFold];
            float4 lv[kBwdFold];
#pragma unroll
            for (int q = 0; q < kBwdFold; ++q) {
                const bool ok = chain && k0 - q > k;
                const int64_t sg = seg0 + (k0 - q) * D;
                dec[q] = ok ? a.sdl[sg] : 0.0f;
                lv[q] = ok ? *reinterpret_cast<const float4 *>(a.gl + sg * NP + kBwdS * j) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int q = 0; q < kBwdFold; ++q) {
                if (k0 - q > k) {
                    const float2 d2 = f2(dec[q]);
                    g[0] = __ffma2_rn(ex2v(__fmul2_rn(d2, A2[0])), g[0], make_float2(lv[q].x, lv[q].y));
                    g[1] = __ffma2_rn(ex2v(__fmul2_rn(d2, A2[1])), g[1], make_float2(lv[q].z, lv[q].w));
                }
            }
        }
    }
    for (int64_t ci = ci1 - 1; ci >= ci0; --ci) {
        const int64_t t0 = ci * kBwdT;
        const int cur = (int)(ci & 1);
        cp_async_wait_all();
        __syncthreads();   // the chunk has landed; the one before is done with s_in
        if (ci > ci0)
            stage(ci - 1, cur ^ 1);
        {
            const float *ru = s_raw + (cur * NRAW) * TC, *rx = ru + TC, *rg = rx + TC;
            for (int e = tid; e < TC; e += kBwdThreads) {
                const int i = e / CPB, cc = e % CPB;
                const bool ok = t0 + i < L && d0 + cc < D;
                const float u = ru[e];
                const float dl = !ok ? 0.0f : (a.softplus ? softplus(u) : u);
                const float sg = (ok && a.softplus) ? bwd_sigmoid(u) : 1.0f;
                float gv = rg[e];
                if (has_z) {   // the scan's share silu(z) of gy; dz's factor gy silu'(z)
                    const float zv = rg[TC + e], sz = silu_gate(zv);
                    s_zf[e] = gv * sz * fmaf(zv, 1.0f - sz, 1.0f);
                    gv *= zv * sz;
                }
                s_in[e] = make_float4(dl, rx[e], gv, sg);
            }
        }
        __syncthreads();
        const float *s_B = s_rB + cur * TN, *s_C = s_rC + cur * TN;

        // The chunk's states: from the true state at its start.
        float2 hs[kBwdT][2];
        {
            const float4 ck = s_ck[cur * kBwdThreads + tid];
            const float2 sp2 = f2(s_sp[cur * CPB + c]);
            float2 h0v = __ffma2_rn(ex2v(__fmul2_rn(sp2, A2[0])), hin[0], make_float2(ck.x, ck.y));
            float2 h1v = __ffma2_rn(ex2v(__fmul2_rn(sp2, A2[1])), hin[1], make_float2(ck.z, ck.w));
#pragma unroll
            for (int i = 0; i < kBwdT; ++i) {
                const float4 in = s_in[i * CPB + c];
                const float4 B4 = *reinterpret_cast<const float4 *>(s_B + i * NP + kBwdS * j);
                const float2 dl2 = f2(in.x), u2 = f2(in.x * in.y);
                h0v = __ffma2_rn(ex2v(__fmul2_rn(dl2, A2[0])), h0v, __fmul2_rn(u2, make_float2(B4.x, B4.y)));
                h1v = __ffma2_rn(ex2v(__fmul2_rn(dl2, A2[1])), h1v, __fmul2_rn(u2, make_float2(B4.z, B4.w)));
                hs[i][0] = h0v;
                hs[i][1] = h1v;
            }
        }

        // The adjoint back through the chunk.
#pragma unroll
        for (int i = kBwdT - 1; i >= 0; --i) {
            const float4 in = lds4_fresh(s_in + i * CPB + c);
            const float4 B4 = lds4_fresh(reinterpret_cast<const float4 *>(s_B + i * NP + kBwdS * j));
            const float4 C4 = *reinterpret_cast<const float4 *>(s_C + i * NP + kBwdS * j);
            const float dl = in.x, xv = in.y, gyv = in.z, sg = in.w, u = dl * xv;
            const float2 dl2 = f2(dl), u2 = f2(u), gy2 = f2(gyv), nu2 = f2(-u);
            const float2 Bp[2] = {make_float2(B4.x, B4.y), make_float2(B4.z, B4.w)};
            const float2 Cp[2] = {make_float2(C4.x, C4.y), make_float2(C4.z, C4.w)};
            float2 pB[2], pC[2], sdl2 = make_float2(0.f, 0.f), sgb2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                g[e] = __ffma2_rn(gy2, Cp[e], g[e]);                    // dLoss/dh_t
                pC[e] = __fmul2_rn(gy2, hs[i][e]);
                const float2 dan = __fmul2_rn(g[e], __ffma2_rn(nu2, Bp[e], hs[i][e]));   // g a_t h_{t-1}
                sdl2 = __ffma2_rn(dan, An[e], sdl2);
                sgb2 = __ffma2_rn(g[e], Bp[e], sgb2);
                dA[e] = __ffma2_rn(dan, dl2, dA[e]);
                pB[e] = __fmul2_rn(g[e], u2);
                g[e] = __fmul2_rn(g[e], ex2v(__fmul2_rn(dl2, A2[e])));  // into h_{t-1}
            }
            // dx and d delta: the chain's sums over n (and, gated, the
            // scan's read-out s_t for dz)
            float sdl = sdl2.x + sdl2.y, sgb = sgb2.x + sgb2.y, ys = 0.0f;
            if constexpr (GATE) {
                const float2 y2 = __ffma2_rn(Cp[1], hs[i][1], __fmul2_rn(Cp[0], hs[i][0]));
                ys = y2.x + y2.y;
            }
#pragma unroll
            for (int o = 1; o < P; o <<= 1) {
                sdl += __shfl_xor_sync(0xffffffffu, sdl, o);
                sgb += __shfl_xor_sync(0xffffffffu, sgb, o);
                if constexpr (GATE)
                    ys += __shfl_xor_sync(0xffffffffu, ys, o);
            }
            if (j == 0) {
                s_dx[i * CPB + c] = GATE ? fmaf(gyv, dsk, sgb * dl) : sgb * dl;
                s_dd[i * CPB + c] = fmaf(xv, sgb, sdl) * sg;
                if constexpr (GATE) {
                    if (has_z)
                        s_dz[i * CPB + c] = s_zf[i * CPB + c] * fmaf(dsk, xv, ys);
                    ddsk = fmaf(gyv, xv, ddsk);
                }
            }
            // dB and dC: sums over the warp's chains
            float v[8] = {pB[0].x, pB[0].y, pB[1].x, pB[1].y, pC[0].x, pC[0].y, pC[1].x, pC[1].y};
            ChainReduceScatter<16, P, 8>::run(v, lane);
            if (bwd_rs_writer<P>(lane)) {
                const int f = bwd_rs_first<P>(lane);
#pragma unroll
                for (int q = 0; q < RS; ++q) {
                    const int vi = f + q, kind = vi >> 2, n = kBwdS * j + (vi & 3);
                    s_part[((i * kBwdWarps + warp) * 2 + kind) * NP + n] = v[q];
                }
            }
        }
        __syncthreads();

        // The chunk's outputs: dx and d delta rows, the block's dB and dC.
        for (int e = tid; e < TC; e += kBwdThreads) {
            const int i = e / CPB, cc = e % CPB;
            const int64_t t = t0 + i, dd = d0 + cc;
            if (t < L && dd < D) {
                const int64_t idx = (b * L + t) * D + dd;
                a.dx[idx] = s_dx[e];
                a.ddelta[idx] = s_dd[e];
                if (has_z)
                    a.dz[idx] = s_dz[e];
            }
        }
        for (int e = tid; e < kBwdT * 2 * NP; e += kBwdThreads) {
            const int i = e / (2 * NP), rem = e % (2 * NP), kind = rem / NP, n = rem % NP;
            const int64_t t = t0 + i;
            if (t < L && n < N) {
                float sum = 0.0f;
#pragma unroll
                for (int w = 0; w < kBwdWarps; ++w)
                    sum += s_part[(i * kBwdWarps + w) * 2 * NP + rem];
                atomicAdd((kind ? a.dC : a.dB) + (b * L + t) * N + n, sum);
            }
        }
    }
    bwd_dep_trigger();   // the next call's local kernel may be scheduled
    if (chain) {
        if (has_sk && j == 0)
            atomicAdd(a.dDskip + d, ddsk);
        const float dv[4] = {dA[0].x, dA[0].y, dA[1].x, dA[1].y}, gv[4] = {g[0].x, g[0].y, g[1].x, g[1].y};
#pragma unroll
        for (int e = 0; e < kBwdS; ++e) {
            const int64_t n = kBwdS * j + e;
            if (n < N) {
                atomicAdd(a.dA + d * N + n, dv[e]);
                if (k == 0 && a.dh0)
                    a.dh0[(b * D + d) * N + n] = gv[e];
            }
        }
    }
}

// ---- host side: the launch shape and the launches -------------------------

struct BwdShape {
    int P;           // threads per chain
    int NP;          // padded states per chain (kBwdS * P)
    int cpb;         // chains per block
    int64_t nch;     // chunks of kBwdT steps
    int64_t cps;     // chunks per segment
    int K;           // segments
    int64_t gx;      // blocks along D
};

// Segments: as many as fill the resident blocks of the main kernel in one
// wave, each at least 4 chunks long.
inline BwdShape bwd_shape(int64_t Bsz, int64_t L, int64_t D, int64_t N, int resident_blocks)
{
    BwdShape s;
    s.P = 1;
    while (s.P * kBwdS < N) s.P <<= 1;
    s.NP = kBwdS * s.P;
    s.cpb = kBwdThreads / s.P;
    s.nch = (L + kBwdT - 1) / kBwdT;
    s.gx = (D + s.cpb - 1) / s.cpb;
    int64_t K = 1;
    const int64_t cols = s.gx * Bsz;
    if (cols > 0 && cols < resident_blocks) K = resident_blocks / cols;
    const int64_t maxK = (s.nch + 3) / 4;
    if (K > maxK) K = maxK;
    if (K > 65535) K = 65535;
    if (K < 1) K = 1;
    s.cps = (s.nch + K - 1) / K;
    if (s.cps < 1) s.cps = 1;
    s.K = (int)((s.nch + s.cps - 1) / s.cps);
    if (s.K < 1) s.K = 1;
    return s;
}

// The three launches; bwd_prepare(P) must have run on this device.
template <int P, bool GATE>
inline cudaError_t launch_bwd_p(const BwdArgs &a, const BwdShape &s, cudaStream_t st)
{
    const dim3 grid((unsigned)s.gx, (unsigned)a.Bsz, (unsigned)s.K);
    // Both kernels are programmatic dependents of the kernel before them
    // (each waits in the kernel before it touches what that one uses).
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kBwdThreads);
    cfg.dynamicSmemBytes = bwd_local_smem(P);
    cfg.stream = st;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, bwd_local_kernel<P, GATE>, a);
    cfg.dynamicSmemBytes = bwd_main_smem(P, GATE);
    if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, bwd_main_kernel<P, GATE>, a);
    return e == cudaSuccess ? cudaGetLastError() : e;
}

// GATE kernels when the call has a skip or a gate.
inline cudaError_t launch_scan_bwd(BwdArgs a, const BwdShape &s, cudaStream_t st)
{
    a.nch = s.nch;
    a.cps = s.cps;
    a.K = s.K;
    const bool gate = a.Dskip != nullptr || a.z != nullptr;
    switch (s.P) {
    case 1: return gate ? launch_bwd_p<1, true>(a, s, st) : launch_bwd_p<1, false>(a, s, st);
    case 2: return gate ? launch_bwd_p<2, true>(a, s, st) : launch_bwd_p<2, false>(a, s, st);
    case 4: return gate ? launch_bwd_p<4, true>(a, s, st) : launch_bwd_p<4, false>(a, s, st);
    default: return gate ? launch_bwd_p<8, true>(a, s, st) : launch_bwd_p<8, false>(a, s, st);
    }
}

// Sets the kernels' shared-memory limits for threads-per-chain P and returns
// how many blocks of the main kernel are resident per SM (0 on error).
template <int P, bool GATE>
inline int bwd_prepare_p()
{
    if (cudaFuncSetAttribute(bwd_main_kernel<P, GATE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             bwd_main_smem(P, GATE)) != cudaSuccess ||
        cudaFuncSetAttribute(bwd_local_kernel<P, GATE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             bwd_local_smem(P)) != cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, bwd_main_kernel<P, GATE>, kBwdThreads,
                                                      bwd_main_smem(P, GATE)) != cudaSuccess)
        return 0;
    return n;
}

inline int bwd_prepare(int P, bool gate)
{
    switch (P) {
    case 1: return gate ? bwd_prepare_p<1, true>() : bwd_prepare_p<1, false>();
    case 2: return gate ? bwd_prepare_p<2, true>() : bwd_prepare_p<2, false>();
    case 4: return gate ? bwd_prepare_p<4, true>() : bwd_prepare_p<4, false>();
    default: return gate ? bwd_prepare_p<8, true>() : bwd_prepare_p<8, false>();
    }
}

} // namespace selscan
