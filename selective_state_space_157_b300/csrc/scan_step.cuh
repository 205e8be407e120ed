// scan_step.cuh -- the O(1)-state decode step (youngju.dev "Mamba: Selective
// State Space Models", section 6: one token updates a fixed-size state).
//
//   state'[b,d,n] = exp(delta[b,d]*A[d,n]) * state[b,d,n] + delta[b,d]*B[b,n]*x[b,d]
//   y[b,d]        = sum_n state'[b,d,n] * C[b,n]
//
// The step reads and writes the whole state once: it is bound by HBM
// bandwidth. G consecutive lanes share a chain, each holding 4V states moved
// as V 16-byte loads and stores issued together, so a warp streams contiguous
// state and every lane keeps several requests in flight; the outputs of the G
// lanes are summed with warp shuffles.
#pragma once

#include "device_math.cuh"

namespace selscan {

constexpr int kStepThreads = 256;

struct StepArgs {
    float *state;
    const float *x, *delta, *A, *B, *C;
    float *y;
    const float *Dskip;   // (D) or null: the block's skip term
    const float *z;       // (Bsz, D) or null: the block's gate
    int64_t Bsz, D, N;
};

// One state: h' = e^(dl a) h + Bbar x, with Bbar = dl * b, or the
// zero-order-hold form (compiled separately, so the simplified form keeps
// its short instruction stream).
template <bool ZOH>
__device__ __forceinline__ float step_state(float h, float a, float b, float dl, float dk, float u, float xv)
{
    const float decay = ex2(dk * a);
    if constexpr (ZOH)
        return fmaf(decay, h, zoh_coef(dl, a, decay) * xv * b);
    return fmaf(decay, h, u * b);
}

// The block's skip and gate on a chain's read-out (block_out), if asked for.
__device__ __forceinline__ float step_block(const StepArgs &a, float yv, float xv, int64_t chain, int64_t d)
{
    if (!a.Dskip && !a.z)
        return yv;
    return block_out(yv, a.Dskip ? __ldg(a.Dskip + d) : 0.0f, xv, a.z != nullptr, a.z ? __ldg(a.z + chain) : 0.0f);
}

// V 16-byte groups (4V states) per lane, G lanes per chain (N = 4 V G).
// Launched as a programmatic dependent of the kernel before it on the stream
// (the previous decode step, typically): it may be scheduled while that one
// drains, and waits for it to complete before reading anything; it lets the
// next step be scheduled as soon as all of its own CTAs have started.
template <int G, int V, bool ZOH>
__global__ void __launch_bounds__(kStepThreads) step_vec_kernel(const StepArgs a)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t chains = a.Bsz * a.D;
    const int64_t gt = (int64_t)blockIdx.x * kStepThreads + threadIdx.x;
    const int64_t chain_raw = gt / G;
    const int q = (int)(gt % G);
    const bool active = chain_raw < chains;
    const int64_t chain = active ? chain_raw : chains - 1;
    const int64_t b = chain / a.D, d = chain - b * a.D;

    // All loads first, so that each lane has V + 3V + 2 requests in flight.
    float4 *sp = reinterpret_cast<float4 *>(a.state) + (chain * G + q) * V;
    float4 s[V], A4[V], B4[V], C4[V];
#pragma unroll
    for (int v = 0; v < V; ++v) {
        s[v] = __ldcs(sp + v);   // read once: streaming
        A4[v] = __ldg(reinterpret_cast<const float4 *>(a.A) + (d * G + q) * V + v);
        B4[v] = __ldg(reinterpret_cast<const float4 *>(a.B) + (b * G + q) * V + v);
        C4[v] = __ldg(reinterpret_cast<const float4 *>(a.C) + (b * G + q) * V + v);
    }
    const float dl = __ldg(a.delta + chain);
    const float xv = __ldg(a.x + chain);
    const float u = dl * xv;
    const float dk = dl * kLog2e;

    float yv = 0.0f;
#pragma unroll
    for (int v = 0; v < V; ++v) {
        s[v].x = step_state<ZOH>(s[v].x, A4[v].x, B4[v].x, dl, dk, u, xv);
        s[v].y = step_state<ZOH>(s[v].y, A4[v].y, B4[v].y, dl, dk, u, xv);
        s[v].z = step_state<ZOH>(s[v].z, A4[v].z, B4[v].z, dl, dk, u, xv);
        s[v].w = step_state<ZOH>(s[v].w, A4[v].w, B4[v].w, dl, dk, u, xv);
        yv += fmaf(s[v].x, C4[v].x, s[v].y * C4[v].y) + fmaf(s[v].z, C4[v].z, s[v].w * C4[v].w);
    }
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1)
        yv += __shfl_xor_sync(0xffffffffu, yv, o);
    if (active) {
#pragma unroll
        for (int v = 0; v < V; ++v)
            __stcs(sp + v, s[v]);   // written once: streaming
        if (q == 0)
            a.y[chain] = step_block(a, yv, xv, chain, d);
    }
}

// Any N <= 64 and any 4-byte alignment: one thread per chain.
template <bool ZOH>
__global__ void __launch_bounds__(kStepThreads) step_scalar_kernel(const StepArgs a)
{
    const int64_t chain = (int64_t)blockIdx.x * kStepThreads + threadIdx.x;
    if (chain >= a.Bsz * a.D)
        return;
    const int64_t b = chain / a.D, d = chain - b * a.D;
    const float dl = a.delta[chain];
    const float xv = a.x[chain];
    const float u = dl * xv;
    const float dk = dl * kLog2e;
    float *sp = a.state + chain * a.N;
    const float *Ap = a.A + d * a.N;
    const float *Bp = a.B + b * a.N;
    const float *Cp = a.C + b * a.N;
    float yv = 0.0f;
    for (int64_t n = 0; n < a.N; ++n) {
        const float s = step_state<ZOH>(sp[n], Ap[n], Bp[n], dl, dk, u, xv);
        sp[n] = s;
        yv = fmaf(s, Cp[n], yv);
    }
    a.y[chain] = step_block(a, yv, xv, chain, d);
}

} // namespace selscan
