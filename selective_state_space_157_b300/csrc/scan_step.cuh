// scan_step.cuh -- the O(1)-state decode step (youngju.dev "Mamba: Selective
// State Space Models", section 6: one token updates a fixed-size state).
//
//   state'[b,d,n] = exp(delta[b,d]*A[d,n]) * state[b,d,n] + delta[b,d]*B[b,n]*x[b,d]
//   y[b,d]        = sum_n state'[b,d,n] * C[b,n]
//
// The step reads and writes the whole state once: it is bound by HBM
// bandwidth. G = N/4 consecutive lanes share a chain, each holding 4 states
// moved as one 16-byte load and store, so a warp streams 32 contiguous
// 16-byte pieces of the state; the outputs of the G lanes are summed with
// warp shuffles.
#pragma once

#include "device_math.cuh"

namespace selscan {

constexpr int kStepThreads = 256;

struct StepArgs {
    float *state;
    const float *x, *delta, *A, *B, *C;
    float *y;
    int64_t Bsz, D, N;
};

template <int G>
__global__ void __launch_bounds__(kStepThreads) step_vec_kernel(const StepArgs a)
{
    const int64_t chains = a.Bsz * a.D;
    const int64_t gt = (int64_t)blockIdx.x * kStepThreads + threadIdx.x;
    const int64_t chain_raw = gt / G;
    const int q = (int)(gt % G);
    const bool active = chain_raw < chains;
    const int64_t chain = active ? chain_raw : chains - 1;
    const int64_t b = chain / a.D, d = chain - b * a.D;

    float4 *sp = reinterpret_cast<float4 *>(a.state) + chain * G + q;
    float4 s = *sp;
    const float4 A4 = __ldg(reinterpret_cast<const float4 *>(a.A) + d * G + q);
    const float4 B4 = __ldg(reinterpret_cast<const float4 *>(a.B) + b * G + q);
    const float4 C4 = __ldg(reinterpret_cast<const float4 *>(a.C) + b * G + q);
    const float dl = __ldg(a.delta + chain);
    const float u = dl * __ldg(a.x + chain);
    const float dk = dl * kLog2e;

    s.x = fmaf(ex2(dk * A4.x), s.x, u * B4.x);
    s.y = fmaf(ex2(dk * A4.y), s.y, u * B4.y);
    s.z = fmaf(ex2(dk * A4.z), s.z, u * B4.z);
    s.w = fmaf(ex2(dk * A4.w), s.w, u * B4.w);
    float yv = fmaf(s.x, C4.x, s.y * C4.y) + fmaf(s.z, C4.z, s.w * C4.w);
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1)
        yv += __shfl_xor_sync(0xffffffffu, yv, o);
    if (active) {
        *sp = s;
        if (q == 0)
            a.y[chain] = yv;
    }
}

// Any N <= 64 and any 4-byte alignment: one thread per chain.
__global__ void __launch_bounds__(kStepThreads) step_scalar_kernel(const StepArgs a)
{
    const int64_t chain = (int64_t)blockIdx.x * kStepThreads + threadIdx.x;
    if (chain >= a.Bsz * a.D)
        return;
    const int64_t b = chain / a.D, d = chain - b * a.D;
    const float dl = a.delta[chain];
    const float u = dl * a.x[chain];
    const float dk = dl * kLog2e;
    float *sp = a.state + chain * a.N;
    const float *Ap = a.A + d * a.N;
    const float *Bp = a.B + b * a.N;
    const float *Cp = a.C + b * a.N;
    float yv = 0.0f;
    for (int64_t n = 0; n < a.N; ++n) {
        const float s = fmaf(ex2(dk * Ap[n]), sp[n], u * Bp[n]);
        sp[n] = s;
        yv = fmaf(s, Cp[n], yv);
    }
    a.y[chain] = yv;
}

} // namespace selscan
