// conv1d.cuh -- the causal depthwise convolution and SiLU in front of the
// scan (youngju.dev "Mamba: Selective State Space Models", section 3.4, the
// MambaBlock listing: one filter of K taps per channel, padded by K - 1 in
// front and cut back to L outputs, then SiLU):
//
//   out[b,t,d] = silu(bias[d] + sum_{k<K} w[d,k] * x[b, t-K+1+k, d])
//
// with inputs before t = 0 taken from a carried state of the previous K - 1
// inputs per channel (oldest first), zeros when there is none.
//
// Bound by HBM: x is read once and out written once. A thread owns one
// channel of one batch row over a run of kConvT timesteps; lanes take
// consecutive channels, so every load and store is a coalesced row. The K - 1
// previous inputs slide through registers, so each input is loaded once per
// run, plus K - 1 halo values at the run's start (from x, or from the state
// for the first run).
#pragma once

#include "device_math.cuh"

namespace selscan {

constexpr int kConvThreads = 128;
constexpr int kConvT = 64;        // timesteps per thread
constexpr int kConvMaxK = 8;

struct ConvArgs {
    const void *x;
    const float *w;          // (D, K)
    const float *bias;       // (D) or null
    void *out;
    const float *state_in;   // (Bsz, D, K-1) or null
    float *state_out;        // (Bsz, D, K-1) or null
    int64_t Bsz, L, D;
    int silu;
};

template <int K>
__device__ __forceinline__ float conv_state_value(const ConvArgs &a, int64_t b, int64_t d, int64_t tau)
{
    // Input at time tau < 0: the carried state's entry K-1+tau (oldest first).
    return a.state_in ? a.state_in[(b * a.D + d) * (K - 1) + (K - 1 + tau)] : 0.0f;
}

template <typename T, int K>
__global__ void __launch_bounds__(kConvThreads) conv1d_kernel(const ConvArgs a)
{
    const int64_t d = (int64_t)blockIdx.x * kConvThreads + threadIdx.x;
    const int64_t b = blockIdx.y;
    const int64_t t0 = (int64_t)blockIdx.z * kConvT;
    if (d >= a.D)
        return;
    const int64_t D = a.D, L = a.L;
    float w[K];
#pragma unroll
    for (int k = 0; k < K; ++k)
        w[k] = __ldg(a.w + d * K + k);
    const float bias = a.bias ? __ldg(a.bias + d) : 0.0f;

    const T *xp = static_cast<const T *>(a.x) + b * L * D + d;
    // win[j] = x at time t0 - (K-1) + j: the K - 1 inputs before the run.
    float win[K > 1 ? K - 1 : 1];
#pragma unroll
    for (int j = 0; j < K - 1; ++j) {
        const int64_t tau = t0 - (K - 1) + j;
        win[j] = tau >= 0 ? Io<T>::load(xp + tau * D) : conv_state_value<K>(a, b, d, tau);
    }

    T *op = static_cast<T *>(a.out) + b * L * D + d;
    const int64_t n = L - t0 < kConvT ? L - t0 : kConvT;
#pragma unroll 8
    for (int64_t t = t0; t < t0 + n; ++t) {
        const float xv = Io<T>::load(xp + t * D);
        float acc = bias;
#pragma unroll
        for (int k = 0; k < K - 1; ++k)
            acc = fmaf(w[k], win[k], acc);
        acc = fmaf(w[K - 1], xv, acc);
#pragma unroll
        for (int k = 0; k + 1 < K - 1; ++k)
            win[k] = win[k + 1];
        if (K > 1)
            win[K > 1 ? K - 2 : 0] = xv;
        Io<T>::store(op + t * D, a.silu ? acc * silu_gate(acc) : acc);
    }

    // The run that ends the sequence hands the last K - 1 inputs over.
    if (a.state_out && t0 + n == L) {
#pragma unroll
        for (int j = 0; j < K - 1; ++j) {
            const int64_t tau = L - (K - 1) + j;
            a.state_out[(b * D + d) * (K - 1) + j] =
                tau >= 0 ? Io<T>::load(xp + tau * D) : conv_state_value<K>(a, b, d, tau);
        }
    }
}

// One decode step: out = silu(bias + sum_{k<K-1} w[k] state[k] + w[K-1] x),
// then the state shifts by one and takes x. One thread per channel; fp32.
struct ConvStepArgs {
    float *state;            // (Bsz, D, K-1), in place
    const float *x;          // (Bsz, D)
    const float *w, *bias;
    float *out;              // (Bsz, D)
    int64_t Bsz, D;
    int silu;
};

template <int K>
__global__ void __launch_bounds__(kConvThreads) conv1d_step_kernel(const ConvStepArgs a)
{
    const int64_t c = (int64_t)blockIdx.x * kConvThreads + threadIdx.x;
    if (c >= a.Bsz * a.D)
        return;
    const int64_t d = c % a.D;
    float *st = a.state + c * (K - 1);
    const float xv = a.x[c];
    float acc = a.bias ? __ldg(a.bias + d) : 0.0f;
    float prev[K > 1 ? K - 1 : 1];
#pragma unroll
    for (int k = 0; k < K - 1; ++k) {
        prev[k] = st[k];
        acc = fmaf(__ldg(a.w + d * K + k), prev[k], acc);
    }
    acc = fmaf(__ldg(a.w + d * K + K - 1), xv, acc);
#pragma unroll
    for (int k = 0; k + 1 < K - 1; ++k)
        st[k] = prev[k + 1];
    if (K > 1)
        st[K > 1 ? K - 2 : 0] = xv;
    a.out[c] = a.silu ? acc * silu_gate(acc) : acc;
}

} // namespace selscan
