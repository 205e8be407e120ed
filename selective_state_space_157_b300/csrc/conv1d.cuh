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
constexpr int kConvBatch = 8;     // inputs loaded ahead of the stores that use them

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
    // kConvBatch inputs are loaded before any output of the batch is stored:
    // out never overlaps x (checked on the host), but the compiler cannot
    // know that, and would otherwise wait for each load in turn.
    for (int64_t tb = t0; tb < t0 + n; tb += kConvBatch) {
        float xv[kConvBatch];
#pragma unroll
        for (int i = 0; i < kConvBatch; ++i)
            xv[i] = tb + i < t0 + n ? Io<T>::load(xp + (tb + i) * D) : 0.0f;
#pragma unroll
        for (int i = 0; i < kConvBatch; ++i) {
            float acc = bias;
#pragma unroll
            for (int k = 0; k < K - 1; ++k)
                acc = fmaf(w[k], win[k], acc);
            acc = fmaf(w[K - 1], xv[i], acc);
#pragma unroll
            for (int k = 0; k + 1 < K - 1; ++k)
                win[k] = win[k + 1];
            if (K > 1)
                win[K > 1 ? K - 2 : 0] = xv[i];
            if (tb + i < t0 + n)
                Io<T>::store(op + (tb + i) * D, a.silu ? acc * silu_gate(acc) : acc);
        }
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

// Four consecutive channels per thread (16-byte fp32 or 8-byte bf16 loads
// and stores) over a run of kConvVecRun timesteps; taken when D is a
// multiple of 4 and x and out are aligned for it. Lanes cover 4 * 32
// channels of a row. The run's inputs are loaded in batches of 16, each
// batch (with the K - 1 halo inputs for the first) issued before any of its
// outputs is computed, so a thread waits on memory twice per run. Measured
// on B300 (Bsz=2 L=2048 D=1536 K=4 fp32): 11.4 us, against 11.7 us for runs
// of 16 and 12.6 us for runs of 8 (more, shorter threads) or for batches of 8.
constexpr int kConvVecRun = 32;

template <typename T> struct Vec4;
template <> struct Vec4<float> {
    using S = float4;
    __device__ __forceinline__ static float4 load(const float *p) { return *reinterpret_cast<const float4 *>(p); }
    __device__ __forceinline__ static void store(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
};
template <> struct Vec4<__nv_bfloat16> {
    __device__ __forceinline__ static float4 load(const __nv_bfloat16 *p)
    {
        const uint2 u = *reinterpret_cast<const uint2 *>(p);
        return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                           __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
    }
    __device__ __forceinline__ static void store(__nv_bfloat16 *p, float4 v)
    {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
        uint2 u;
        u.x = *reinterpret_cast<const uint32_t *>(&lo);
        u.y = *reinterpret_cast<const uint32_t *>(&hi);
        *reinterpret_cast<uint2 *>(p) = u;
    }
};

__device__ __forceinline__ float conv_out(float acc, int silu)
{
    return silu ? acc * silu_gate(acc) : acc;
}

template <int K>
__device__ __forceinline__ float4 conv_state4(const ConvArgs &a, int64_t b, int64_t d0, int64_t tau)
{
    return make_float4(conv_state_value<K>(a, b, d0, tau), conv_state_value<K>(a, b, d0 + 1, tau),
                       conv_state_value<K>(a, b, d0 + 2, tau), conv_state_value<K>(a, b, d0 + 3, tau));
}

// Inputs loaded ahead per batch of a run, and the CTAs per SM the register
// budget of that batch (x, the filter and the window, 4 floats each, plus
// addressing) leaves room for.
__host__ __device__ constexpr int conv_vec_batch(int run) { return run < 16 ? run : 16; }
__host__ __device__ constexpr int conv_vec_min_blocks(int run, int K)
{
    return 65536 / (kConvThreads * (4 * (conv_vec_batch(run) + 2 * K) + 24)) < 1
               ? 1
               : 65536 / (kConvThreads * (4 * (conv_vec_batch(run) + 2 * K) + 24));
}

template <typename T, int K, int RUN>
__global__ void __launch_bounds__(kConvThreads, conv_vec_min_blocks(RUN, K)) conv1d_vec_kernel(const ConvArgs a)
{
    constexpr int BATCH = conv_vec_batch(RUN);
    const int64_t d0 = ((int64_t)blockIdx.x * kConvThreads + threadIdx.x) * 4;
    const int64_t b = blockIdx.y;
    const int64_t t0 = (int64_t)blockIdx.z * RUN;
    if (d0 >= a.D)
        return;
    const int64_t D = a.D, L = a.L;
    const int64_t n = L - t0 < RUN ? L - t0 : RUN;
    const T *xp = static_cast<const T *>(a.x) + b * L * D + d0;
    T *op = static_cast<T *>(a.out) + b * L * D + d0;

    float4 xb[BATCH];
#pragma unroll
    for (int i = 0; i < BATCH; ++i)
        xb[i] = i < n ? Vec4<T>::load(xp + (t0 + i) * D) : make_float4(0.f, 0.f, 0.f, 0.f);
    float4 win[K > 1 ? K - 1 : 1];
#pragma unroll
    for (int j = 0; j < K - 1; ++j) {
        const int64_t tau = t0 - (K - 1) + j;
        win[j] = tau >= 0 ? Vec4<T>::load(xp + tau * D) : conv_state4<K>(a, b, d0, tau);
    }
    float4 w[K];
#pragma unroll
    for (int k = 0; k < K; ++k)
        w[k] = make_float4(__ldg(a.w + d0 * K + k), __ldg(a.w + (d0 + 1) * K + k),
                           __ldg(a.w + (d0 + 2) * K + k), __ldg(a.w + (d0 + 3) * K + k));
    const float4 bias = a.bias ? *reinterpret_cast<const float4 *>(a.bias + d0) : make_float4(0.f, 0.f, 0.f, 0.f);

#pragma unroll 1
    for (int tb = 0; tb < RUN; tb += BATCH) {
        if (tb > 0) {
#pragma unroll
            for (int i = 0; i < BATCH; ++i)
                xb[i] = tb + i < n ? Vec4<T>::load(xp + (t0 + tb + i) * D) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < BATCH; ++i) {
            const float4 xv = xb[i];
            float4 acc = bias;
#pragma unroll
            for (int k = 0; k < K - 1; ++k) {
                acc.x = fmaf(w[k].x, win[k].x, acc.x);
                acc.y = fmaf(w[k].y, win[k].y, acc.y);
                acc.z = fmaf(w[k].z, win[k].z, acc.z);
                acc.w = fmaf(w[k].w, win[k].w, acc.w);
            }
            acc.x = fmaf(w[K - 1].x, xv.x, acc.x);
            acc.y = fmaf(w[K - 1].y, xv.y, acc.y);
            acc.z = fmaf(w[K - 1].z, xv.z, acc.z);
            acc.w = fmaf(w[K - 1].w, xv.w, acc.w);
#pragma unroll
            for (int k = 0; k + 1 < K - 1; ++k)
                win[k] = win[k + 1];
            if (K > 1)
                win[K > 1 ? K - 2 : 0] = xv;
            if (tb + i < n)
                Vec4<T>::store(op + (t0 + tb + i) * D,
                               make_float4(conv_out(acc.x, a.silu), conv_out(acc.y, a.silu), conv_out(acc.z, a.silu),
                                           conv_out(acc.w, a.silu)));
        }
    }

    if (a.state_out && t0 + n == L) {
#pragma unroll
        for (int j = 0; j < K - 1; ++j) {
            const int64_t tau = L - (K - 1) + j;
            const float4 v = tau >= 0 ? Vec4<T>::load(xp + tau * D) : conv_state4<K>(a, b, d0, tau);
            a.state_out[(b * D + d0) * (K - 1) + j] = v.x;
            a.state_out[(b * D + d0 + 1) * (K - 1) + j] = v.y;
            a.state_out[(b * D + d0 + 2) * (K - 1) + j] = v.z;
            a.state_out[(b * D + d0 + 3) * (K - 1) + j] = v.w;
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
