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

// Loads and stores of four consecutive channels (16-byte fp32 or 8-byte
// bf16), widened to fp32.
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

// Four consecutive channels per thread, taken when D is a multiple of 4 and x
// and out are aligned for vector access. The inputs stream through a
// per-thread ring of kConvRing slots in shared memory filled by cp.async:
// the thread keeps kConvRing - 1 rows in flight while it computes and stores
// the oldest, so it never waits a whole round trip between batches. Each
// thread reads back only the slots it filled itself, so the block needs no
// barrier. A CTA walks one segment of seg consecutive timesteps of one batch
// row and 4 * 128 channels; the K - 1 inputs before the segment are plain
// loads. The row loop is unrolled by four, so that the window slides by
// register renaming rather than moves. Measured on B300 (Bsz=2 L=2048 D=1536
// K=4 fp32, CUDA graph): 11.0 us with segments for three CTAs per SM (11.4 us
// without the unrolling; 11.8, 12.1 and 14.7 us for four, six and eight CTAs
// per SM), against 11.7 us for the earlier register-batched form (runs of 32
// timesteps in two batches of 16) and 9.8 us for a plain device copy of the
// same bytes.
constexpr int kConvRing = 16;
constexpr int kConvRingPerSm = 3;   // CTAs per SM the segments are sized for

template <typename T> struct RingIo;
template <> struct RingIo<float> {
    using Slot = float4;
    __device__ __forceinline__ static void copy(Slot *dst, const float *src)
    {
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                     "l"(src)
                     : "memory");
    }
    __device__ __forceinline__ static float4 get(const Slot *s) { return *s; }
};
template <> struct RingIo<__nv_bfloat16> {
    using Slot = uint2;
    __device__ __forceinline__ static void copy(Slot *dst, const __nv_bfloat16 *src)
    {
        asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                     "l"(src)
                     : "memory");
    }
    __device__ __forceinline__ static float4 get(const Slot *s)
    {
        const uint2 u = *s;
        return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                           __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
    }
};

// Launched as a programmatic dependent of the kernel before it: it may be
// scheduled while that one drains and waits for it before touching memory.
template <typename T, int K>
__global__ void __launch_bounds__(kConvThreads) conv1d_ring_kernel(const ConvArgs a, int64_t seg)
{
    using Slot = typename RingIo<T>::Slot;
    __shared__ Slot ring[kConvRing][kConvThreads];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int tid = threadIdx.x;
    const int64_t d0 = ((int64_t)blockIdx.x * kConvThreads + tid) * 4;
    const int64_t b = blockIdx.y;
    const int64_t t0 = (int64_t)blockIdx.z * seg;
    if (d0 >= a.D)
        return;
    const int64_t D = a.D, L = a.L;
    const int64_t n = L - t0 < seg ? L - t0 : seg;
    const T *xp = static_cast<const T *>(a.x) + (b * L + t0) * D + d0;
    T *op = static_cast<T *>(a.out) + (b * L + t0) * D + d0;

    // Rows 0 .. kConvRing - 2 of the segment in flight (one commit group per
    // row, empty past the segment's end).
#pragma unroll
    for (int i = 0; i < kConvRing - 1; ++i) {
        if (i < n)
            RingIo<T>::copy(&ring[i][tid], xp + i * D);
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    float4 win[K > 1 ? K - 1 : 1];
#pragma unroll
    for (int j = 0; j < K - 1; ++j) {
        const int64_t tau = t0 - (K - 1) + j;
        win[j] = tau >= 0 ? Vec4<T>::load(xp + (j - (K - 1)) * D) : conv_state4<K>(a, b, d0, tau);
    }
    float4 w[K];
#pragma unroll
    for (int k = 0; k < K; ++k)
        w[k] = make_float4(__ldg(a.w + d0 * K + k), __ldg(a.w + (d0 + 1) * K + k),
                           __ldg(a.w + (d0 + 2) * K + k), __ldg(a.w + (d0 + 3) * K + k));
    const float4 bias = a.bias ? *reinterpret_cast<const float4 *>(a.bias + d0) : make_float4(0.f, 0.f, 0.f, 0.f);

#pragma unroll 4
    for (int64_t i = 0; i < n; ++i) {
        // Row i has landed once at most kConvRing - 2 younger groups are pending.
        asm volatile("cp.async.wait_group %0;" ::"n"(kConvRing - 2) : "memory");
        const float4 xv = RingIo<T>::get(&ring[i % kConvRing][tid]);
        // The slot row i - 1 used (consumed last iteration) takes row
        // i + kConvRing - 1.
        const int64_t nx = i + kConvRing - 1;
        if (nx < n)
            RingIo<T>::copy(&ring[nx % kConvRing][tid], xp + nx * D);
        asm volatile("cp.async.commit_group;" ::: "memory");
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
        Vec4<T>::store(op + i * D, make_float4(conv_out(acc.x, a.silu), conv_out(acc.y, a.silu),
                                               conv_out(acc.z, a.silu), conv_out(acc.w, a.silu)));
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");

    if (a.state_out && t0 + n == L) {
#pragma unroll
        for (int j = 0; j < K - 1; ++j) {
            const int64_t tau = L - (K - 1) + j;
            const float4 v = tau >= 0 ? Vec4<T>::load(xp + (tau - t0) * D) : conv_state4<K>(a, b, d0, tau);
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
