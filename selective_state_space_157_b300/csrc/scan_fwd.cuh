// scan_fwd.cuh -- forward selective-scan kernels.
//
// The recurrence (youngju.dev "Mamba: Selective State Space Models",
// section 3.3):  h[n] = exp(dl*A[d,n]) * h[n] + (dl*B[b,t,n]) * x[b,t,d],
// y[b,t,d] = sum_n h[n]*C[b,t,n], with dl = delta or softplus(delta).
//
// Work split. One thread owns one (b, d) chain and NS of its N states, held
// in registers for the whole chunk of timesteps it scans (NSPLIT threads
// share a chain when N > 16; their partial outputs are summed with warp
// shuffles). Lanes of a warp take consecutive channels d, so every load of
// x and delta and every store of y is one coalesced 128-byte row; B and C
// rows are the same for all lanes of a warp and arrive as broadcast vector
// loads. The (B, L, D, N) decay and input tensors of the listing are never
// formed: each exp(dl*A) lives for one FMA.
//
// Long sequences (the associative scan of booiljung.github.io "3.1 LTI
// systems ...", section 3.1.5.2). L is cut into K chunks so that enough
// chains run at once to fill the GPU:
//   1. scan_chunk_kernel<READOUT=false> reduces chunks 0..K-2 from a zero
//      state to (h_end, sum of dl), i.e. the pair (decay, offset) with
//      decay[n] = exp(A[d,n] * sum dl);
//   2. scan_carry_kernel composes the pairs, (a1,b1) o (a2,b2) =
//      (a2 a1, a2 b1 + b2), starting from h0, giving each chunk's true
//      incoming state;
//   3. scan_chunk_kernel<READOUT=true> rescans every chunk from its
//      incoming state and writes y (and hT from the last chunk).
// With K == 1 only step 3 runs, from h0.
#pragma once

#include "device_math.cuh"

namespace selscan {

constexpr int kScanThreads = 128;

struct ScanArgs {
    const void *x, *delta, *B, *C;
    const float *A;
    void *y;
    const float *Dskip;   // (D) or null: the block's skip term Dskip[d] * x
    const void *z;        // (Bsz, L, D) like x, or null: the block's gate silu(z)
    const float *h0;   // (Bsz, D, N) or null
    float *hT;         // (Bsz, D, N) or null
    float *agg_h;      // (K-1, Bsz, D, N): chunk end states from zero; overwritten by carries
    float *agg_s;      // (K-1, Bsz, D): sum of dl over each chunk
    int64_t Bsz, L, D, N;
    int64_t chunk;     // timesteps per chunk
    int K;             // number of chunks
    int dtiles;        // ceil(D / channels per CTA)
    int softplus;
    int zoh;           // zero-order-hold Bbar (zoh_coef) instead of dl * B
};

// The zero-order-hold input term of a pair of states: Bbar x with
// Bbar = zoh_coef * B, from the log2(e)-scaled A pair.
__device__ __forceinline__ float2 zoh_input(float dl, float xv, float2 A2, float2 decay, float b0, float b1)
{
    return make_float2(zoh_coef(dl, A2.x * kLn2, decay.x) * xv * b0,
                       zoh_coef(dl, A2.y * kLn2, decay.y) * xv * b1);
}

template <typename T, int NS, int NSPLIT, bool READOUT, bool VEC>
__global__ void __launch_bounds__(kScanThreads)
scan_chunk_kernel(const ScanArgs a)
{
    static_assert(NS % 2 == 0, "states are processed in pairs");
    constexpr int kChanPerCta = kScanThreads / NSPLIT;
    constexpr int NP = NS / 2;

    const int grp = threadIdx.x / NSPLIT;          // channel within the CTA
    const int q = threadIdx.x % NSPLIT;            // which NS-state slice
    const int64_t b = blockIdx.x / a.dtiles;
    const int64_t d_raw = (int64_t)(blockIdx.x % a.dtiles) * kChanPerCta + grp;
    const bool active = d_raw < a.D;
    const int64_t d = active ? d_raw : a.D - 1;    // idle lanes shadow a real channel
    const int k = blockIdx.y;
    const int64_t t0 = (int64_t)k * a.chunk;
    const int64_t t1 = min(a.L, t0 + a.chunk);
    const int n0 = q * NS;
    const int64_t left = a.N - n0;
    const int valid = left <= 0 ? 0 : (left >= NS ? NS : (int)left);
    const int64_t N = a.N, D = a.D, L = a.L;

    // A pre-scaled by log2(e), in (even, odd) pairs for the packed fp32 ops.
    float2 A2[NP];
#pragma unroll
    for (int j = 0; j < NP; ++j) {
        float lo = (2 * j < valid) ? __ldg(a.A + d * N + n0 + 2 * j) : 0.0f;
        float hi = (2 * j + 1 < valid) ? __ldg(a.A + d * N + n0 + 2 * j + 1) : 0.0f;
        A2[j] = make_float2(lo * kLog2e, hi * kLog2e);
    }

    // Incoming state.
    float2 h[NP];
    {
        const float *src = nullptr;
        if (READOUT) {
            if (k > 0)
                src = a.agg_h + (((int64_t)(k - 1) * a.Bsz + b) * D + d) * N + n0;
            else if (a.h0)
                src = a.h0 + (b * D + d) * N + n0;
        }
#pragma unroll
        for (int j = 0; j < NP; ++j) {
            float lo = (src && 2 * j < valid) ? src[2 * j] : 0.0f;
            float hi = (src && 2 * j + 1 < valid) ? src[2 * j + 1] : 0.0f;
            h[j] = make_float2(lo, hi);
        }
    }

    const T *xp = static_cast<const T *>(a.x) + (b * L + t0) * D + d;
    const T *dp = static_cast<const T *>(a.delta) + (b * L + t0) * D + d;
    const T *Bp = static_cast<const T *>(a.B) + (b * L + t0) * N + n0;
    const T *Cp = static_cast<const T *>(a.C) + (b * L + t0) * N + n0;
    T *yp = static_cast<T *>(a.y) + (b * L + t0) * D + d;
    const T *zp = a.z ? static_cast<const T *>(a.z) + (b * L + t0) * D + d : nullptr;
    const bool block = READOUT && (a.Dskip || a.z);
    const float dsk = (READOUT && a.Dskip) ? __ldg(a.Dskip + d) : 0.0f;

    float s = 0.0f, s_err = 0.0f;   // compensated sum of dl (aggregate pass)

#pragma unroll 2
    for (int64_t t = t0; t < t1; ++t) {
        float dl = Io<T>::load(dp);
        const float xv = Io<T>::load(xp);
        if (a.softplus)
            dl = softplus(dl);
        const float u = dl * xv;
        float Bv[NS];
        StateLoad<T, NS, VEC>::run(Bp, valid, Bv);
        const float2 dl2 = make_float2(dl, dl);
        const float2 u2 = make_float2(u, u);
        if (READOUT) {
            float Cv[NS];
            StateLoad<T, NS, VEC>::run(Cp, valid, Cv);
            float2 acc0 = make_float2(0.0f, 0.0f), acc1 = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int j = 0; j < NP; ++j) {
                const float2 e = __fmul2_rn(dl2, A2[j]);
                const float2 decay = make_float2(ex2(e.x), ex2(e.y));
                const float2 inp = a.zoh ? zoh_input(dl, xv, A2[j], decay, Bv[2 * j], Bv[2 * j + 1])
                                         : __fmul2_rn(u2, make_float2(Bv[2 * j], Bv[2 * j + 1]));
                h[j] = __ffma2_rn(decay, h[j], inp);
                const float2 c = make_float2(Cv[2 * j], Cv[2 * j + 1]);
                if (j & 1)
                    acc1 = __ffma2_rn(h[j], c, acc1);
                else
                    acc0 = __ffma2_rn(h[j], c, acc0);
            }
            float yv = (acc0.x + acc0.y) + (acc1.x + acc1.y);
#pragma unroll
            for (int o = NSPLIT / 2; o > 0; o >>= 1)
                yv += __shfl_xor_sync(0xffffffffu, yv, o);
            if (block) {
                yv = block_out(yv, dsk, xv, zp != nullptr, zp ? Io<T>::load(zp) : 0.0f);
                if (zp) zp += D;
            }
            if (active && q == 0)
                Io<T>::store(yp, yv);
            Cp += N;
            yp += D;
        } else {
#pragma unroll
            for (int j = 0; j < NP; ++j) {
                const float2 e = __fmul2_rn(dl2, A2[j]);
                const float2 decay = make_float2(ex2(e.x), ex2(e.y));
                const float2 inp = a.zoh ? zoh_input(dl, xv, A2[j], decay, Bv[2 * j], Bv[2 * j + 1])
                                         : __fmul2_rn(u2, make_float2(Bv[2 * j], Bv[2 * j + 1]));
                h[j] = __ffma2_rn(decay, h[j], inp);
            }
            // Kahan summation keeps sum(dl) to fp32 rounding over long chunks.
            const float yk = dl - s_err;
            const float tk = s + yk;
            s_err = (tk - s) - yk;
            s = tk;
        }
        xp += D;
        dp += D;
        Bp += N;
    }

    if (!active)
        return;
    float *dst = nullptr;
    if (READOUT) {
        if (k == a.K - 1 && a.hT)
            dst = a.hT + (b * D + d) * N + n0;
    } else {
        dst = a.agg_h + (((int64_t)k * a.Bsz + b) * D + d) * N + n0;
        if (q == 0)
            a.agg_s[((int64_t)k * a.Bsz + b) * D + d] = s;
    }
    if (dst) {
#pragma unroll
        for (int j = 0; j < NP; ++j) {
            if (2 * j < valid) dst[2 * j] = h[j].x;
            if (2 * j + 1 < valid) dst[2 * j + 1] = h[j].y;
        }
    }
}

} // namespace selscan
