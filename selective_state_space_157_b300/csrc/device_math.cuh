// device_math.cuh -- small device helpers shared by the libselscan kernels:
// element loads/stores for fp32 and bf16, the base-2 exponential on the
// MUFU unit, and softplus.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace selscan {

// log2(e): exp(v) = 2^(v * log2 e), so A is pre-scaled once per thread and
// every per-step exponential is one MUFU ex2.
constexpr float kLog2e = 1.4426950408889634f;

// 2^v on the special-function unit (PTX ex2.approx.ftz.f32: relative error
// of a few ulp; results below the normal range flush to zero).
__device__ __forceinline__ float ex2(float v)
{
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

// softplus(u) = log(1 + e^u) (booiljung.github.io, "3.1 LTI systems and
// input-dependent parameters", section 0.4.2), evaluated as
// max(u, 0) + log1p(e) with e = e^-|u| in (0, 1], so neither term overflows.
// log1p(e) = e * P(e) with P a degree-8 fit of log1p(e)/e on [0, 1]
// (derived by csrc/fit_log1p_poly.py; relative error <= 2e-7 in fp32). It
// runs on the FMA pipe: one MUFU op (the exponential) per softplus.
// Coefficients c0..c8 of P, lowest degree first.
__device__ constexpr float kLog1pPoly[9] = {9.999999404e-01f, -4.999949336e-01f, 3.331909776e-01f,
                                            -2.484298497e-01f, 1.910601407e-01f, -1.366325915e-01f,
                                            7.822608948e-02f, -2.950531431e-02f, 5.232710857e-03f};

__device__ __forceinline__ float softplus(float u)
{
    const float e = ex2(-fabsf(u) * kLog2e);
    float p = kLog1pPoly[8];
#pragma unroll
    for (int c = 7; c >= 0; --c)
        p = fmaf(p, e, kLog1pPoly[c]);
    return fmaf(p, e, fmaxf(u, 0.0f));
}

// The block's output around the scan's read-out (youngju.dev "Mamba:
// Selective State Space Models", section 3.4, the MambaBlock listing): the
// per-channel skip term dsk * x, then the gate silu(z) = z / (1 + e^-z).
// ex2 of a large positive argument gives +inf and the quotient 0, the limit.
__device__ __forceinline__ float silu(float z)
{
    return __fdividef(z, 1.0f + ex2(-z * kLog2e));
}

// sigmoid(z) = 1 / (1 + e^-z), so that silu(z) = z * silu_gate(z).
__device__ __forceinline__ float silu_gate(float z)
{
    return __fdividef(1.0f, 1.0f + ex2(-z * kLog2e));
}

__device__ __forceinline__ float block_out(float y, float dsk, float x, bool gated, float z)
{
    y = fmaf(dsk, x, y);
    return gated ? y * silu(z) : y;
}

// Zero-order-hold input coefficient (youngju.dev "Mamba: Selective State
// Space Models", section 2.2, for a diagonal A): Bbar / B = dl * phi(w) with
// phi(w) = (e^w - 1) / w and w = dl * a, given the decay e^w already
// computed. For |w| < 1/16 the difference e^w - 1 would lose digits, so phi
// comes from its series 1 + w/2 + w^2/6 + w^3/24 (truncation below
// w^4/120 < 1.3e-7, and exact at w = 0 where the limit is dl); elsewhere
// (e^w - 1) / a, where a != 0.
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float zoh_coef(float dl, float a, float decay)
{
    const float w = dl * a;
    if (fabsf(w) < 0.0625f)
        return dl * fmaf(w, fmaf(w, fmaf(w, 1.0f / 24.0f, 1.0f / 6.0f), 0.5f), 1.0f);
    return __fdividef(decay - 1.0f, a);
}

template <typename T> struct Io;

// load: read-only data (may be cached anywhere); load_cg: data written
// earlier in the same launch by another CTA (read from L2, not L1).
template <> struct Io<float> {
    __device__ __forceinline__ static float load(const float *p) { return __ldg(p); }
    __device__ __forceinline__ static float load_cg(const float *p) { return __ldcg(p); }
    __device__ __forceinline__ static void store(float *p, float v) { *p = v; }
};

template <> struct Io<__nv_bfloat16> {
    __device__ __forceinline__ static float load(const __nv_bfloat16 *p)
    {
        return __bfloat162float(__ldg(p));
    }
    __device__ __forceinline__ static float load_cg(const __nv_bfloat16 *p)
    {
        return __uint_as_float((uint32_t)__ldcg(reinterpret_cast<const unsigned short *>(p)) << 16);
    }
    __device__ __forceinline__ static void store(__nv_bfloat16 *p, float v)
    {
        *p = __float2bfloat16_rn(v);
    }
};

// Loads NS consecutive state-indexed values p[0..NS) as fp32.
// VEC: the caller guarantees p is 16-byte aligned (8-byte for 4 bf16) and
// all NS values exist. Otherwise only the first `valid` are read and the
// rest are zero.
template <typename T, int NS, bool VEC> struct StateLoad;

template <int NS> struct StateLoad<float, NS, true> {
    __device__ __forceinline__ static void run(const float *p, int, float (&v)[NS])
    {
        static_assert(NS % 4 == 0, "fp32 vector loads take 4 states");
#pragma unroll
        for (int j = 0; j < NS; j += 4) {
            float4 w = __ldg(reinterpret_cast<const float4 *>(p + j));
            v[j] = w.x; v[j + 1] = w.y; v[j + 2] = w.z; v[j + 3] = w.w;
        }
    }
};

template <int NS> struct StateLoad<__nv_bfloat16, NS, true> {
    __device__ __forceinline__ static void run(const __nv_bfloat16 *p, int, float (&v)[NS])
    {
        static_assert(NS % 4 == 0, "bf16 vector loads take 4 states");
        if constexpr (NS % 8 == 0) {
#pragma unroll
            for (int j = 0; j < NS; j += 8) {
                uint4 w = __ldg(reinterpret_cast<const uint4 *>(p + j));
                const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    v[j + 2 * i] = __uint_as_float(u[i] << 16);
                    v[j + 2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < NS; j += 4) {
                uint2 w = __ldg(reinterpret_cast<const uint2 *>(p + j));
                v[j] = __uint_as_float(w.x << 16);
                v[j + 1] = __uint_as_float(w.x & 0xffff0000u);
                v[j + 2] = __uint_as_float(w.y << 16);
                v[j + 3] = __uint_as_float(w.y & 0xffff0000u);
            }
        }
    }
};

template <typename T, int NS> struct StateLoad<T, NS, false> {
    __device__ __forceinline__ static void run(const T *p, int valid, float (&v)[NS])
    {
#pragma unroll
        for (int j = 0; j < NS; ++j)
            v[j] = (j < valid) ? Io<T>::load(p + j) : 0.0f;
    }
};

} // namespace selscan
