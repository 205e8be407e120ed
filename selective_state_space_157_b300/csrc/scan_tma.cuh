// scan_tma.cuh -- shared-memory side of the TMA-staged scan: loads of a
// timestep's B or C row (NS states, fp32 or bf16, vectorised when the row is
// 16-byte aligned and full) and of x / delta entries from the staged tiles.
#pragma once

#include "device_math.cuh"
#include "scan_fwd.cuh"
#include "tma.cuh"

namespace selscan {

constexpr int kMaxStages = 8;


template <typename T, int NS, bool VEC> struct SmemStateLoad;

template <int NS> struct SmemStateLoad<float, NS, true> {
    __device__ __forceinline__ static void run(const float *p, int, float (&v)[NS])
    {
#pragma unroll
        for (int j = 0; j < NS; j += 4) {
            const float4 w = *reinterpret_cast<const float4 *>(p + j);
            v[j] = w.x; v[j + 1] = w.y; v[j + 2] = w.z; v[j + 3] = w.w;
        }
    }
};

template <int NS> struct SmemStateLoad<__nv_bfloat16, NS, true> {
    __device__ __forceinline__ static void run(const __nv_bfloat16 *p, int, float (&v)[NS])
    {
        if constexpr (NS % 8 == 0) {
#pragma unroll
            for (int j = 0; j < NS; j += 8) {
                const uint4 w = *reinterpret_cast<const uint4 *>(p + j);
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
                const uint2 w = *reinterpret_cast<const uint2 *>(p + j);
                v[j] = __uint_as_float(w.x << 16);
                v[j + 1] = __uint_as_float(w.x & 0xffff0000u);
                v[j + 2] = __uint_as_float(w.y << 16);
                v[j + 3] = __uint_as_float(w.y & 0xffff0000u);
            }
        }
    }
};

template <typename T, int NS> struct SmemStateLoad<T, NS, false> {
    __device__ __forceinline__ static void run(const T *p, int valid, float (&v)[NS])
    {
#pragma unroll
        for (int j = 0; j < NS; ++j)
            v[j] = (j < valid) ? static_cast<float>(p[j]) : 0.0f;
    }
};

__device__ __forceinline__ float smem_val(const float *p) { return *p; }
__device__ __forceinline__ float smem_val(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

} // namespace selscan
