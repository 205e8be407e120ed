// fwd_fused_impl.cuh -- instantiation and launch description of the
// persistent forward kernel (scan_fused.cuh) for one element type and
// either form (one pass, or chunked); included by the four fwd_fused_*.cu
// units, which compile in parallel.
#pragma once

#include <mutex>

#include "launch.h"

namespace selscan {
namespace {

constexpr int kTT = 16;   // timesteps per pipeline stage

// Resident CTAs per SM for a kernel at a shared-memory size (cached).
int occupancy(const void *fn, int threads, size_t smem)
{
    struct Entry { const void *fn; size_t smem; int n; };
    static std::mutex mu;
    static Entry cache[64];
    static int used = 0;
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < used; ++i)
        if (cache[i].fn == fn && cache[i].smem == smem) return cache[i].n;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem) != cudaSuccess) {
        cudaGetLastError();
        n = 1;
    }
    if (n < 1) n = 1;
    if (used < 64) cache[used++] = Entry{fn, smem, n};
    return n;
}

template <typename T, bool CH, int NS, int NSPLIT, bool VEC, bool SP, bool GATE = false, bool ZOH = false>
bool prepare_fused_sp(int64_t N, int stages, FusedLaunch *out)
{
    constexpr int THREADS = fused_threads(CH, NSPLIT);
    constexpr int DPB = THREADS / NSPLIT;
    auto k = scan_fused_kernel<T, NS, NSPLIT, VEC, kTT, SP, GATE, ZOH, CH, THREADS>;
    const int64_t nrow = VEC ? NS * NSPLIT : N;
    const size_t smem = fused_smem_bytes(sizeof(T), kTT, DPB, nrow, stages, GATE, NSPLIT);
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    const void *fn = reinterpret_cast<const void *>(k);
    *out = FusedLaunch{fn, smem, occupancy(fn, THREADS, smem), kTT, stages, THREADS, DPB > 256 ? DPB / 2 : DPB};
    return true;
}

// The block's skip and gate run fused on the vectorised, softplus form (the
// block's own use); other gated forms take the plain-load path. So does the
// zero-order hold, for one thread per chain (N <= 16).
template <typename T, bool CH, int NS, int NSPLIT>
bool prepare_fused(bool vec, bool softplus, bool gate, bool zoh, int64_t N, int stages, FusedLaunch *out)
{
    if (zoh) {
        if constexpr (NSPLIT == 1) {
            if (!(vec && softplus)) return false;
            return gate ? prepare_fused_sp<T, CH, NS, NSPLIT, true, true, true, true>(N, stages, out)
                        : prepare_fused_sp<T, CH, NS, NSPLIT, true, true, false, true>(N, stages, out);
        }
        return false;
    }
    if (gate)
        return vec && softplus && prepare_fused_sp<T, CH, NS, NSPLIT, true, true, true>(N, stages, out);
    if (vec)
        return softplus ? prepare_fused_sp<T, CH, NS, NSPLIT, true, true>(N, stages, out)
                        : prepare_fused_sp<T, CH, NS, NSPLIT, true, false>(N, stages, out);
    return softplus ? prepare_fused_sp<T, CH, NS, NSPLIT, false, true>(N, stages, out)
                    : prepare_fused_sp<T, CH, NS, NSPLIT, false, false>(N, stages, out);
}

template <typename T, bool CH>
bool pick_fused(int ns, int nsplit, bool vec, bool softplus, bool gate, bool zoh, int64_t N, int stages,
                FusedLaunch *out)
{
    if (stages < 2) stages = 2;
    if (stages > kMaxStages) stages = kMaxStages;
    switch (ns * 100 + nsplit) {
    case 401: return prepare_fused<T, CH, 4, 1>(vec, softplus, gate, zoh, N, stages, out);
    case 801: return prepare_fused<T, CH, 8, 1>(vec, softplus, gate, zoh, N, stages, out);
    case 1601: return prepare_fused<T, CH, 16, 1>(vec, softplus, gate, zoh, N, stages, out);
    case 1602: return prepare_fused<T, CH, 16, 2>(vec, softplus, gate, zoh, N, stages, out);
    case 1604: return prepare_fused<T, CH, 16, 4>(vec, softplus, gate, zoh, N, stages, out);
    case 802: return prepare_fused<T, CH, 8, 2>(vec, softplus, gate, zoh, N, stages, out);
    case 404: return prepare_fused<T, CH, 4, 4>(vec, softplus, gate, zoh, N, stages, out);
    default: return false;
    }
}

} // namespace
} // namespace selscan
