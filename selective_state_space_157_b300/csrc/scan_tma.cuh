// scan_tma.cuh -- the forward scan with its inputs staged through shared
// memory by TMA.
//
// Same work split and arithmetic as scan_chunk_kernel (scan_fwd.cuh): one
// thread per (b, d) chain and NS of its states in registers, lanes over
// consecutive channels. What changes is how inputs arrive. A CTA covers
// DPB = 128 / NSPLIT channels of one batch row over one chunk of timesteps;
// the chunk is consumed in stages of TT timesteps. For each stage one
// elected thread issues 3-D TMA boxes for
//     x, delta : TT x DPB   (rows t, columns d)
//     B (, C)  : TT x N
// into one of STAGES shared-memory buffers, completing on an mbarrier with
// the expected byte count. Threads wait on that barrier, run TT steps of the
// recurrence reading x/delta with conflict-free 4-byte loads and B/C rows
// with broadcast 16-byte loads, and release the buffer. The last warp to
// release a buffer refills it with the stage STAGES ahead, so loads run
// STAGES * TT timesteps ahead of the arithmetic and no thread waits for
// another to finish reading. Boxes that run past D or L are zero-filled by
// the TMA unit; those lanes and rows are never stored.
#pragma once

#include "device_math.cuh"
#include "scan_fwd.cuh"
#include "tma.cuh"

namespace selscan {

constexpr int kMaxStages = 8;

struct TmaScanArgs {
    CUtensorMap mx, md, mB, mC;   // 3-D maps: (D, L, Bsz) for x/delta, (N, L, Bsz) for B/C
    ScanArgs s;
    int stages;                   // shared-memory buffers in flight (2..kMaxStages)
};

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

// Dynamic shared memory of one CTA: STAGES buffers of x, delta, B (and C)
// tiles, then per buffer an mbarrier and two counters.
inline size_t tma_smem_bytes(size_t es, int TT, int DPB, int64_t N, bool with_C, int stages)
{
    const size_t stage = (2 * (size_t)TT * DPB + (with_C ? 2 : 1) * (size_t)TT * (size_t)N) * es;
    return (size_t)stages * stage + (size_t)stages * (8 + 4 + 4);
}

template <typename T, int NS, int NSPLIT, bool READOUT, bool VEC, int TT>
__global__ void __launch_bounds__(kScanThreads)
scan_tma_kernel(const __grid_constant__ TmaScanArgs ta)
{
    static_assert(NS % 2 == 0, "states are processed in pairs");
    constexpr int DPB = kScanThreads / NSPLIT;
    constexpr int NP = NS / 2;
    constexpr int kWarps = kScanThreads / 32;
    const ScanArgs &a = ta.s;
    const int STAGES = ta.stages;

    extern __shared__ __align__(128) unsigned char smem[];
    const int64_t N = a.N, D = a.D, L = a.L;
    const int xbytes = TT * DPB * (int)sizeof(T);
    const int nbytes = TT * (int)N * (int)sizeof(T);
    const int sbytes = 2 * xbytes + (READOUT ? 2 : 1) * nbytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * sbytes);
    unsigned *drained = reinterpret_cast<unsigned *>(full + STAGES);   // warps done with the buffer
    unsigned *issued = drained + STAGES;                                // fills issued into the buffer

    const int grp = threadIdx.x / NSPLIT;
    const int q = threadIdx.x % NSPLIT;
    const int lane = threadIdx.x & 31;
    const int64_t b = blockIdx.x / a.dtiles;
    const int d0 = (blockIdx.x % a.dtiles) * DPB;
    const int64_t d_raw = (int64_t)d0 + grp;
    const bool active = d_raw < D;
    const int64_t d = active ? d_raw : D - 1;
    const int k = blockIdx.y;
    const int64_t t0 = (int64_t)k * a.chunk;
    const int64_t nsteps = min(L, t0 + a.chunk) - t0;
    const int nst = (int)((nsteps + TT - 1) / TT);
    const int n0 = q * NS;
    const int64_t left = N - n0;
    const int valid = left <= 0 ? 0 : (left >= NS ? NS : (int)left);

    auto stage_x = [&](int s) { return reinterpret_cast<T *>(smem + s * sbytes); };
    auto stage_d = [&](int s) { return reinterpret_cast<T *>(smem + s * sbytes + xbytes); };
    auto stage_B = [&](int s) { return reinterpret_cast<T *>(smem + s * sbytes + 2 * xbytes); };
    auto stage_C = [&](int s) { return reinterpret_cast<T *>(smem + s * sbytes + 2 * xbytes + nbytes); };
    auto issue = [&](int s, int i) {
        const int t = (int)(t0 + (int64_t)i * TT);
        issued[s] += 1;
        mbar_arrive_expect_tx(&full[s], (uint32_t)sbytes);
        tma_load_3d(stage_x(s), &ta.mx, &full[s], d0, t, (int)b);
        tma_load_3d(stage_d(s), &ta.md, &full[s], d0, t, (int)b);
        tma_load_3d(stage_B(s), &ta.mB, &full[s], 0, t, (int)b);
        if (READOUT)
            tma_load_3d(stage_C(s), &ta.mC, &full[s], 0, t, (int)b);
    };

    if (threadIdx.x == 0) {
        prefetch_tensormap(&ta.mx);
        prefetch_tensormap(&ta.md);
        prefetch_tensormap(&ta.mB);
        if (READOUT)
            prefetch_tensormap(&ta.mC);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            drained[s] = 0;
            issued[s] = 0;
        }
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0)
        for (int s = 0; s < STAGES && s < nst; ++s)
            issue(s, s);

    float2 A2[NP];
#pragma unroll
    for (int j = 0; j < NP; ++j) {
        const float lo = (2 * j < valid) ? __ldg(a.A + d * N + n0 + 2 * j) : 0.0f;
        const float hi = (2 * j + 1 < valid) ? __ldg(a.A + d * N + n0 + 2 * j + 1) : 0.0f;
        A2[j] = make_float2(lo * kLog2e, hi * kLog2e);
    }
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
            const float lo = (src && 2 * j < valid) ? src[2 * j] : 0.0f;
            const float hi = (src && 2 * j + 1 < valid) ? src[2 * j + 1] : 0.0f;
            h[j] = make_float2(lo, hi);
        }
    }

    T *yp = static_cast<T *>(a.y) + (b * L + t0) * D + d;
    float s_sum = 0.0f, s_err = 0.0f;
    bool ok = true;

    for (int i = 0; i < nst; ++i) {
        const int s = i % STAGES;
        const bool arrived = mbar_wait(&full[s], (uint32_t)((i / STAGES) & 1));
        if (!__all_sync(0xffffffffu, arrived)) {   // leave the loop as a whole warp
            ok = false;
            break;
        }
        const T *xs = stage_x(s) + grp;
        const T *ds = stage_d(s) + grp;
        const T *Bs = stage_B(s) + n0;
        const T *Cs = stage_C(s) + n0;
        const int64_t rem = nsteps - (int64_t)i * TT;
        const int tc = rem < TT ? (int)rem : TT;

        // Phase 1: the per-timestep scalars of the whole stage (independent
        // across timesteps, so their latency overlaps): dl and u = dl * x.
        float dlv[TT], uv[TT];
#pragma unroll
        for (int tt = 0; tt < TT; ++tt) {
            float dl = smem_val(ds + tt * DPB);
            if (a.softplus)
                dl = softplus(dl);
            dlv[tt] = dl;
            uv[tt] = dl * smem_val(xs + tt * DPB);
        }
        if (!READOUT) {
#pragma unroll
            for (int tt = 0; tt < TT; ++tt) {
                if (tt < tc) {   // Kahan summation keeps sum(dl) to fp32 rounding
                    const float yk = dlv[tt] - s_err;
                    const float tk = s_sum + yk;
                    s_err = (tk - s_sum) - yk;
                    s_sum = tk;
                }
            }
        }

        // Phase 2: the recurrence; only h carries a dependence between steps.
        auto step = [&](int tt) {
            float Bv[NS];
            SmemStateLoad<T, NS, VEC>::run(Bs + tt * N, valid, Bv);
            const float2 dl2 = make_float2(dlv[tt], dlv[tt]);
            const float2 u2 = make_float2(uv[tt], uv[tt]);
            if (READOUT) {
                float Cv[NS];
                SmemStateLoad<T, NS, VEC>::run(Cs + tt * N, valid, Cv);
                float2 acc0 = make_float2(0.0f, 0.0f), acc1 = make_float2(0.0f, 0.0f);
#pragma unroll
                for (int j = 0; j < NP; ++j) {
                    const float2 e = __fmul2_rn(dl2, A2[j]);
                    const float2 decay = make_float2(ex2(e.x), ex2(e.y));
                    const float2 inp = __fmul2_rn(u2, make_float2(Bv[2 * j], Bv[2 * j + 1]));
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
                if (active && q == 0)
                    Io<T>::store(yp + tt * D, yv);
            } else {
#pragma unroll
                for (int j = 0; j < NP; ++j) {
                    const float2 e = __fmul2_rn(dl2, A2[j]);
                    const float2 decay = make_float2(ex2(e.x), ex2(e.y));
                    const float2 inp = __fmul2_rn(u2, make_float2(Bv[2 * j], Bv[2 * j + 1]));
                    h[j] = __ffma2_rn(decay, h[j], inp);
                }
            }
        };
        if (tc == TT) {
#pragma unroll
            for (int tt = 0; tt < TT; ++tt)
                step(tt);
        } else {
#pragma unroll
            for (int tt = 0; tt < TT; ++tt)
                if (tt < tc)
                    step(tt);
        }
        if (READOUT)
            yp += (int64_t)TT * D;

        // Release the buffer; the last warp out refills it STAGES stages ahead.
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            const unsigned prev = atomicAdd(&drained[s], 1u);
            if (prev == kWarps - 1) {
                drained[s] = 0;
                __threadfence_block();
                if (i + STAGES < nst) {
                    fence_proxy_async_smem();
                    issue(s, i + STAGES);
                }
            }
        }
    }

    // A tile that never arrived: every warp leaves its loop (each wait is
    // bounded), then the copies this CTA issued are allowed to land before
    // its shared memory is released (again bounded) and the fault is recorded.
    if (__syncthreads_or(!ok)) {
        if (threadIdx.x == 0) {
            record_fault(kFaultTmaTimeout);
            for (int s = 0; s < STAGES; ++s)
                if (issued[s] > 0)
                    mbar_wait(&full[s], (issued[s] - 1) & 1u);
        }
        return;
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
            a.agg_s[((int64_t)k * a.Bsz + b) * D + d] = s_sum;
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
