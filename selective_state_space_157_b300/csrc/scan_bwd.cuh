// scan_bwd.cuh -- the backward pass of the selective scan (fp32).
//
// The hardware-aware design of booiljung.github.io "3.1 LTI systems and
// input-dependent parameters", section 3.1.5.3, trains through the scan by
// recomputing the states in the backward pass instead of storing them. The
// pages give no gradient formulas; these are the chain rule applied to the
// recurrence h_t = a_t h_{t-1} + dl_t B_t x_t, a_t = exp(dl_t A), y_t =
// sum_n h_t C_t. With g_t = dLoss/dh_t (the adjoint, carried backwards as
// g_t = gy_t C_t + a_{t+1} g_{t+1}, starting from dLoss/dhT):
//   dC_t += gy_t h_t                dB_t += g_t dl_t x_t
//   dx_t  = sum_n g_t dl_t B_t      dA   += g_t h_{t-1} a_t dl_t
//   d dl_t = sum_n (g_t h_{t-1} a_t A + g_t B_t x_t),  times sigmoid(u)
//            when dl = softplus(u)
//   dh0   = a_0 g_0.
//
// Layout of the work. One chain (b, d) is P lanes (P = the power of two
// >= N, at most 32), one state index n per lane, so the sums over n are
// shuffles within the lane group and the state of a whole chunk fits in
// registers. A block is kBwdThreads lanes = cpb chains of one batch row b.
//   1. A forward pass over L writes the state at the start of every chunk of
//      kBwdT steps to a workspace (b, chunk, d, n).
//   2. The chunks are then taken last to first: the chunk's states and decays
//      are recomputed from its checkpoint into registers, and the adjoint runs
//      backwards through them.
// Per-timestep inputs of a chunk are loaded by the whole block with
// coalesced loads (one row of cpb channels per step) into registers one
// chunk ahead, then staged in shared memory. Each lane keeps its dx and
// d delta terms for the chunk's steps; one reduce-scatter over the lane group
// per chunk leaves every lane with whole steps to store. dB and dC are summed
// over the chains of a warp with shuffles, over the warps in shared memory,
// and added to global memory with one atomic per block, timestep and state;
// dA is summed over t in registers and added with one atomic per chain.
// Chunks that lie wholly inside L run without per-step bounds checks.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "device_math.cuh"

namespace selscan {

// 128-lane blocks with 32-step chunks: fewer, longer chunks amortise the
// per-chunk barriers, staging latency and atomics, and three blocks fit on
// an SM at N = 16 (measured on B300 for the 130M-like layer: 0.384 ms per
// call, against 0.418 ms for 16-step chunks and 0.476 ms for 16-step chunks
// in 256-lane blocks).
constexpr int kBwdThreads = 128;
constexpr int kBwdWarps = kBwdThreads / 32;
constexpr int kBwdT = 32;      // timesteps per chunk (registers per lane: about 2 * kBwdT)

struct BwdArgs {
    const float *x, *delta, *A, *B, *C, *h0, *gy, *ghT;
    float *dx, *ddelta, *dA, *dB, *dC, *dh0;
    float *ckpt;               // (Bsz, nch, D, P) chunk-start states
    int64_t Bsz, L, D, N;
    int64_t nch;               // chunks of kBwdT steps
    int P;                     // lanes per chain: power of two >= N, <= 32
    int cpb;                   // chains per block = kBwdThreads / P
    int softplus;
};

// Shared memory of one block, in floats.
__host__ __device__ constexpr int64_t bwd_smem_floats(int P, int cpb)
{
    return 4 * int64_t(kBwdT) * cpb + 2 * int64_t(kBwdT) * P + 2 * int64_t(kBwdT) * kBwdWarps * P;
}

// sigmoid(u) = d softplus(u) / du. ex2 of a large argument gives +inf and
// the quotient 0, the limit.
__device__ __forceinline__ float bwd_sigmoid(float u)
{
    return 1.0f / (1.0f + ex2(-u * kLog2e));
}

// The raw per-timestep inputs of one chunk that this thread stages: it loads
// them into registers one chunk ahead, so the loads are in flight while the
// block works on the current chunk. Element j = threadIdx.x + r * kBwdThreads
// of the chunk's (step, channel) rows and (step, state) rows.
template <int P> struct BwdChunkRegs {
    static constexpr int CPB = kBwdThreads / P;
    static constexpr int RX = (kBwdT * CPB + kBwdThreads - 1) / kBwdThreads;
    static constexpr int RB = (kBwdT * P + kBwdThreads - 1) / kBwdThreads;
    float x[RX], u[RX], gy[RX], B[RB], C[RB];
};

// Loads chunk t0 .. t0 + kBwdT of batch row b for channels d0 .. d0 + CPB
// (zeros beyond L, D and N). ADJ: also gy and C (the adjoint pass).
template <int P, bool ADJ>
__device__ __forceinline__ void bwd_load(const BwdArgs &a, int64_t b, int64_t d0, int64_t t0, BwdChunkRegs<P> &r)
{
    using R = BwdChunkRegs<P>;
#pragma unroll
    for (int q = 0; q < R::RX; ++q) {
        const int j = threadIdx.x + q * kBwdThreads;
        const int i = j / R::CPB, c = j % R::CPB;
        const bool ok = j < kBwdT * R::CPB && t0 + i < a.L && d0 + c < a.D;
        const int64_t idx = (b * a.L + t0 + i) * a.D + d0 + c;
        r.x[q] = ok ? __ldg(a.x + idx) : 0.0f;
        r.u[q] = ok ? __ldg(a.delta + idx) : 0.0f;
        if (ADJ)
            r.gy[q] = ok ? __ldg(a.gy + idx) : 0.0f;
    }
#pragma unroll
    for (int q = 0; q < R::RB; ++q) {
        const int j = threadIdx.x + q * kBwdThreads;
        const int i = j / P, m = j % P;
        const bool ok = j < kBwdT * P && t0 + i < a.L && m < a.N;
        const int64_t idx = (b * a.L + t0 + i) * a.N + m;
        r.B[q] = ok ? __ldg(a.B + idx) : 0.0f;
        if (ADJ)
            r.C[q] = ok ? __ldg(a.C + idx) : 0.0f;
    }
}

// Writes loaded inputs to the block's staging rows, with dl = softplus(u)
// and its derivative when asked.
template <int P, bool ADJ>
__device__ __forceinline__ void bwd_put(const BwdArgs &a, const BwdChunkRegs<P> &r, float *s_x, float *s_dl,
                                        float *s_sg, float *s_gy, float *s_B, float *s_C)
{
    using R = BwdChunkRegs<P>;
#pragma unroll
    for (int q = 0; q < R::RX; ++q) {
        const int j = threadIdx.x + q * kBwdThreads;
        if (j < kBwdT * R::CPB) {
            s_x[j] = r.x[q];
            s_dl[j] = a.softplus ? softplus(r.u[q]) : r.u[q];
            if (ADJ) {
                s_sg[j] = a.softplus ? bwd_sigmoid(r.u[q]) : 1.0f;
                s_gy[j] = r.gy[q];
            }
        }
    }
#pragma unroll
    for (int q = 0; q < R::RB; ++q) {
        const int j = threadIdx.x + q * kBwdThreads;
        if (j < kBwdT * P) {
            s_B[j] = r.B[q];
            if (ADJ)
                s_C[j] = r.C[q];
        }
    }
}

// Reduce-scatter of v[0 .. T) over the P lanes of a lane group (recursive
// halving). Lane n of the group ends with, for P <= T, the sums of entries
// n*T/P .. (n+1)*T/P - 1 in v[0 .. T/P); for P > T, the sum of entry
// n / (P/T) in v[0].
template <int O, int M, int T> struct GroupReduceScatter {
    __device__ __forceinline__ static void run(float (&v)[T], int n)
    {
        if constexpr (O >= 1) {
            if constexpr (M > 1) {
                const bool up = (n & O) != 0;
#pragma unroll
                for (int j = 0; j < M / 2; ++j) {
                    const float keep = up ? v[j + M / 2] : v[j];
                    const float send = up ? v[j] : v[j + M / 2];
                    v[j] = keep + __shfl_xor_sync(0xffffffffu, send, O);
                }
                GroupReduceScatter<O / 2, M / 2, T>::run(v, n);
            } else {
                v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
                GroupReduceScatter<O / 2, 1, T>::run(v, n);
            }
        }
    }
};

// The state recurrence over one staged chunk (forward pass).
template <int P, bool TAIL>
__device__ __forceinline__ float bwd_fwd_chunk(float h, float A2, int64_t t0, int64_t L, int n, int c,
                                               const float *s_x, const float *s_dl, const float *s_B)
{
    constexpr int CPB = kBwdThreads / P;
#pragma unroll
    for (int i = 0; i < kBwdT; ++i) {
        if (!TAIL || t0 + i < L) {
            const float dl = s_dl[i * CPB + c];
            h = fmaf(ex2(dl * A2), h, dl * s_B[i * P + n] * s_x[i * CPB + c]);
        }
    }
    return h;
}

// One staged chunk of the adjoint pass: recompute its states and decays from
// hs, run the adjoint g back through them, write dx and d delta, leave the
// chain-group sums of the dB and dC terms in s_pB / s_pC, and return the
// chunk's dA term.
template <int P, bool TAIL>
__device__ __forceinline__ float bwd_adj_chunk(const BwdArgs &a, float &g, float hs, float An, float A2,
                                               int64_t b, int64_t d, bool chain, int64_t t0, int n, int c,
                                               int lane, int warp, const float *s_x, const float *s_dl,
                                               const float *s_sg, const float *s_gy, const float *s_B,
                                               const float *s_C, float *s_pB, float *s_pC)
{
    constexpr int CPB = kBwdThreads / P;
    const int64_t L = a.L;
    float hc[kBwdT], ac[kBwdT];
    float hh = hs;
#pragma unroll
    for (int i = 0; i < kBwdT; ++i) {
        hc[i] = 0.0f;
        ac[i] = 1.0f;
        if (!TAIL || t0 + i < L) {
            const float dl = s_dl[i * CPB + c];
            const float av = ex2(dl * A2);
            hh = fmaf(av, hh, dl * s_B[i * P + n] * s_x[i * CPB + c]);
            hc[i] = hh;
            ac[i] = av;
        }
    }

    float gx[kBwdT], gdl[kBwdT];
    float dAk = 0.0f;
#pragma unroll
    for (int i = kBwdT - 1; i >= 0; --i) {
        gx[i] = 0.0f;
        gdl[i] = 0.0f;
        if (!TAIL || t0 + i < L) {                 // uniform over the block
            const float dl = s_dl[i * CPB + c], xv = s_x[i * CPB + c], gyv = s_gy[i * CPB + c];
            const float Bn = s_B[i * P + n], Cn = s_C[i * P + n];
            g = fmaf(gyv, Cn, g);                          // y_t reads h_t
            float pC = gyv * hc[i];
            const float hp = i > 0 ? hc[i - 1] : hs;       // h_{t-1}
            const float dan = g * hp * ac[i];
            gdl[i] = fmaf(dan, An, g * Bn * xv);
            dAk = fmaf(dan, dl, dAk);
            float pB = g * dl * xv;
            gx[i] = g * dl * Bn;
            g *= ac[i];                                    // into h_{t-1}
#pragma unroll
            for (int off = P; off < 32; off <<= 1) {
                pB += __shfl_xor_sync(0xffffffffu, pB, off);
                pC += __shfl_xor_sync(0xffffffffu, pC, off);
            }
            if (lane < P) {
                s_pB[(i * kBwdWarps + warp) * P + lane] = pB;
                s_pC[(i * kBwdWarps + warp) * P + lane] = pC;
            }
        }
    }

    // dx and d delta: sums over the P states of the chain, one step per lane
    GroupReduceScatter<P / 2, kBwdT, kBwdT>::run(gx, n);
    GroupReduceScatter<P / 2, kBwdT, kBwdT>::run(gdl, n);
    if constexpr (P <= kBwdT) {
        constexpr int S = kBwdT / P;
#pragma unroll
        for (int q = 0; q < S; ++q) {
            const int i = n * S + q;
            if (chain && (!TAIL || t0 + i < L)) {
                const int64_t idx = (b * L + t0 + i) * a.D + d;
                a.dx[idx] = gx[q];
                a.ddelta[idx] = gdl[q] * s_sg[i * CPB + c];
            }
        }
    } else {
        constexpr int R = P / kBwdT;
        const int i = n / R;
        if (chain && n % R == 0 && (!TAIL || t0 + i < L)) {
            const int64_t idx = (b * L + t0 + i) * a.D + d;
            a.dx[idx] = gx[0];
            a.ddelta[idx] = gdl[0] * s_sg[i * CPB + c];
        }
    }
    return dAk;
}

// grid (ceil(D / CPB), Bsz), kBwdThreads threads,
// bwd_smem_floats(P, CPB) * 4 bytes of dynamic shared memory.
// dA, dB and dC must be zero on entry (they are accumulated atomically).
template <int P>
__global__ void __launch_bounds__(kBwdThreads) scan_bwd_kernel(BwdArgs a)
{
    constexpr int CPB = kBwdThreads / P;
    extern __shared__ float bwd_smem[];
    float *s_x = bwd_smem;
    float *s_dl = s_x + kBwdT * CPB;
    float *s_sg = s_dl + kBwdT * CPB;
    float *s_gy = s_sg + kBwdT * CPB;
    float *s_B = s_gy + kBwdT * CPB;
    float *s_C = s_B + kBwdT * P;
    float *s_pB = s_C + kBwdT * P;              // [kBwdT][kBwdWarps][P]
    float *s_pC = s_pB + kBwdT * kBwdWarps * P;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = tid % P, c = tid / P;
    const int64_t b = blockIdx.y;
    const int64_t d0 = int64_t(blockIdx.x) * CPB, d = d0 + c;
    const bool chain = d < a.D;                 // this lane's chain exists
    const bool act = chain && n < a.N;          // ... and its state index too
    const int64_t L = a.L, D = a.D, N = a.N, nch = a.nch;

    const float An = act ? __ldg(a.A + d * N + n) : 0.0f;
    const float A2 = An * kLog2e;
    BwdChunkRegs<P> r;

    // 1. forward pass: the state at the start of every chunk
    float h = (act && a.h0) ? __ldg(a.h0 + (b * D + d) * N + n) : 0.0f;
    bwd_load<P, false>(a, b, d0, 0, r);
    for (int64_t k = 0; k < nch; ++k) {
        const int64_t t0 = k * kBwdT;
        bwd_put<P, false>(a, r, s_x, s_dl, s_sg, s_gy, s_B, s_C);
        if (chain)
            a.ckpt[((b * nch + k) * D + d) * P + n] = h;
        if (k + 1 < nch)
            bwd_load<P, false>(a, b, d0, t0 + kBwdT, r);
        __syncthreads();
        if (t0 + kBwdT <= L)
            h = bwd_fwd_chunk<P, false>(h, A2, t0, L, n, c, s_x, s_dl, s_B);
        else
            h = bwd_fwd_chunk<P, true>(h, A2, t0, L, n, c, s_x, s_dl, s_B);
        __syncthreads();
    }

    // 2. the chunks last to first: recompute, then run the adjoint back
    float g = (act && a.ghT) ? __ldg(a.ghT + (b * D + d) * N + n) : 0.0f;
    float dAacc = 0.0f;
    bwd_load<P, true>(a, b, d0, (nch - 1) * kBwdT, r);
    float hs_next = chain ? a.ckpt[((b * nch + nch - 1) * D + d) * P + n] : 0.0f;
    for (int64_t k = nch - 1; k >= 0; --k) {
        const int64_t t0 = k * kBwdT;
        bwd_put<P, true>(a, r, s_x, s_dl, s_sg, s_gy, s_B, s_C);
        const float hs = hs_next;
        if (k > 0) {
            bwd_load<P, true>(a, b, d0, t0 - kBwdT, r);
            hs_next = chain ? a.ckpt[((b * nch + k - 1) * D + d) * P + n] : 0.0f;
        }
        __syncthreads();
        if (t0 + kBwdT <= L)
            dAacc += bwd_adj_chunk<P, false>(a, g, hs, An, A2, b, d, chain, t0, n, c, lane, warp, s_x, s_dl, s_sg,
                                             s_gy, s_B, s_C, s_pB, s_pC);
        else
            dAacc += bwd_adj_chunk<P, true>(a, g, hs, An, A2, b, d, chain, t0, n, c, lane, warp, s_x, s_dl, s_sg,
                                            s_gy, s_B, s_C, s_pB, s_pC);
        __syncthreads();
        for (int j = tid; j < kBwdT * N; j += kBwdThreads) {
            const int i = j / int(N), m = j - i * int(N);
            const int64_t t = t0 + i;
            if (t < L) {
                float sB = 0.0f, sC = 0.0f;
#pragma unroll
                for (int w = 0; w < kBwdWarps; ++w) {
                    sB += s_pB[(i * kBwdWarps + w) * P + m];
                    sC += s_pC[(i * kBwdWarps + w) * P + m];
                }
                atomicAdd(a.dB + (b * L + t) * N + m, sB);
                atomicAdd(a.dC + (b * L + t) * N + m, sC);
            }
        }
    }
    if (act) {
        atomicAdd(a.dA + d * N + n, dAacc);
        if (a.dh0)
            a.dh0[(b * D + d) * N + n] = g;
    }
}

// ---- host side: the launch shape and the launch --------------------------

// The checkpoint workspace of a call is Bsz * nch * D * P floats.
struct BwdShape {
    int P;           // lanes per chain
    int cpb;         // chains per block
    int64_t nch;     // chunks of kBwdT steps
    int64_t gx;      // blocks along D
    size_t smem;     // dynamic shared memory per block, bytes
};

inline BwdShape bwd_shape(int64_t L, int64_t D, int64_t N)
{
    BwdShape s;
    s.P = 1;
    while (s.P < N) s.P <<= 1;
    s.cpb = kBwdThreads / s.P;
    s.nch = (L + kBwdT - 1) / kBwdT;
    s.gx = (D + s.cpb - 1) / s.cpb;
    s.smem = (size_t)bwd_smem_floats(s.P, s.cpb) * 4;
    return s;
}

// a.P, a.cpb and a.nch are filled in from s; grid (s.gx, Bsz).
inline cudaError_t launch_scan_bwd(BwdArgs a, const BwdShape &s, cudaStream_t st)
{
    a.P = s.P;
    a.cpb = s.cpb;
    a.nch = s.nch;
    void (*kern)(BwdArgs);
    switch (s.P) {
    case 1: kern = scan_bwd_kernel<1>; break;
    case 2: kern = scan_bwd_kernel<2>; break;
    case 4: kern = scan_bwd_kernel<4>; break;
    case 8: kern = scan_bwd_kernel<8>; break;
    case 16: kern = scan_bwd_kernel<16>; break;
    default: kern = scan_bwd_kernel<32>; break;
    }
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s.smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)s.gx, (unsigned)a.Bsz), kBwdThreads, s.smem, st>>>(a);
    return cudaGetLastError();
}

} // namespace selscan
