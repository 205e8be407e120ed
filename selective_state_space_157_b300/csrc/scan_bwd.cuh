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
// Per-timestep inputs of a chunk are staged in shared memory by the whole
// block with coalesced loads (one row of cpb channels per step). dx and
// d delta are written by lane 0 of each chain; dB and dC are summed over the
// chains of a warp with shuffles, over the warps in shared memory, and added
// to global memory with one atomic per block, timestep and state; dA is
// summed over t in registers and added with one atomic per chain.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "device_math.cuh"

namespace selscan {

constexpr int kBwdThreads = 256;
constexpr int kBwdWarps = kBwdThreads / 32;
constexpr int kBwdT = 16;      // timesteps per chunk (registers per lane: 2 * kBwdT)

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

// Stages the per-timestep inputs of chunk t0 .. t0 + kBwdT of batch row b:
// x, dl (after softplus), its derivative and gy for the block's channels
// d0 .. d0 + cpb, and B, C for states 0 .. P (zero beyond L, D and N).
__device__ __forceinline__ void bwd_stage(const BwdArgs &a, int64_t b, int64_t d0, int64_t t0, bool adjoint,
                                          float *s_x, float *s_dl, float *s_sg, float *s_gy, float *s_B,
                                          float *s_C)
{
    const int cpb = a.cpb, P = a.P;
    for (int j = threadIdx.x; j < kBwdT * cpb; j += kBwdThreads) {
        const int i = j / cpb, c = j - i * cpb;
        const int64_t t = t0 + i, d = d0 + c;
        const bool ok = t < a.L && d < a.D;
        const int64_t idx = (b * a.L + t) * a.D + d;
        const float u = ok ? __ldg(a.delta + idx) : 0.0f;
        s_x[j] = ok ? __ldg(a.x + idx) : 0.0f;
        s_dl[j] = a.softplus ? softplus(u) : u;
        if (adjoint) {
            s_sg[j] = a.softplus ? bwd_sigmoid(u) : 1.0f;
            s_gy[j] = ok ? __ldg(a.gy + idx) : 0.0f;
        }
    }
    for (int j = threadIdx.x; j < kBwdT * P; j += kBwdThreads) {
        const int i = j / P, n = j - i * P;
        const int64_t t = t0 + i;
        const bool ok = t < a.L && n < a.N;
        const int64_t idx = (b * a.L + t) * a.N + n;
        s_B[j] = ok ? __ldg(a.B + idx) : 0.0f;
        if (adjoint)
            s_C[j] = ok ? __ldg(a.C + idx) : 0.0f;
    }
}

// grid (ceil(D / cpb), Bsz), kBwdThreads threads,
// bwd_smem_floats(P, cpb) * 4 bytes of dynamic shared memory.
// dA, dB and dC must be zero on entry (they are accumulated atomically).
__global__ void __launch_bounds__(kBwdThreads) scan_bwd_kernel(BwdArgs a)
{
    extern __shared__ float bwd_smem[];
    const int P = a.P, cpb = a.cpb;
    float *s_x = bwd_smem;
    float *s_dl = s_x + kBwdT * cpb;
    float *s_sg = s_dl + kBwdT * cpb;
    float *s_gy = s_sg + kBwdT * cpb;
    float *s_B = s_gy + kBwdT * cpb;
    float *s_C = s_B + kBwdT * P;
    float *s_pB = s_C + kBwdT * P;              // [kBwdT][kBwdWarps][P]
    float *s_pC = s_pB + kBwdT * kBwdWarps * P;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = tid & (P - 1), c = tid / P;
    const int64_t b = blockIdx.y;
    const int64_t d0 = int64_t(blockIdx.x) * cpb, d = d0 + c;
    const bool chain = d < a.D;                 // this lane's chain exists
    const bool act = chain && n < a.N;          // ... and its state index too
    const int64_t L = a.L, D = a.D, N = a.N, nch = a.nch;

    const float An = act ? __ldg(a.A + d * N + n) : 0.0f;
    const float A2 = An * kLog2e;

    // 1. forward pass: the state at the start of every chunk
    float h = (act && a.h0) ? __ldg(a.h0 + (b * D + d) * N + n) : 0.0f;
    for (int64_t k = 0; k < nch; ++k) {
        const int64_t t0 = k * kBwdT;
        if (chain)
            a.ckpt[((b * nch + k) * D + d) * P + n] = h;
        bwd_stage(a, b, d0, t0, false, s_x, s_dl, s_sg, s_gy, s_B, s_C);
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kBwdT; ++i) {
            if (t0 + i < L) {
                const float dl = s_dl[i * cpb + c];
                h = fmaf(ex2(dl * A2), h, dl * s_B[i * P + n] * s_x[i * cpb + c]);
            }
        }
        __syncthreads();
    }

    // 2. the chunks last to first: recompute, then run the adjoint back
    float g = (act && a.ghT) ? __ldg(a.ghT + (b * D + d) * N + n) : 0.0f;
    float dAacc = 0.0f;
    for (int64_t k = nch - 1; k >= 0; --k) {
        const int64_t t0 = k * kBwdT;
        bwd_stage(a, b, d0, t0, true, s_x, s_dl, s_sg, s_gy, s_B, s_C);
        const float hs = chain ? a.ckpt[((b * nch + k) * D + d) * P + n] : 0.0f;
        __syncthreads();

        float hc[kBwdT], ac[kBwdT];
        float hh = hs;
#pragma unroll
        for (int i = 0; i < kBwdT; ++i) {
            hc[i] = 0.0f;
            ac[i] = 1.0f;
            if (t0 + i < L) {
                const float dl = s_dl[i * cpb + c];
                const float av = ex2(dl * A2);
                hh = fmaf(av, hh, dl * s_B[i * P + n] * s_x[i * cpb + c]);
                hc[i] = hh;
                ac[i] = av;
            }
        }

        float dAk = 0.0f;
#pragma unroll
        for (int i = kBwdT - 1; i >= 0; --i) {
            if (t0 + i < L) {                  // uniform over the block
                const float dl = s_dl[i * cpb + c], xv = s_x[i * cpb + c], gyv = s_gy[i * cpb + c];
                const float Bn = s_B[i * P + n], Cn = s_C[i * P + n];
                g = fmaf(gyv, Cn, g);                      // y_t reads h_t
                float pC = gyv * hc[i];
                const float hp = i > 0 ? hc[i - 1] : hs;   // h_{t-1}
                const float dan = g * hp * ac[i];
                float gdl = fmaf(dan, An, g * Bn * xv);
                dAk = fmaf(dan, dl, dAk);
                float pB = g * dl * xv;
                float gx = g * dl * Bn;
                g *= ac[i];                                // into h_{t-1}
                for (int off = P >> 1; off > 0; off >>= 1) {
                    gx += __shfl_xor_sync(0xffffffffu, gx, off);
                    gdl += __shfl_xor_sync(0xffffffffu, gdl, off);
                }
                if (n == 0 && chain) {
                    const int64_t idx = (b * L + t0 + i) * D + d;
                    a.dx[idx] = gx;
                    a.ddelta[idx] = gdl * s_sg[i * cpb + c];
                }
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
        dAacc += dAk;
        __syncthreads();
        for (int j = tid; j < kBwdT * N; j += kBwdThreads) {
            const int i = j / int(N), m = j - i * int(N);
            const int64_t t = t0 + i;
            if (t < L) {
                float sB = 0.0f, sC = 0.0f;
                for (int w = 0; w < kBwdWarps; ++w) {
                    sB += s_pB[(i * kBwdWarps + w) * P + m];
                    sC += s_pC[(i * kBwdWarps + w) * P + m];
                }
                atomicAdd(a.dB + (b * L + t) * N + m, sB);
                atomicAdd(a.dC + (b * L + t) * N + m, sC);
            }
        }
        __syncthreads();
    }
    if (act) {
        atomicAdd(a.dA + d * N + n, dAacc);
        if (a.dh0)
            a.dh0[(b * D + d) * N + n] = g;
    }
}

// ---- host side: the launch shape and the launch --------------------------

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

// Checkpoint workspace of a call, in floats: Bsz * nch * D * P (the caller
// checks the product for overflow).
inline int64_t bwd_ckpt_floats(const BwdShape &s, int64_t Bsz, int64_t D)
{
    return Bsz * s.nch * D * s.P;
}

// a.P, a.cpb and a.nch are filled in from s; grid (s.gx, Bsz).
inline cudaError_t launch_scan_bwd(BwdArgs a, const BwdShape &s, cudaStream_t st)
{
    a.P = s.P;
    a.cpb = s.cpb;
    a.nch = s.nch;
    cudaError_t e = cudaFuncSetAttribute(scan_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s.smem);
    if (e != cudaSuccess) return e;
    scan_bwd_kernel<<<dim3((unsigned)s.gx, (unsigned)a.Bsz), kBwdThreads, s.smem, st>>>(a);
    return cudaGetLastError();
}

} // namespace selscan
