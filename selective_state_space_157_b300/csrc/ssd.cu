// ssd.cu -- Mamba-2's state space duality (SSD) forward on the tensor cores
// (youngju.dev "Mamba: Selective State Space Models", section 4.1: the
// recurrence h_t = A_t h_{t-1} + B_t x_t, y_t = C_t h_t, and its dual form
// Y = (T o M) X with M semiseparable; section 5.2: heads of headdim P with a
// state of size N).
//
// Per batch row b and head h, with a scalar decay per step a_t =
// exp(dl_t A[h]) (dl = dt, or softplus(dt)), the input term dl_t B_t x_t, and
// B, C shared by all heads, the state is N x P:
//   H_t[n][p] = a_t H_{t-1}[n][p] + dl_t B_t[n] x_t[p],   y_t[p] = sum_n C_t[n] H_t[n][p].
// The sequence is cut into chunks of Q = 64 steps. With s_t the cumulative
// sum of dl A inside a chunk (inclusive), the chunk's outputs are the dual
// form inside the chunk plus the decayed incoming state,
//   Y = ((C B^T) o L o exp(s_t - s_r) o dl_r) X + diag(exp(s_t)) C H_in,
// and the chunk's own contribution to the state is
//   S = (B o w)^T X,   w_r = exp(s_last - s_r) dl_r,
// with H_out = exp(s_last) H_in + S. Three kernels:
//   1. ssd_state_kernel: S of every chunk (tcgen05: M = N, N = P, K = Q);
//   2. ssd_carry_kernel: H_in of every chunk in order, elementwise, and hT;
//   3. ssd_out_kernel: G = C B^T (M = Q, N = Q, K = N), the masked, decayed
//      G times X (M = Q, N = P, K = Q) and C e^s times H_in (K = N), both
//      accumulated into one TMEM tile, then y.
// Operands are fp16 in shared memory (bf16 and fp32 inputs are converted
// on the way in; fp16 keeps three more mantissa bits than bf16, and every
// operand here stays far inside its range), accumulators fp32 in TMEM.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "device_math.cuh"
#include "host_common.h"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace selscan {
namespace {

constexpr int kSsdQ = 64;          // steps per chunk
constexpr int kSsdThreads = 128;   // four warps: one per TMEM lane quarter
constexpr unsigned kFaultMmaTimeout = 3;   // an MMA's completion never arrived

struct SsdArgs {
    const void *x;       // (Bsz, L, H, P), dtype
    const float *dt;     // (Bsz, L, H)
    const float *A;      // (H)
    const void *B, *C;   // (Bsz, L, N), dtype
    void *y;             // (Bsz, L, H, P), dtype
    const float *h0;     // (Bsz, H, N, P) or null
    float *hT;           // (Bsz, H, N, P) or null
    float *S;            // (Bsz, H, nch, N, P): chunk states from zero, then the state entering each chunk
    float *dec;          // (Bsz, H, nch): exp(s_last) of each chunk
    unsigned *fault;
    int64_t Bsz, L, H;
    int nch;
    int softplus;
};

__device__ __forceinline__ float ld_in(const float *p) { return __ldg(p); }
__device__ __forceinline__ float ld_in(const __nv_bfloat16 *p) { return __bfloat162float(__ldg(p)); }
__device__ __forceinline__ void st_out(float *p, float v) { *p = v; }
__device__ __forceinline__ void st_out(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

// Eight consecutive inputs as fp32 (one 16-byte load for bf16, two for fp32).
__device__ __forceinline__ void ld8(const float *p, float (&v)[8])
{
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p)), b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void ld8(const __nv_bfloat16 *p, float (&v)[8])
{
    const uint4 w = __ldg(reinterpret_cast<const uint4 *>(p));
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(u[i] << 16);
        v[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
    }
}

// Eight fp32 values as eight fp16 in one 16-byte word.
__device__ __forceinline__ uint4 pack8(const float (&v)[8])
{
    uint4 r;
    uint32_t *u = reinterpret_cast<uint32_t *>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2 h = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
        u[i] = *reinterpret_cast<const uint32_t *>(&h);
    }
    return r;
}

// Rows [0, Q) of a row-major global tile (row stride ld elements, K columns,
// rows >= rows zero) as a K-major fp16 operand in core-matrix order, scaled
// row by row by scale[] when given. Each thread moves eight columns at a time.
template <typename T, int Q, int K>
__device__ __forceinline__ void stage_rows(const T *g, int64_t ld, int rows, const float *scale, __half *dst)
{
#pragma unroll 4
    for (int e = threadIdx.x; e < Q * (K / 8); e += kSsdThreads) {
        const int r = e / (K / 8), k = (e % (K / 8)) * 8;
        float v[8];
        if (r < rows) {
            ld8(g + r * ld + k, v);
            if (scale) {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    v[i] *= scale[r];
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                v[i] = 0.0f;
        }
        *reinterpret_cast<uint4 *>(dst + core_index(r, k, K)) = pack8(v);
    }
}

// The transpose of rows [0, Q) of a row-major global tile with R columns
// (row stride ld; rows >= rows zero), optionally scaled per source row by
// scale[]: a K-major operand with R rows and K = Q, in core-matrix order.
// The tile goes through a padded fp16 staging buffer (row stride R + 8, so
// the column reads below hit distinct banks), then each thread gathers eight
// source rows of one column into one 16-byte core row.
template <typename T, int Q, int R>
__device__ __forceinline__ void stage_transposed(const T *g, int64_t ld, int rows, const float *scale, __half *stg,
                                                 __half *dst)
{
    constexpr int S = R + 8;
#pragma unroll 4
    for (int e = threadIdx.x; e < Q * (R / 8); e += kSsdThreads) {
        const int k = e / (R / 8), r = (e % (R / 8)) * 8;
        float v[8];
        if (k < rows) {
            ld8(g + k * ld + r, v);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                v[i] = 0.0f;
        }
        *reinterpret_cast<uint4 *>(stg + k * S + r) = pack8(v);
    }
    __syncthreads();
#pragma unroll 4
    for (int e = threadIdx.x; e < R * (Q / 8); e += kSsdThreads) {
        const int r = e % R, k = (e / R) * 8;
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            v[i] = __half2float(stg[(k + i) * S + r]) * (scale ? scale[k + i] : 1.0f);
        *reinterpret_cast<uint4 *>(dst + core_index(r, k, Q)) = pack8(v);
    }
}

// Step sizes and cumulative log-decays of one chunk: dl[t] (after softplus)
// and s[t] = sum_{r <= t} dl[r] A[h], t < Q. Rows past the sequence get
// dl = 0, so they neither decay nor add. Warp 0 only.
__device__ __forceinline__ void ssd_decays(const SsdArgs &a, int64_t b, int64_t h, int64_t t0, int rows, float *dl,
                                           float *s)
{
    const int lane = threadIdx.x;
    const float Ah = __ldg(a.A + h);
    float v[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int t = lane + 32 * i;
        float d = 0.0f;
        if (t < rows) {
            d = __ldg(a.dt + (b * a.L + t0 + t) * a.H + h);
            if (a.softplus)
                d = softplus(d);
        }
        dl[t] = d;
        v[i] = d * Ah;
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float u = __shfl_up_sync(0xffffffffu, v[i], o);
            if (lane >= o)
                v[i] += u;
        }
    }
    const float first_half = __shfl_sync(0xffffffffu, v[0], 31);
    s[lane] = v[0];
    s[lane + 32] = v[1] + first_half;
}

// Waits (bounded) for the phase with the given parity of an MMA completion
// barrier; every thread of the CTA learns the same answer.
__device__ __forceinline__ bool mma_wait(uint64_t *bar, uint32_t parity)
{
    return __syncthreads_and(mbar_wait(bar, parity));
}

// 1. Each chunk's contribution to the state, S = (B o w)^T X (N x P),
// stored transposed, [p][n], for the carry scan and the output kernel.
template <typename T, int N, int P>
__global__ void __launch_bounds__(kSsdThreads) ssd_state_kernel(const SsdArgs a)
{
    constexpr int Q = kSsdQ;
    extern __shared__ __align__(1024) unsigned char sm[];
    __half *A3 = reinterpret_cast<__half *>(sm);                  // (B o w)^T: N rows, K = Q
    __half *BX = A3 + N * Q;                                       // X^T: P rows, K = Q
    __half *stg = BX + P * Q;                                      // staging, Q x (max(N, P) + 8)
    float *dl = reinterpret_cast<float *>(stg + Q * ((N > P ? N : P) + 8));
    float *s = dl + Q;
    float *w = s + Q;
    __shared__ uint32_t tbase;
    __shared__ __align__(8) uint64_t mbar;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t b = blockIdx.z, h = blockIdx.y, c = blockIdx.x;
    const int64_t t0 = c * Q;
    const int rows = (int)min((int64_t)Q, a.L - t0);
    const T *xg = static_cast<const T *>(a.x) + ((b * a.L + t0) * a.H + h) * P;
    const T *Bg = static_cast<const T *>(a.B) + (b * a.L + t0) * N;

    if (tid == 0) {
        mbar_init(&mbar, 1);
        fence_mbar_init();
    }
    if (warp == 0)
        ssd_decays(a, b, h, t0, rows, dl, s);
    __syncthreads();
    const float slast = s[Q - 1];
    if (tid < Q)
        w[tid] = ex2((slast - s[tid]) * kLog2e) * dl[tid];
    __syncthreads();
    stage_transposed<T, Q, N>(Bg, N, rows, w, stg, A3);
    __syncthreads();
    stage_transposed<T, Q, P>(xg, a.H * P, rows, nullptr, stg, BX);
    fence_proxy_async_smem();   // the tensor core reads shared memory through the async proxy
    if (warp == 0)
        tmem_alloc(&tbase, P);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = tbase;
    if (tid == 0) {
        constexpr uint32_t id = umma_idesc_f16(N, P);
#pragma unroll
        for (int kk = 0; kk < Q / 16; ++kk)
            umma_f16(tm, umma_tile_desc(A3, Q, kk), umma_tile_desc(BX, Q, kk), id, kk > 0);
        umma_commit(&mbar);
    }
    const bool ok = mma_wait(&mbar, 0);
    tc_fence_after();
    // Row n of S sits in TMEM lane n (N = 128) or lane 32w + (n - 16w) (N = 64);
    // a warp's lanes hold consecutive n, so the [p][n] stores coalesce.
    const int n = N == 128 ? 32 * warp + lane : 16 * warp + lane;
    const bool mine = ok && (N == 128 || lane < 16);
    float *dst = a.S + ((b * a.H + h) * a.nch + c) * N * P + n;
#pragma unroll
    for (int p0 = 0; p0 < P; p0 += 16) {
        float v[16];
        tmem_ld16(tm + ((uint32_t)(32 * warp) << 16) + (uint32_t)p0, v);
        if (mine) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
                dst[(p0 + i) * N] = v[i];
        }
    }
    if (tid == 0) {
        a.dec[(b * a.H + h) * a.nch + c] = ex2(slast * kLog2e);
        if (!ok)
            record_fault(a.fault, kFaultMmaTimeout);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        tmem_dealloc(tm, P);
}

// 2. The state entering each chunk, in chunk order (in place of S, still
// [p][n]), and hT ([n][p]). A thread's chunk states are all loaded before
// the serial fold, up to kCarryBatch at a time.
constexpr int kCarryBatch = 16;

__global__ void __launch_bounds__(256) ssd_carry_kernel(const SsdArgs a, int N, int P)
{
    const int64_t NP = (int64_t)N * P;
    const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (i >= a.Bsz * a.H * NP)
        return;
    const int64_t bh = i / NP, pn = i - bh * NP;
    const int64_t p = pn / N, n = pn - p * N;
    float carry = a.h0 ? __ldg(a.h0 + bh * NP + n * P + p) : 0.0f;
    float *Sp = a.S + bh * a.nch * NP + pn;
    const float *dp = a.dec + bh * a.nch;
    for (int c0 = 0; c0 < a.nch; c0 += kCarryBatch) {
        float sv[kCarryBatch], dv[kCarryBatch];
#pragma unroll
        for (int j = 0; j < kCarryBatch; ++j) {
            const int cc = c0 + j < a.nch ? c0 + j : a.nch - 1;
            sv[j] = __ldcg(Sp + (int64_t)cc * NP);
            dv[j] = __ldg(dp + cc);
        }
#pragma unroll
        for (int j = 0; j < kCarryBatch; ++j) {
            if (c0 + j < a.nch) {
                Sp[(int64_t)(c0 + j) * NP] = carry;
                carry = fmaf(dv[j], carry, sv[j]);
            }
        }
    }
    if (a.hT)
        a.hT[bh * NP + n * P + p] = carry;
}

// 3. Each chunk's outputs: the masked dual form inside the chunk plus the
// decayed incoming state.
template <typename T, int N, int P>
__global__ void __launch_bounds__(kSsdThreads) ssd_out_kernel(const SsdArgs a)
{
    constexpr int Q = kSsdQ;
    constexpr int COLS = 64 + P <= 128 ? 128 : 256;   // G (64 columns) and Y (P)
    extern __shared__ __align__(1024) unsigned char sm[];
    __half *A1 = reinterpret_cast<__half *>(sm);                       // C: Q rows, K = N
    __half *A4 = A1 + Q * N;                                            // C e^s: Q rows, K = N
    __half *B1 = A4 + Q * N;                                            // B: Q rows, K = N
    __half *B4 = B1 + Q * N;                                            // H_in^T: P rows, K = N
    __half *BX = B4 + P * N;                                            // X^T: P rows, K = Q
    __half *A2 = BX + P * Q;                                            // masked G: Q rows, K = Q
    __half *stg = A2 + Q * Q;                                           // staging, Q x (P + 8)
    float *dl = reinterpret_cast<float *>(stg + Q * (P + 8));
    float *s = dl + Q;
    float *es = s + Q;
    __shared__ uint32_t tbase;
    __shared__ __align__(8) uint64_t mbar;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t b = blockIdx.z, h = blockIdx.y, c = blockIdx.x;
    const int64_t t0 = c * Q;
    const int rows = (int)min((int64_t)Q, a.L - t0);
    const bool carry = c > 0 || a.h0 != nullptr;
    const T *xg = static_cast<const T *>(a.x) + ((b * a.L + t0) * a.H + h) * P;
    const T *Bg = static_cast<const T *>(a.B) + (b * a.L + t0) * N;
    const T *Cg = static_cast<const T *>(a.C) + (b * a.L + t0) * N;

    if (tid == 0) {
        mbar_init(&mbar, 1);
        fence_mbar_init();
    }
    if (warp == 0)
        ssd_decays(a, b, h, t0, rows, dl, s);
    __syncthreads();
    if (tid < Q)
        es[tid] = ex2(s[tid] * kLog2e);
    __syncthreads();
    stage_rows<T, Q, N>(Cg, N, rows, nullptr, A1);
    stage_rows<T, Q, N>(Cg, N, rows, es, A4);
    stage_rows<T, Q, N>(Bg, N, rows, nullptr, B1);
    if (carry)   // the incoming state, [p][n] fp32: P rows of K = N
        stage_rows<float, P, N>(a.S + ((b * a.H + h) * a.nch + c) * N * P, N, P, nullptr, B4);
    stage_transposed<T, Q, P>(xg, a.H * P, rows, nullptr, stg, BX);
    fence_proxy_async_smem();
    if (warp == 0)
        tmem_alloc(&tbase, COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tG = tbase, tY = tbase + 64;
    if (tid == 0) {
        constexpr uint32_t id = umma_idesc_f16(Q, Q);
#pragma unroll
        for (int kk = 0; kk < N / 16; ++kk)
            umma_f16(tG, umma_tile_desc(A1, N, kk), umma_tile_desc(B1, N, kk), id, kk > 0);
        umma_commit(&mbar);
    }
    bool ok = mma_wait(&mbar, 0);
    tc_fence_after();
    // Row t of G sits in lane 32w + (t - 16w) of warp w (M = 64). Mask,
    // decay and scale it into the masked product's A operand, eight
    // columns (one core row) per 16-byte store.
    const int t = 16 * warp + lane;
    const uint32_t lanes = (uint32_t)(32 * warp) << 16;
#pragma unroll
    for (int s0 = 0; s0 < Q; s0 += 16) {
        float g[16];
        tmem_ld16(tG + lanes + (uint32_t)s0, g);
        if (lane < 16) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float m[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int r = s0 + 8 * half + i;
                    m[i] = r <= t ? g[8 * half + i] * ex2((s[t] - s[r]) * kLog2e) * dl[r] : 0.0f;
                }
                *reinterpret_cast<uint4 *>(A2 + core_index(t, s0 + 8 * half, Q)) = pack8(m);
            }
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
        constexpr uint32_t id = umma_idesc_f16(Q, P);
#pragma unroll
        for (int kk = 0; kk < Q / 16; ++kk)
            umma_f16(tY, umma_tile_desc(A2, Q, kk), umma_tile_desc(BX, Q, kk), id, kk > 0);
        if (carry) {
#pragma unroll
            for (int kk = 0; kk < N / 16; ++kk)
                umma_f16(tY, umma_tile_desc(A4, N, kk), umma_tile_desc(B4, N, kk), id, true);
        }
        umma_commit(&mbar);
    }
    ok = mma_wait(&mbar, 1) && ok;
    tc_fence_after();
    T *yg = static_cast<T *>(a.y) + ((b * a.L + t0 + t) * a.H + h) * P;
    const bool mine = ok && lane < 16 && t < rows;
#pragma unroll
    for (int p0 = 0; p0 < P; p0 += 16) {
        float v[16];
        tmem_ld16(tY + lanes + (uint32_t)p0, v);
        if (mine) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
                st_out(yg + p0 + i, v[i]);
        }
    }
    if (tid == 0 && !ok)
        record_fault(a.fault, kFaultMmaTimeout);
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        tmem_dealloc(tbase, COLS);
}

template <int N, int P>
constexpr size_t ssd_state_smem()
{
    return ((size_t)(N + P) * kSsdQ + (size_t)kSsdQ * ((N > P ? N : P) + 8)) * 2 + 3 * kSsdQ * 4;
}

template <int N, int P>
constexpr size_t ssd_out_smem()
{
    return ((size_t)3 * kSsdQ * N + (size_t)P * N + (size_t)P * kSsdQ + (size_t)kSsdQ * kSsdQ +
            (size_t)kSsdQ * (P + 8)) * 2 + 3 * kSsdQ * 4;
}

template <typename T, int N, int P>
int launch_ssd_t(const SsdArgs &a, cudaStream_t st)
{
    auto k1 = ssd_state_kernel<T, N, P>;
    auto k3 = ssd_out_kernel<T, N, P>;
    // At most 512 / P state-kernel CTAs per SM (P TMEM columns each), so that
    // their allocations never exceed the SM's 512 columns: shared memory is
    // padded to keep more from fitting.
    constexpr size_t kPad = (size_t)228 * 1024 / (512 / P) - 1024 + 1;
    const size_t s1 = ssd_state_smem<N, P>() > kPad ? ssd_state_smem<N, P>() : kPad;
    const size_t s3 = ssd_out_smem<N, P>();
    cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k3, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s3);
    if (e != cudaSuccess) return cuda_fail(e, "SSD kernel attributes");
    const dim3 grid((unsigned)a.nch, (unsigned)a.H, (unsigned)a.Bsz);
    k1<<<grid, kSsdThreads, s1, st>>>(a);
    const int64_t NP = (int64_t)N * P;
    const int64_t total = a.Bsz * a.H * NP;
    ssd_carry_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(a, N, P);
    k3<<<grid, kSsdThreads, s3, st>>>(a);
    e = cudaGetLastError();
    return e == cudaSuccess ? SELSCAN_OK : cuda_fail(e, "SSD kernel launch");
}

template <typename T>
int launch_ssd(const SsdArgs &a, int64_t N, int64_t P, cudaStream_t st)
{
    switch (N * 1000 + P) {
    case 64032: return launch_ssd_t<T, 64, 32>(a, st);
    case 64064: return launch_ssd_t<T, 64, 64>(a, st);
    case 64128: return launch_ssd_t<T, 64, 128>(a, st);
    case 128032: return launch_ssd_t<T, 128, 32>(a, st);
    case 128064: return launch_ssd_t<T, 128, 64>(a, st);
    case 128128: return launch_ssd_t<T, 128, 128>(a, st);
    default: return fail(SELSCAN_ERR_UNSUPPORTED, "SSD: N=%lld P=%lld (N must be 64 or 128, P 32, 64 or 128)",
                         (long long)N, (long long)P);
    }
}

} // namespace
} // namespace selscan

using namespace selscan;

extern "C" int selscan_ssd_fwd(const void *x, const float *dt, const float *A, const void *B, const void *C,
                               void *y, const float *h0, float *hT, int64_t Bsz, int64_t L, int64_t H, int64_t P,
                               int64_t N, int dtype, int dt_softplus, void *stream)
{
    g_err[0] = '\0';
    if (dtype != SELSCAN_F32 && dtype != SELSCAN_BF16)
        return fail(SELSCAN_ERR_INVALID_ARG, "dtype %d is neither SELSCAN_F32 nor SELSCAN_BF16", dtype);
    if (Bsz < 0 || L < 0 || H < 0 || P < 1 || N < 1)
        return fail(SELSCAN_ERR_INVALID_ARG, "bad sizes (Bsz=%lld L=%lld H=%lld P=%lld N=%lld)", (long long)Bsz,
                    (long long)L, (long long)H, (long long)P, (long long)N);
    if (!((N == 64 || N == 128) && (P == 32 || P == 64 || P == 128)))
        return fail(SELSCAN_ERR_UNSUPPORTED, "SSD: N=%lld P=%lld (N must be 64 or 128, P 32, 64 or 128)",
                    (long long)N, (long long)P);
    int64_t elx, eln, eld, els;
    if (!mul_ok(Bsz, L, H * P, &elx) || !mul_ok(Bsz, L, N, &eln) || !mul_ok(Bsz, L, H, &eld) ||
        !mul_ok(Bsz, H, N * P, &els))
        return fail(SELSCAN_ERR_INVALID_ARG, "sizes overflow");
    if (Bsz == 0 || H == 0)
        return SELSCAN_OK;
    if (Bsz > 65535 || H > 65535)
        return fail(SELSCAN_ERR_UNSUPPORTED, "SSD: Bsz and H must be at most 65535");
    if (!A || (L > 0 && (!x || !dt || !B || !C || !y)))
        return fail(SELSCAN_ERR_INVALID_ARG, "A, and x, dt, B, C, y when L > 0, must be non-NULL");
    const size_t es = dtype == SELSCAN_F32 ? 4 : 2;   // element size of x, B, C, y
    if (!aligned(x, 16) || !aligned(B, 16) || !aligned(C, 16) || !aligned(y, 16) || !aligned(dt, 4) ||
        !aligned(A, 4) || !aligned(h0, 16) || !aligned(hT, 16))
        return fail(SELSCAN_ERR_INVALID_ARG, "x, B, C, y, h0, hT must be 16-byte aligned, dt and A 4-byte aligned");
    const Range ry = range(L > 0 ? y : nullptr, elx * (int64_t)es, "y"), rh = range(hT, els * 4, "hT");
    const Range ins[] = {range(x, elx * (int64_t)es, "x"), range(dt, eld * 4, "dt"), range(A, H * 4, "A"),
                         range(B, eln * (int64_t)es, "B"), range(C, eln * (int64_t)es, "C"),
                         range(h0, els * 4, "h0")};
    for (const Range &r : ins) {
        if (overlaps(ry, r)) return fail(SELSCAN_ERR_INVALID_ARG, "y overlaps %s", r.name);
        if (overlaps(rh, r)) return fail(SELSCAN_ERR_INVALID_ARG, "hT overlaps %s", r.name);
    }
    if (overlaps(ry, rh))
        return fail(SELSCAN_ERR_INVALID_ARG, "y overlaps hT");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (L == 0) {
        if (!hT) return SELSCAN_OK;
        const cudaError_t e = h0 ? cudaMemcpyAsync(hT, h0, (size_t)els * 4, cudaMemcpyDeviceToDevice, st)
                                 : cudaMemsetAsync(hT, 0, (size_t)els * 4, st);
        return e == cudaSuccess ? SELSCAN_OK : cuda_fail(e, "L == 0 state copy");
    }
    const int64_t nch = (L + kSsdQ - 1) / kSsdQ;
    if (nch > 0x7fffffffLL) return fail(SELSCAN_ERR_UNSUPPORTED, "sequence too long");
    int dev = 0, sms = 0;
    int rc = device_info(&dev, &sms);
    if (rc != SELSCAN_OK) return rc;
    cudaMemPool_t pool = nullptr;
    rc = workspace_pool(dev, &pool);
    if (rc != SELSCAN_OK) return rc;
    const size_t sbytes = (size_t)(Bsz * H * nch) * (size_t)(N * P) * 4, dbytes = (size_t)(Bsz * H * nch) * 4;
    void *ws = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&ws, sbytes + dbytes, pool, st);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(SELSCAN_ERR_NO_MEMORY, "SSD workspace of %zu bytes: %s", sbytes + dbytes, cudaGetErrorString(e));
    }
    SsdArgs a;
    memset(&a, 0, sizeof a);
    a.x = x; a.dt = dt; a.A = A; a.B = B; a.C = C; a.y = y; a.h0 = h0; a.hT = hT;
    a.S = static_cast<float *>(ws);
    a.dec = a.S + sbytes / 4;
    a.Bsz = Bsz; a.L = L; a.H = H;
    a.nch = (int)nch;
    a.softplus = dt_softplus ? 1 : 0;
    rc = fault_word(dev, st, &a.fault);
    if (rc == SELSCAN_OK)
        rc = dtype == SELSCAN_F32 ? launch_ssd<float>(a, N, P, st) : launch_ssd<__nv_bfloat16>(a, N, P, st);
    cudaFreeAsync(ws, st);
    return rc;
}
