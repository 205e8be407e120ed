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
//   1. ssd_state_kernel: S of every chunk (tcgen05: M = N, N = P, K = Q),
//      stored fp16 (the precision it has as an operand anyway). The same
//      launch has one more CTA per batch row and chunk that forms
//      G = C B^T (M = Q, N = Q, K = N), which no head changes, and stores it,
//      and C, as fp16 in the output kernel's operand order;
//   2. ssd_carry_kernel: H_in of every chunk in order, elementwise in fp32,
//      written as fp16 in the output kernel's operand layout, and hT;
//   3. ssd_out_kernel: G masked and decayed in place in shared memory, times
//      X (M = Q, N = P, K = Q) into one TMEM tile, C H_in (K = N) into a
//      second; y = G X + diag(e^s) C H_in.
// Kernels 2 and 3 are launched as programmatic dependents of the one before.
// Each CTA brings every tile it needs into shared memory in one round trip
// (cp.async, zeros past the sequence), then converts and transposes there.
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
    __half *S;           // (Bsz, H, nch, P, N): each chunk's state from zero, [p][n], fp16
    __half *Hin;         // (Bsz, H, nch, P x N): the state entering each chunk, fp16 operand order
    __half *G;           // (Bsz, nch, Q x Q): C B^T of each chunk, fp16, in operand order (K = Q)
    __half *Cop;         // (Bsz, nch, Q x N): C of each chunk as the output kernel's fp16 A operand
    float *dec;          // (Bsz, H, nch): exp(s_last) of each chunk
    unsigned *fault;
    int64_t Bsz, L, H;
    int nch;
    int softplus;
};

// Programmatic dependent launch: a kernel launched with it may start while
// the kernel before it on the stream is still running; it calls
// grid_dep_wait() before it reads anything that kernel wrote (the wait
// returns once that whole grid has completed and its writes are visible).
// grid_dep_trigger() lets the next such kernel start early.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// 16-byte asynchronous copy global -> shared; zeros instead when !ok.
__device__ __forceinline__ void ssd_cp16(void *dst, const void *src, bool ok)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(ok ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void ssd_cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void ssd_cp_wait() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Copies rows [0, Q) of a global tile (rows >= rows zero) of W elements per
// row, row stride ld elements, into dst[Q][W] (row-major, contiguous).
template <typename T, int Q, int W>
__device__ __forceinline__ void copy_tile(const T *g, int64_t ld, int rows, T *dst)
{
    constexpr int PR = W * (int)sizeof(T) / 16;   // 16-byte pieces per row
    for (int e = threadIdx.x; e < Q * PR; e += kSsdThreads) {
        const int r = e / PR, pc = e % PR;
        const bool ok = r < rows;
        ssd_cp16(reinterpret_cast<char *>(dst) + (size_t)e * 16,
                 ok ? reinterpret_cast<const char *>(g + (int64_t)r * ld) + pc * 16 : reinterpret_cast<const char *>(g),
                 ok);
    }
}

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

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

// A row-major [R][K] tile in shared memory as a K-major fp16 operand with R
// rows, in core-matrix order. Each thread moves eight columns at a time.
template <typename T, int R, int K>
__device__ __forceinline__ void rows_to_operand(const T *src, __half *dst)
{
#pragma unroll 4
    for (int e = threadIdx.x; e < R * (K / 8); e += kSsdThreads) {
        const int r = e / (K / 8), k = (e % (K / 8)) * 8;
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            v[i] = to_f32(src[r * K + k + i]);
        *reinterpret_cast<uint4 *>(dst + core_index(r, k, K)) = pack8(v);
    }
}

// Rows [0, Q) of a row-major global tile (row stride ld elements, K columns,
// rows >= rows zero) as a K-major fp16 operand in core-matrix order. Every
// load of the tile is issued before the first store, so a thread waits on
// memory once.
template <typename T, int Q, int K>
__device__ __forceinline__ void global_rows_to_operand(const T *g, int64_t ld, int rows, __half *dst)
{
    constexpr int PER = Q * (K / 8) / kSsdThreads;   // eight-column pieces per thread
    static_assert(PER * kSsdThreads == Q * (K / 8), "the tile must split evenly over the threads");
    constexpr int W = (int)sizeof(T) * 8 / 16;       // 16-byte words per piece
    uint4 raw[PER][W];
#pragma unroll
    for (int q = 0; q < PER; ++q) {
        const int e = threadIdx.x + q * kSsdThreads, r = e / (K / 8), k = (e % (K / 8)) * 8;
#pragma unroll
        for (int w = 0; w < W; ++w)
            raw[q][w] = r < rows ? __ldg(reinterpret_cast<const uint4 *>(g + (int64_t)r * ld + k) + w)
                                 : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int q = 0; q < PER; ++q) {
        const int e = threadIdx.x + q * kSsdThreads, r = e / (K / 8), k = (e % (K / 8)) * 8;
        float v[8];
        if constexpr (sizeof(T) == 2) {
            const uint32_t u[4] = {raw[q][0].x, raw[q][0].y, raw[q][0].z, raw[q][0].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[2 * i] = __uint_as_float(u[i] << 16);
                v[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
            }
        } else {
#pragma unroll
            for (int w = 0; w < W; ++w) {
                v[4 * w] = __uint_as_float(raw[q][w].x);
                v[4 * w + 1] = __uint_as_float(raw[q][w].y);
                v[4 * w + 2] = __uint_as_float(raw[q][w].z);
                v[4 * w + 3] = __uint_as_float(raw[q][w].w);
            }
        }
        *reinterpret_cast<uint4 *>(dst + core_index(r, k, K)) = pack8(v);
    }
}

// The transpose of a row-major [Q][R] tile in shared memory, scaled per
// source row by scale[] when given: a K-major operand with R rows and K = Q,
// in core-matrix order. Each thread gathers eight source rows of one column
// (consecutive lanes take consecutive columns: no bank conflicts) into one
// 16-byte core row.
template <typename T, int Q, int R>
__device__ __forceinline__ void transpose_to_operand(const T *src, const float *scale, __half *dst)
{
#pragma unroll 4
    for (int e = threadIdx.x; e < R * (Q / 8); e += kSsdThreads) {
        const int r = e % R, k = (e / R) * 8;
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            v[i] = to_f32(src[(k + i) * R + r]) * (scale ? scale[k + i] : 1.0f);
        *reinterpret_cast<uint4 *>(dst + core_index(r, k, Q)) = pack8(v);
    }
}

// The raw step pre-activations of one chunk, dt[t] for t = lane and
// lane + 32 (0 past the sequence); warp 0 loads them ahead of other work.
struct SsdDt {
    float v[2];
    float Ah;
};

__device__ __forceinline__ SsdDt ssd_dt_load(const SsdArgs &a, int64_t b, int64_t h, int64_t t0, int rows)
{
    const int lane = threadIdx.x & 31;
    SsdDt r;
    r.Ah = __ldg(a.A + h);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int t = lane + 32 * i;
        r.v[i] = t < rows ? __ldg(a.dt + (b * a.L + t0 + t) * a.H + h) : 0.0f;
    }
    return r;
}

// A step's log-decay dl A is taken as at least -kSsdMinLogDecay. The chunk's
// products use differences s_t - s_r of the cumulative sums; after a step of
// dl A = -1280 (dl = 80, A = -16) the sums reach magnitudes where fp32 keeps
// those differences only to about 1e-2. A decay of e^-40 already leaves less
// than fp32 resolution of anything carried across that step (as the true,
// smaller decay does), and with the bound |s| stays below 64 * 40 within a
// chunk, where differences keep about 2e-4.
constexpr float kSsdMinLogDecay = 40.0f;

// Step sizes and cumulative log-decays of one chunk: dl[t] (after softplus)
// and s[t] = sum_{r <= t} max(dl[r] A[h], -kSsdMinLogDecay), t < Q. Rows past
// the sequence get dl = 0, so they neither decay nor add. One warp.
__device__ __forceinline__ void ssd_decays_from(const SsdArgs &a, const SsdDt &raw, int rows, float *dl, float *s)
{
    const int lane = threadIdx.x & 31;
    float v[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int t = lane + 32 * i;
        float d = raw.v[i];
        if (t < rows && a.softplus)
            d = softplus(d);
        dl[t] = d;
        v[i] = fmaxf(d * raw.Ah, -kSsdMinLogDecay);
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

// The same, loaded and computed in one go. One warp.
__device__ __forceinline__ void ssd_decays(const SsdArgs &a, int64_t b, int64_t h, int64_t t0, int rows, float *dl,
                                           float *s)
{
    ssd_decays_from(a, ssd_dt_load(a, b, h, t0, rows), rows, dl, s);
}

// Waits (bounded) for the phase with the given parity of an MMA completion
// barrier; every thread of the CTA learns the same answer.
__device__ __forceinline__ bool mma_wait(uint64_t *bar, uint32_t parity)
{
    return __syncthreads_and(mbar_wait(bar, parity));
}

// Heads per CTA of the state kernel: they share the chunk's B^T operand.
template <typename T, int P>
__host__ __device__ constexpr int ssd_state_heads()
{
    return sizeof(T) == 2 ? (P <= 64 ? 4 : 2) : (P <= 64 ? 2 : 1);
}

// TMEM columns of the state kernel: P for each of its heads, or the 64 of
// C B^T.
template <typename T, int P>
__host__ __device__ constexpr int ssd_state_cols()
{
    return ssd_state_heads<T, P>() * P < 64 ? 64 : ssd_state_heads<T, P>() * P;
}

// 1. Each chunk's contribution to the state, S = (B o w)^T X = B^T (w o X)
// (N x P), stored transposed, [p][n], fp16, for the carry scan. A CTA takes
// HPC heads of one chunk: the chunk's B^T is converted once and serves as the
// A operand of every head's product; each head's X rows are scaled by its
// own w. CTAs with blockIdx.y == the number of head groups instead form
// C B^T of their chunk for the output kernel, and C, both as fp16 operands.
template <typename T, int N, int P>
__global__ void __launch_bounds__(kSsdThreads) ssd_state_kernel(const SsdArgs a)
{
    constexpr int Q = kSsdQ;
    constexpr int HPC = ssd_state_heads<T, P>();
    constexpr int COLS = ssd_state_cols<T, P>();
    extern __shared__ __align__(1024) unsigned char sm[];
    __half *A3 = reinterpret_cast<__half *>(sm);                  // B^T: N rows, K = Q
    __half *BX = A3 + N * Q;                                       // HPC x (w o X)^T: P rows, K = Q
    T *rB = reinterpret_cast<T *>(BX + HPC * P * Q);               // B tile [Q][N]
    T *rX = rB + Q * N;                                            // HPC x X tile [Q][P]
    float *dl = reinterpret_cast<float *>(rX + HPC * Q * P);       // HPC x [Q]
    float *s = dl + HPC * Q;
    float *w = s + HPC * Q;
    __shared__ uint32_t tbase;
    __shared__ __align__(8) uint64_t mbar;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t b = blockIdx.z, c = blockIdx.x;
    const int64_t ngroups = (a.H + HPC - 1) / HPC;
    const int64_t h0 = (int64_t)blockIdx.y * HPC;    // the group's first head
    const int nh = (int)min((int64_t)HPC, a.H - h0);
    const int64_t t0 = c * Q;
    const int rows = (int)min((int64_t)Q, a.L - t0);
    // TMEM first: the allocation permit is given up at once, so the SM can
    // start the next CTA while this one loads.
    if (warp == 0)
        tmem_alloc(&tbase, COLS);
    // Launched as a programmatic dependent of the kernel before it (the
    // previous call's output kernel, typically, whose workspace this call's
    // may reuse): nothing is read or written before it has completed.
    grid_dep_wait();

    if ((int64_t)blockIdx.y == ngroups) {
        // C B^T of the chunk: C and B rows as K-major operands (over the
        // space the state's operands use in the other CTAs).
        __half *A1 = A3, *B1 = reinterpret_cast<__half *>(rB);
        global_rows_to_operand<T, Q, N>(static_cast<const T *>(a.C) + (b * a.L + t0) * N, N, rows, A1);
        global_rows_to_operand<T, Q, N>(static_cast<const T *>(a.B) + (b * a.L + t0) * N, N, rows, B1);
        if (tid == 0) {
            mbar_init(&mbar, 1);
            fence_mbar_init();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        const uint32_t tm = tbase;
        if (tid == 0) {
            constexpr uint32_t id = umma_idesc_f16(Q, Q);
#pragma unroll
            for (int kk = 0; kk < N / 16; ++kk)
                umma_f16(tm, umma_tile_desc(A1, N, kk), umma_tile_desc(B1, N, kk), id, kk > 0);
            umma_commit(&mbar);
        }
        const bool ok = mma_wait(&mbar, 0);
        tc_fence_after();
        grid_dep_trigger();
        // Row t of C B^T sits in lane 32w + (t - 16w) of warp w (M = 64).
        uint32_t graw[Q / 16][16];
#pragma unroll
        for (int q = 0; q < Q / 16; ++q)
            tmem_ld16_async(tm + ((uint32_t)(32 * warp) << 16) + (uint32_t)(16 * q), graw[q]);
        tmem_wait_ld();
        if (ok && lane < 16) {
            // Row t as fp16 core rows of the output kernel's A operand (K = Q).
            const int t = 16 * warp + lane;
            __half *dst = a.G + (b * a.nch + c) * Q * Q;
#pragma unroll
            for (int r0 = 0; r0 < Q; r0 += 8) {
                float v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    v[i] = __uint_as_float(graw[(r0 + i) / 16][(r0 + i) % 16]);
                *reinterpret_cast<uint4 *>(dst + core_index(t, r0, Q)) = pack8(v);
            }
        }
        // C as the output kernel's A operand, already in core-matrix order.
        {
            const uint4 *src = reinterpret_cast<const uint4 *>(A1);
            uint4 *dst = reinterpret_cast<uint4 *>(a.Cop + (b * a.nch + c) * Q * N);
#pragma unroll 4
            for (int e = tid; e < Q * N / 8; e += kSsdThreads)
                dst[e] = src[e];
        }
        if (tid == 0 && !ok)
            record_fault(a.fault, kFaultMmaTimeout);
        tc_fence_before();
        __syncthreads();
        if (warp == 0)
            tmem_dealloc(tm, COLS);
        return;
    }

    copy_tile<T, Q, N>(static_cast<const T *>(a.B) + (b * a.L + t0) * N, N, rows, rB);
    for (int j = 0; j < nh; ++j)
        copy_tile<T, Q, P>(static_cast<const T *>(a.x) + ((b * a.L + t0) * a.H + h0 + j) * P, a.H * P, rows,
                           rX + j * Q * P);
    ssd_cp_commit();
    if (tid == 0) {
        mbar_init(&mbar, 1);
        fence_mbar_init();
    }
    if (warp < nh)   // warp j: head j's step sizes and decays
        ssd_decays(a, b, h0 + warp, t0, rows, dl + warp * Q, s + warp * Q);
    ssd_cp_wait();
    __syncthreads();
    for (int e = tid; e < nh * Q; e += kSsdThreads)   // w = exp(s_last - s_t) dl_t, head e / Q
        w[e] = ex2((s[(e / Q) * Q + Q - 1] - s[e]) * kLog2e) * dl[e];
    __syncthreads();
    transpose_to_operand<T, Q, N>(rB, nullptr, A3);
    for (int j = 0; j < nh; ++j)
        transpose_to_operand<T, Q, P>(rX + j * Q * P, w + j * Q, BX + j * P * Q);
    fence_proxy_async_smem();   // the tensor core reads shared memory through the async proxy
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = tbase;
    if (tid == 0) {
        constexpr uint32_t id = umma_idesc_f16(N, P);
        for (int j = 0; j < nh; ++j) {
#pragma unroll
            for (int kk = 0; kk < Q / 16; ++kk)
                umma_f16(tm + (uint32_t)(j * P), umma_tile_desc(A3, Q, kk), umma_tile_desc(BX + j * P * Q, Q, kk),
                         id, kk > 0);
        }
        umma_commit(&mbar);
    }
    const bool ok = mma_wait(&mbar, 0);
    tc_fence_after();
    grid_dep_trigger();
    // Row n of S sits in TMEM lane n (N = 128) or lane 32w + (n - 16w) (N = 64);
    // a warp's lanes hold consecutive n, so the [p][n] stores coalesce.
    const int n = N == 128 ? 32 * warp + lane : 16 * warp + lane;
    const bool mine = ok && (N == 128 || lane < 16);
    for (int j = 0; j < nh; ++j) {
        __half *dst = a.S + ((b * a.H + h0 + j) * a.nch + c) * N * P + n;
#pragma unroll
        for (int p0 = 0; p0 < P; p0 += 16) {
            float v[16];
            tmem_ld16(tm + ((uint32_t)(32 * warp) << 16) + (uint32_t)(j * P + p0), v);
            if (mine) {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    dst[(p0 + i) * N] = __float2half_rn(v[i]);
            }
        }
    }
    if (tid < nh)
        a.dec[(b * a.H + h0 + tid) * a.nch + c] = ex2(s[tid * Q + Q - 1] * kLog2e);
    if (tid == 0 && !ok)
        record_fault(a.fault, kFaultMmaTimeout);
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        tmem_dealloc(tm, COLS);
}

// 2. The state entering each chunk, in chunk order: fp32 carries, stored as
// fp16 in the output kernel's operand order (P rows, K = N, core-matrix
// order), and hT ([n][p], fp32). A thread owns four consecutive n of one p
// (half a 16-byte core row); consecutive threads take consecutive half rows
// of the operand, so a warp's stores are 256 contiguous bytes (and its loads
// of the [p][n] chunk states 32-byte runs). The chunk states are loaded
// kCarryBatch chunks ahead of the serial fold.
constexpr int kCarryBatch = 8;
constexpr int kCarryE = 4;   // n per thread

template <int N, int P>
__global__ void __launch_bounds__(256) ssd_carry_kernel(const SsdArgs a)
{
    constexpr int NP = N * P, E = kCarryE;
    grid_dep_wait();      // the chunk states and decays of the state kernel
    grid_dep_trigger();   // the output kernel may start its own loads
    const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (i >= a.Bsz * a.H * (NP / E))
        return;
    const int64_t bh = i / (NP / E);
    const int hr = (int)(i - bh * (NP / E));           // half row hr of the operand
    const int r = hr >> 1, q0 = (hr & 1) * E;          // core row r, its n offset
    const int p = ((r >> 3) / (N / 8)) * 8 + (r & 7), n0 = ((r >> 3) % (N / 8)) * 8 + q0;
    const int pn = p * N + n0;
    float carry[E];
#pragma unroll
    for (int q = 0; q < E; ++q)
        carry[q] = a.h0 ? __ldg(a.h0 + bh * NP + (int64_t)(n0 + q) * P + p) : 0.0f;
    const __half *Sp = a.S + bh * a.nch * NP + pn;
    __half *Hp = a.Hin + bh * a.nch * NP + (int64_t)r * 8 + q0;   // = core_index(p, n0, N)
    const float *dp = a.dec + bh * a.nch;
    for (int c0 = 0; c0 < a.nch; c0 += kCarryBatch) {
        uint2 sv[kCarryBatch];
        float dv[kCarryBatch];
#pragma unroll
        for (int j = 0; j < kCarryBatch; ++j) {
            const int cc = c0 + j < a.nch ? c0 + j : a.nch - 1;
            sv[j] = __ldcg(reinterpret_cast<const uint2 *>(Sp + (int64_t)cc * NP));
            dv[j] = __ldg(dp + cc);
        }
#pragma unroll
        for (int j = 0; j < kCarryBatch; ++j) {
            if (c0 + j < a.nch) {
                uint2 o;
                __half2 *oh = reinterpret_cast<__half2 *>(&o);
                oh[0] = __floats2half2_rn(carry[0], carry[1]);
                oh[1] = __floats2half2_rn(carry[2], carry[3]);
                *reinterpret_cast<uint2 *>(Hp + (int64_t)(c0 + j) * NP) = o;
                const __half2 *hs = reinterpret_cast<const __half2 *>(&sv[j]);
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const float2 f = __half22float2(hs[q]);
                    carry[2 * q] = fmaf(dv[j], carry[2 * q], f.x);
                    carry[2 * q + 1] = fmaf(dv[j], carry[2 * q + 1], f.y);
                }
            }
        }
    }
    if (a.hT) {
#pragma unroll
        for (int q = 0; q < E; ++q)
            a.hT[bh * NP + (int64_t)(n0 + q) * P + p] = carry[q];
    }
}

// 3. Each chunk's outputs: the masked dual form inside the chunk plus the
// decayed incoming state.
template <int P>
__host__ __device__ constexpr int ssd_out_cols()   // TMEM columns: G X (P) and C H_in (P)
{
    return 2 * P <= 32 ? 32 : (2 * P <= 64 ? 64 : (2 * P <= 128 ? 128 : 256));
}

// The first shared-memory region holds the X tile until it is transposed,
// then the incoming state's operand.
template <typename T, int N, int P>
__host__ __device__ constexpr int ssd_out_region1()
{
    return P * N * 2 > kSsdQ * P * (int)sizeof(T) ? P * N * 2 : kSsdQ * P * (int)sizeof(T);
}

template <typename T, int N, int P>
__global__ void __launch_bounds__(kSsdThreads) ssd_out_kernel(const SsdArgs a)
{
    constexpr int Q = kSsdQ;
    constexpr int COLS = ssd_out_cols<P>();
    extern __shared__ __align__(1024) unsigned char sm[];
    __half *B4 = reinterpret_cast<__half *>(sm);                        // H_in^T: P rows, K = N ...
    T *rX = reinterpret_cast<T *>(sm);                                  // ... after the X tile [Q][P]
    __half *A1 = reinterpret_cast<__half *>(sm + ssd_out_region1<T, N, P>());   // C: Q rows, K = N
    __half *BX = A1 + Q * N;                                            // X^T: P rows, K = Q
    __half *GA = BX + P * Q;                                            // C B^T, then masked: Q rows, K = Q
    float *dl = reinterpret_cast<float *>(GA + Q * Q);
    float *s = dl + Q;
    float *es = s + Q;
    float *wr = es + Q;   // exp(-s_r) dl_r
    __shared__ uint32_t tbase;
    __shared__ __align__(8) uint64_t mbar;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t b = blockIdx.z, h = blockIdx.y, c = blockIdx.x;
    const int64_t t0 = c * Q;
    const int rows = (int)min((int64_t)Q, a.L - t0);
    const bool carry = c > 0 || a.h0 != nullptr;
    if (warp == 0)   // first, as in the state kernel
        tmem_alloc(&tbase, COLS);
    // The call's own inputs, and what the state kernel wrote (C B^T and C,
    // already in operand order): this kernel starts only once every CTA of
    // the carry kernel has passed its own wait for the state kernel, so that
    // kernel has completed. The incoming state, the carry kernel's result,
    // comes once the X tile is out of its space.
    copy_tile<T, Q, P>(static_cast<const T *>(a.x) + ((b * a.L + t0) * a.H + h) * P, a.H * P, rows, rX);
    SsdDt dtv{};
    if (warp == 0)
        dtv = ssd_dt_load(a, b, h, t0, rows);
    copy_tile<__half, Q, Q>(a.G + (b * a.nch + c) * Q * Q, Q, Q, GA);
    copy_tile<__half, Q, N>(a.Cop + (b * a.nch + c) * Q * N, N, Q, A1);
    ssd_cp_commit();
    if (tid == 0) {
        mbar_init(&mbar, 1);
        fence_mbar_init();
    }
    if (warp == 0)
        ssd_decays_from(a, dtv, rows, dl, s);
    ssd_cp_wait();
    __syncthreads();
    if (tid < Q) {
        es[tid] = ex2(s[tid] * kLog2e);
        wr[tid] = ex2(-s[tid] * kLog2e) * dl[tid];
    }
    transpose_to_operand<T, Q, P>(rX, nullptr, BX);
    // The X tile is consumed. exp(s_t - s_r) = exp(s_t) exp(-s_r) when no
    // |s| exceeds 80 (both factors then stay inside fp32's normal range);
    // otherwise each term takes its own exponential.
    const bool wide = __syncthreads_or(tid < Q && !(fabsf(s[tid]) <= 80.0f));
    // Every CTA waits for the carry kernel, also when it reads nothing of it,
    // so that this grid never completes before that one.
    grid_dep_wait();
    if (carry) {
        copy_tile<__half, P, N>(a.Hin + ((b * a.H + h) * a.nch + c) * N * P, N, P, B4);
        ssd_cp_commit();
    }
    // Mask, decay and scale C B^T in place into the masked product's A
    // operand while the incoming state arrives: every thread takes one core
    // row (eight columns of one row) at a time.
#pragma unroll 2
    for (int e = tid; e < Q * (Q / 8); e += kSsdThreads) {
        const int t = e / (Q / 8), r0 = (e % (Q / 8)) * 8;
        uint4 *cell = reinterpret_cast<uint4 *>(GA + core_index(t, r0, Q));
        const uint4 graw = *cell;
        const __half2 *g2 = reinterpret_cast<const __half2 *>(&graw);
        const float st = s[t], et = es[t];
        float m[8];
        if (!wide) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 gf = __half22float2(g2[i]);
                const int r = r0 + 2 * i;
                m[2 * i] = r <= t ? gf.x * et * wr[r] : 0.0f;
                m[2 * i + 1] = r + 1 <= t ? gf.y * et * wr[r + 1] : 0.0f;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 gf = __half22float2(g2[i]);
                const int r = r0 + 2 * i;
                m[2 * i] = r <= t ? gf.x * ex2((st - s[r]) * kLog2e) * dl[r] : 0.0f;
                m[2 * i + 1] = r + 1 <= t ? gf.y * ex2((st - s[r + 1]) * kLog2e) * dl[r + 1] : 0.0f;
            }
        }
        *cell = pack8(m);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tY = tbase, tH = tbase + P;
    if (tid == 0) {
        constexpr uint32_t id = umma_idesc_f16(Q, P);
#pragma unroll
        for (int kk = 0; kk < Q / 16; ++kk)
            umma_f16(tY, umma_tile_desc(GA, Q, kk), umma_tile_desc(BX, Q, kk), id, kk > 0);
    }
    if (carry) {
        ssd_cp_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    if (tid == 0) {
        if (carry) {
            constexpr uint32_t id = umma_idesc_f16(Q, P);
#pragma unroll
            for (int kk = 0; kk < N / 16; ++kk)
                umma_f16(tH, umma_tile_desc(A1, N, kk), umma_tile_desc(B4, N, kk), id, kk > 0);
        }
        umma_commit(&mbar);   // both products
    }
    const bool ok = mma_wait(&mbar, 0);
    tc_fence_after();
    grid_dep_trigger();   // the next call's state kernel may be scheduled
    // Row t of each product sits in lane 32w + (t - 16w) of warp w (M = 64).
    const int t = 16 * warp + lane;
    const uint32_t lanes = (uint32_t)(32 * warp) << 16;
    T *yg = static_cast<T *>(a.y) + ((b * a.L + t0 + t) * a.H + h) * P;
    const bool mine = ok && lane < 16 && t < rows;
    const float et = es[t < Q ? t : 0];
#pragma unroll
    for (int p0 = 0; p0 < P; p0 += 16) {
        uint32_t vr[16], hr[16];
        tmem_ld16_async(tY + lanes + (uint32_t)p0, vr);
        if (carry)
            tmem_ld16_async(tH + lanes + (uint32_t)p0, hr);
        tmem_wait_ld();
        float v[16], hv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            v[i] = __uint_as_float(vr[i]);
            hv[i] = __uint_as_float(hr[i]);
        }
        if (mine) {
            if (carry) {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    v[i] = fmaf(et, hv[i], v[i]);
            }
            if constexpr (sizeof(T) == 2) {
                uint4 u[2];
                uint32_t *wd = reinterpret_cast<uint32_t *>(u);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const __nv_bfloat162 q = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
                    wd[i] = *reinterpret_cast<const uint32_t *>(&q);
                }
                reinterpret_cast<uint4 *>(yg + p0)[0] = u[0];
                reinterpret_cast<uint4 *>(yg + p0)[1] = u[1];
            } else {
#pragma unroll
                for (int i = 0; i < 16; i += 4)
                    *reinterpret_cast<float4 *>(yg + p0 + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
            }
        }
    }
    if (tid == 0 && !ok)
        record_fault(a.fault, kFaultMmaTimeout);
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        tmem_dealloc(tbase, COLS);
}

template <typename T, int N, int P>
constexpr size_t ssd_state_smem()
{
    constexpr size_t hpc = (size_t)ssd_state_heads<T, P>();
    return ((size_t)N + hpc * P) * kSsdQ * 2 + (size_t)kSsdQ * ((size_t)N + hpc * P) * sizeof(T) +
           3 * hpc * kSsdQ * 4;
}

// The X tile and the incoming state's operand share their space; C B^T is
// masked in place.
template <typename T, int N, int P>
constexpr size_t ssd_out_smem()
{
    return (size_t)ssd_out_region1<T, N, P>() + ((size_t)kSsdQ * N + (size_t)P * kSsdQ + (size_t)kSsdQ * kSsdQ) * 2 +
           4 * kSsdQ * 4;
}

// Shared memory that keeps at most max_ctas CTAs of a kernel on one SM, so
// that their TMEM allocations never exceed the SM's 512 columns: max_ctas + 1
// CTAs (each with the 1 KB the runtime reserves) must not fit in the SM's
// 228 KB. Never above the 227 KB a CTA may have.
inline size_t ssd_pad(size_t smem, int max_ctas)
{
    constexpr size_t kSm = (size_t)228 * 1024, kReserved = 1024, kMax = (size_t)227 * 1024;
    size_t pad = kSm / (size_t)(max_ctas + 1) - kReserved + 1;
    if (pad > kMax) pad = kMax;
    return smem > pad ? smem : pad;
}

template <typename T, int N, int P>
int launch_ssd_t(const SsdArgs &a, cudaStream_t st)
{
    auto k1 = ssd_state_kernel<T, N, P>;
    auto k3 = ssd_out_kernel<T, N, P>;
    const size_t s1 = ssd_pad(ssd_state_smem<T, N, P>(), 512 / ssd_state_cols<T, P>());
    const size_t s3 = ssd_pad(ssd_out_smem<T, N, P>(), 512 / ssd_out_cols<P>());
    cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k3, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s3);
    // All of the SM's unified L1/shared storage as shared memory: these
    // kernels read their tiles through cp.async and __ldg only.
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k1, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k3, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return cuda_fail(e, "SSD kernel attributes");
    const dim3 grid((unsigned)a.nch, (unsigned)a.H, (unsigned)a.Bsz);
    const unsigned groups = (unsigned)((a.H + ssd_state_heads<T, P>() - 1) / ssd_state_heads<T, P>());
    const int64_t total = a.Bsz * a.H * (int64_t)(N * P / kCarryE);
    // All three kernels start early (programmatic dependent launch) and wait
    // in the kernel for what the one before wrote.
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    {
        cudaLaunchConfig_t cfg1 = {};
        cfg1.gridDim = dim3(grid.x, groups + 1, grid.z);   // + the C B^T CTAs
        cfg1.blockDim = dim3(kSsdThreads);
        cfg1.dynamicSmemBytes = s1;
        cfg1.stream = st;
        cfg1.attrs = pdl;
        cfg1.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg1, k1, a);
        if (e != cudaSuccess) return cuda_fail(e, "SSD state kernel launch");
    }
    cudaLaunchConfig_t cfg2 = {};
    cfg2.gridDim = dim3((unsigned)((total + 255) / 256));
    cfg2.blockDim = dim3(256);
    cfg2.stream = st;
    cfg2.attrs = pdl;
    cfg2.numAttrs = 1;
    e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg2, ssd_carry_kernel<N, P>, a);
    cudaLaunchConfig_t cfg3 = cfg2;
    cfg3.gridDim = grid;
    cfg3.blockDim = dim3(kSsdThreads);
    cfg3.dynamicSmemBytes = s3;
    if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg3, k3, a);
    if (e == cudaSuccess) e = cudaGetLastError();
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
    if (Bsz > 65535 || H > 65534)
        return fail(SELSCAN_ERR_UNSUPPORTED, "SSD: Bsz must be at most 65535 and H at most 65534");
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
    // Workspace: S and the incoming states (fp16), C B^T and C of every
    // chunk as fp16 operands, the chunk decays.
    const size_t sbytes = (size_t)(Bsz * H * nch) * (size_t)(N * P) * 2, hbytes = sbytes,
                 gbytes = (size_t)(Bsz * nch) * kSsdQ * kSsdQ * 2, cbytes = (size_t)(Bsz * nch) * kSsdQ * N * 2,
                 dbytes = (size_t)(Bsz * H * nch) * 4;
    const size_t total = sbytes + hbytes + gbytes + cbytes + dbytes;
    void *ws = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&ws, total, pool, st);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(SELSCAN_ERR_NO_MEMORY, "SSD workspace of %zu bytes: %s", total, cudaGetErrorString(e));
    }
    SsdArgs a;
    memset(&a, 0, sizeof a);
    a.x = x; a.dt = dt; a.A = A; a.B = B; a.C = C; a.y = y; a.h0 = h0; a.hT = hT;
    a.S = static_cast<__half *>(ws);
    a.Hin = reinterpret_cast<__half *>(static_cast<char *>(ws) + sbytes);
    a.G = reinterpret_cast<__half *>(static_cast<char *>(ws) + sbytes + hbytes);
    a.Cop = reinterpret_cast<__half *>(static_cast<char *>(ws) + sbytes + hbytes + gbytes);
    a.dec = reinterpret_cast<float *>(static_cast<char *>(ws) + sbytes + hbytes + gbytes + cbytes);
    a.Bsz = Bsz; a.L = L; a.H = H;
    a.nch = (int)nch;
    a.softplus = dt_softplus ? 1 : 0;
    rc = fault_word(dev, st, &a.fault);
    if (rc == SELSCAN_OK)
        rc = dtype == SELSCAN_F32 ? launch_ssd<float>(a, N, P, st) : launch_ssd<__nv_bfloat16>(a, N, P, st);
    cudaFreeAsync(ws, st);
    return rc;
}
