// scan_fused.cuh -- the whole forward scan in one persistent kernel.
//
// Work items. The sequence is cut into K chunks; the channels into tiles of
// DPB = 128 / NSPLIT; G = Bsz * tiles groups. Items are numbered
//     0 .. (K-1)*G - 1          aggregate items (chunk k < K-1, group g), k-major
//     (K-1)*G .. (2K-1)*G - 1   readout items  (chunk k,       group g), k-major
// and CTAs take them in that order from an atomic ticket counter. An
// aggregate item scans its chunk from a zero state and publishes the pair
// (decay[n] = exp(A[d,n] * sum dl), end[n]), as sum dl and end[n] -- one operand of the
// associative composition (a1,b1) o (a2,b2) = (a2 a1, a2 b1 + b2) of the
// parallel scan (booiljung.github.io "3.1 LTI systems ...", section 3.1.5.2)
// -- then raises its done flag. A readout item folds the published pairs of
// chunks 0..k-1 of its group onto h0 to get its incoming state, rescans its
// chunk and writes y (and hT from the last chunk).
//
// Progress. A readout item waits only on aggregate items, whose tickets are
// all smaller than its own: they were taken by CTAs already running, which
// never wait while they hold an aggregate item. So every wait ends, whatever
// the number of resident CTAs. Waits are bounded anyway (tma.cuh).
//
// Inputs arrive as 3-D TMA boxes of TT timesteps (x, delta: TT x DPB; B, C:
// TT x N) into a ring of shared-memory buffers, with "full" mbarriers (TMA
// completion, with the expected byte count) and "empty" mbarriers (one
// arrival per warp when it is done with a buffer). The warp whose arrival
// completes an empty barrier refills that buffer with the stage STAGES ahead;
// it learns that from the arrival's result one stage later, so no warp ever
// waits for another. Boxes that run past D or L are zero-filled by the TMA
// unit; those lanes and rows are never stored.
#pragma once

#include <type_traits>

#include "device_math.cuh"
#include "scan_fwd.cuh"
#include "scan_tma.cuh"
#include "tma.cuh"

namespace selscan {

struct FusedArgs {
    CUtensorMap mx, md, mB, mC;
    CUtensorMap mz;       // the gate's z, like x (GATE kernels with z only)
    ScanArgs s;
    float *aggS;          // (K-1, Bsz, D): sum of dl over the chunk
    float *aggH;          // (K-1, Bsz, D, N): chunk end state from zero
    unsigned *ctrl;       // [0]: ticket counter; [1 + k*G + g]: aggregate done flags (zeroed per call)
    unsigned *fault;      // fault word of the launching stream
    uint64_t wait_ns;     // limit of a readout's wait for the done flags
    int publish;          // 0 only for the timeout test: aggregates raise no flags
    int alias_wait;       // y is x, delta or z: readout k also waits for aggregate k, which reads those rows
    int stages;
    int groups;           // G
    int items_agg;        // (K-1) * G
    int items_total;      // items_agg + K * G
};

constexpr unsigned kFaultFlagTimeout = 2;   // a chunk aggregate never appeared
constexpr int kFoldBatch = 4;               // chunk pairs in flight per fold round

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_u32(unsigned *p, unsigned v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Arrives on the barrier; returns the state of the phase arrived on.
__device__ __forceinline__ uint64_t mbar_arrive_state(uint64_t *bar)
{
    uint64_t st;
    asm volatile("mbarrier.arrive.shared::cta.b64 %0, [%1];" : "=l"(st) : "r"(smem_u32(bar)) : "memory");
    return st;
}

// Arrivals still pending in a phase state, before the arrival that returned it.
__device__ __forceinline__ uint32_t mbar_pending(uint64_t st)
{
    uint32_t n;
    asm volatile("mbarrier.pending_count.b64 %0, %1;" : "=r"(n) : "l"(st));
    return n;
}

// Whether the phase captured in `st` has completed (acquire ordering).
__device__ __forceinline__ bool mbar_test_state(uint64_t *bar, uint64_t st)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "l"(st)
        : "memory");
    return done != 0;
}

template <int NS, bool VEC>
__device__ __forceinline__ void load_state_cg(const float *p, int valid, float2 (&v)[NS / 2])
{
    if (VEC) {
#pragma unroll
        for (int j = 0; j < NS / 2; j += 2) {
            const float4 w = __ldcg(reinterpret_cast<const float4 *>(p) + j / 2);
            v[j] = make_float2(w.x, w.y);
            v[j + 1] = make_float2(w.z, w.w);
        }
    } else {
#pragma unroll
        for (int j = 0; j < NS / 2; ++j)
            v[j] = make_float2(2 * j < valid ? __ldcg(p + 2 * j) : 0.0f,
                               2 * j + 1 < valid ? __ldcg(p + 2 * j + 1) : 0.0f);
    }
}

// GATE: the readout also applies the block's skip and gate (block_out),
// with z staged beside x in the ring.
// The zero-order-hold input term of a pair of states, packed and without a
// branch or a divide: the coefficient dl * phi(w) (see zoh_coef) is the
// series where |w| < 1/16 and (decay - 1) / A elsewhere, with 1/A held per
// item (0 where A is 0, where the series is taken). e = dl * A * log2(e).
__device__ __forceinline__ float2 zoh_pair(float2 dl2, float2 e, float2 decay, float2 ainv, float2 xb)
{
    const float2 w = __fmul2_rn(e, make_float2(kLn2, kLn2));
    float2 p = __ffma2_rn(w, make_float2(1.0f / 24.0f, 1.0f / 24.0f), make_float2(1.0f / 6.0f, 1.0f / 6.0f));
    p = __ffma2_rn(w, p, make_float2(0.5f, 0.5f));
    p = __ffma2_rn(w, p, make_float2(1.0f, 1.0f));
    p = __fmul2_rn(p, dl2);
    const float2 q = __fmul2_rn(__fadd2_rn(decay, make_float2(-1.0f, -1.0f)), ainv);
    const float2 c = make_float2(fabsf(w.x) < 0.0625f ? p.x : q.x, fabsf(w.y) < 0.0625f ? p.y : q.y);
    return __fmul2_rn(c, xb);
}

// ZOH: the zero-order-hold input term (zoh_pair) in place of dl * B * x.
template <typename T, int NS, int NSPLIT, bool VEC, int TT, bool SOFTPLUS, bool GATE, bool ZOH = false>
// Three CTAs per SM fit the shared-memory ring; the register cap this implies
// (168) is above what the kernel needs, and measured faster than 128.
__global__ void __launch_bounds__(kScanThreads, 3)
scan_fused_kernel(const __grid_constant__ FusedArgs fa)
{
    static_assert(NS % 4 == 0, "states are processed in pairs of pairs");
    static_assert(TT % 2 == 0, "timesteps are processed in pairs");
    constexpr int DPB = kScanThreads / NSPLIT;
    constexpr int NP = NS / 2;
    constexpr int kWarps = kScanThreads / 32;
    const ScanArgs &a = fa.s;
    const int STAGES = fa.stages;

    extern __shared__ __align__(128) unsigned char smem[];
    // Row stride of the B/C tiles: N, a compile-time constant on the vector path.
    const int64_t Nrow = VEC ? (int64_t)(NS * NSPLIT) : a.N;
    const int64_t N = a.N, D = a.D, L = a.L;
    const int xbytes = TT * DPB * (int)sizeof(T);
    const int nbytes = TT * (int)Nrow * (int)sizeof(T);
    const int sbytes = 2 * xbytes + 2 * nbytes + (GATE ? xbytes : 0);
    const bool has_z = GATE && a.z != nullptr;
    // Bytes a stage brings: x, delta and B, plus C (and z) for a readout.
    const int agg_bytes = 2 * xbytes + nbytes;
    const int ro_bytes = 2 * xbytes + 2 * nbytes + (has_z ? xbytes : 0);
    constexpr bool kBf16 = sizeof(T) == 2;
    const int cfloats = kBf16 ? 2 * TT * (int)Nrow : 0;   // fp32 copy of a stage's B and C rows
    float *conv_buf = reinterpret_cast<float *>(smem + STAGES * sbytes);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * (sbytes + cfloats * 4));
    uint64_t *empty = full + STAGES;
    uint64_t *conv = empty + STAGES;   // bf16: every warp converted its share of the stage
    unsigned *issued = reinterpret_cast<unsigned *>(conv + STAGES);
    volatile int *s_item = reinterpret_cast<volatile int *>(issued + STAGES);
    volatile int *s_abort = s_item + 1;

    const int grp = threadIdx.x / NSPLIT;
    const int q = threadIdx.x % NSPLIT;
    const int lane = threadIdx.x & 31;
    const int n0 = q * NS;
    const int64_t left = N - n0;
    const int valid = left <= 0 ? 0 : (left >= NS ? NS : (int)left);

    if (threadIdx.x == 0) {
        prefetch_tensormap(&fa.mx);
        prefetch_tensormap(&fa.md);
        prefetch_tensormap(&fa.mB);
        prefetch_tensormap(&fa.mC);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWarps);
            mbar_init(&conv[s], kWarps);
            issued[s] = 0;
        }
        *s_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    uint32_t ring = 0;   // buffers this CTA has consumed so far (all items)

    for (int round = 0;; ++round) {
        // With a ticket counter CTAs stay resident and take items in order;
        // without one (a single chunk: no dependences) CTA x runs item x.
        if (threadIdx.x == 0)
            *s_item = fa.ctrl ? (int)atomicAdd(&fa.ctrl[0], 1u) : (round == 0 ? (int)blockIdx.x : fa.items_total);
        __syncthreads();
        const int item = *s_item;
        if (item >= fa.items_total || *s_abort)
            break;
        const bool readout = item >= fa.items_agg;
        const int idx = readout ? item - fa.items_agg : item;
        const int k = idx / fa.groups;
        const int g = idx - k * fa.groups;
        const int64_t b = g / a.dtiles;
        const int d0 = (g % a.dtiles) * DPB;
        const int64_t d_raw = (int64_t)d0 + grp;
        const bool active = d_raw < D;
        const int64_t d = active ? d_raw : D - 1;
        const int64_t t0 = (int64_t)k * a.chunk;
        const int64_t nsteps = min(L, t0 + a.chunk) - t0;
        const int nst = (int)((nsteps + TT - 1) / TT);

        auto buf = [&](uint32_t r) { return smem + (r % STAGES) * sbytes; };
        auto issue = [&](uint32_t r, int i) {   // stage i of this item into ring slot r
            const int s = (int)(r % STAGES);
            unsigned char *p = buf(r);
            const int t = (int)(t0 + (int64_t)i * TT);
            issued[s] += 1;
            mbar_arrive_expect_tx(&full[s], (uint32_t)(readout ? ro_bytes : agg_bytes));
            tma_load_3d(p, &fa.mx, &full[s], d0, t, (int)b);
            tma_load_3d(p + xbytes, &fa.md, &full[s], d0, t, (int)b);
            tma_load_3d(p + 2 * xbytes, &fa.mB, &full[s], 0, t, (int)b);
            if (readout)
                tma_load_3d(p + 2 * xbytes + nbytes, &fa.mC, &full[s], 0, t, (int)b);
            if (readout && has_z)
                tma_load_3d(p + 2 * xbytes + 2 * nbytes, &fa.mz, &full[s], d0, t, (int)b);
        };

        // Every warp finished the previous item: its buffers may be refilled.
        if (threadIdx.x == 0) {
            fence_proxy_async_smem();
            for (int f = 0; f < STAGES && f < nst; ++f)
                issue(ring + f, f);
        }

        const float dsk = (GATE && readout && a.Dskip) ? __ldg(a.Dskip + d) : 0.0f;
        float2 A2[NP];
        float2 Ainv[ZOH ? NP : 1];   // 1/A for the zero-order hold (0 where A is 0)
#pragma unroll
        for (int j = 0; j < NP; ++j) {
            const float lo = (2 * j < valid) ? __ldg(a.A + d * N + n0 + 2 * j) : 0.0f;
            const float hi = (2 * j + 1 < valid) ? __ldg(a.A + d * N + n0 + 2 * j + 1) : 0.0f;
            A2[j] = make_float2(lo * kLog2e, hi * kLog2e);
            if constexpr (ZOH)
                Ainv[j] = make_float2(lo != 0.0f ? __frcp_rn(lo) : 0.0f, hi != 0.0f ? __frcp_rn(hi) : 0.0f);
        }

        // Incoming state: h0 (or zeros), and for a readout of chunk k >= 1
        // the fold of the published pairs of chunks 0..k-1.
        float2 h[NP];
        if (readout && a.h0) {
            load_state_cg<NS, false>(a.h0 + (b * D + d) * N + n0, valid, h);
        } else {
#pragma unroll
            for (int j = 0; j < NP; ++j)
                h[j] = make_float2(0.0f, 0.0f);
        }
        // Flags a readout waits for: chunks 0..k-1 (their pairs are folded),
        // and chunk k as well when y overwrites an input that chunk k's
        // aggregate item reads (in-place output).
        const int kwait = readout ? (fa.alias_wait ? min(k + 1, a.K - 1) : k) : 0;
        if (kwait > 0) {
            // Warp 0 checks the done flags, 32 per round trip.
            if (threadIdx.x < 32) {
                const uint64_t tstart = global_ns();
                for (int j0 = 0; j0 < kwait; j0 += 32) {
                    const int j = j0 + lane;
                    const unsigned *f = fa.ctrl + 1 + (int64_t)j * fa.groups + g;
                    bool done = j >= kwait || ld_acquire_u32(f) != 0u;
                    while (!__all_sync(0xffffffffu, done)) {
                        if (!done)
                            done = ld_acquire_u32(f) != 0u;
                        // Warp-uniform decision: every lane leaves together.
                        if (__any_sync(0xffffffffu, global_ns() - tstart > fa.wait_ns)) {
                            if (lane == 0) {
                                record_fault(fa.fault, kFaultFlagTimeout);
                                *s_abort = 1;
                            }
                            break;
                        }
                    }
                    __syncwarp();
                    if (*s_abort)
                        break;
                }
            }
            __syncthreads();
            if (*s_abort)
                break;
        }
        if (readout && k > 0) {
            // Fold the pairs of chunks 0..k-1, kFoldBatch at a time: all loads
            // of a batch are issued before the first is used. A chunk's decay
            // exp(A * sum dl) is rebuilt here from its sum of dl, exactly as the
            // aggregate item would have computed it.
            const int64_t bd_all = (int64_t)a.Bsz * D;
            const int64_t slot = bd_all * N;
            const int64_t off = (b * D + d) * N + n0;
            const float *Sp = fa.aggS + b * D + d;
            for (int j0 = 0; j0 < k; j0 += kFoldBatch) {
                float S[kFoldBatch];
                float2 E[kFoldBatch][NP];
#pragma unroll
                for (int jj = 0; jj < kFoldBatch; ++jj) {
                    const int64_t j = j0 + jj < k ? j0 + jj : k - 1;   // past the end: a repeat, unused
                    S[jj] = __ldcg(Sp + j * bd_all);
                    load_state_cg<NS, VEC>(fa.aggH + j * slot + off, valid, E[jj]);
                }
#pragma unroll
                for (int jj = 0; jj < kFoldBatch; ++jj) {
                    if (j0 + jj < k) {
                        const float2 s2 = make_float2(S[jj], S[jj]);
#pragma unroll
                        for (int i = 0; i < NP; ++i) {
                            const float2 e = __fmul2_rn(s2, A2[i]);
                            h[i] = __ffma2_rn(make_float2(ex2(e.x), ex2(e.y)), h[i], E[jj][i]);
                        }
                    }
                }
            }
        }

        T *yp = static_cast<T *>(a.y) + (b * L + t0) * D + d;
        float s_sum = 0.0f, s_err = 0.0f;
        bool ok = true;
        // The stage loop, compiled once per item role so that each unrolled
        // step is straight-line code.
        auto run_stages = [&](auto role) {
            constexpr bool RO = decltype(role)::value;

            // Refills: the warp whose arrival completes a buffer's empty barrier
            // (every warp is done with it) loads that buffer with the stage
            // STAGES ahead. The arrival's result is inspected one stage later, so
            // no warp waits for it.
            uint64_t rel_state = 0;   // lane 0: state of this warp's last arrival
            int rel_stage = -1;       // the stage that arrival released

            for (int i = 0; i < nst; ++i) {
                const uint32_t r = ring + i;
                const int s = (int)(r % STAGES);
                const bool arrived = mbar_wait(&full[s], (r / STAGES) & 1u);
                if (!__all_sync(0xffffffffu, arrived)) {
                    ok = false;
                    break;
                }
                const unsigned char *p = buf(r);
                const T *xs = reinterpret_cast<const T *>(p) + grp;
                const T *ds = reinterpret_cast<const T *>(p + xbytes) + grp;
                const T *zs = reinterpret_cast<const T *>(p + 2 * xbytes + 2 * nbytes) + grp;
                // B and C rows in fp32: straight from the tile, or (bf16
                // input) from this stage's fp32 copy, which the four warps
                // convert together -- every thread needs every row, so
                // converting once per CTA instead of once per thread saves
                // most of the unpacking work.
                const float *Bs;
                const float *Cs;
                if constexpr (kBf16) {
                    float *cb = conv_buf + s * cfloats;
                    const __nv_bfloat16 *src = reinterpret_cast<const __nv_bfloat16 *>(p + 2 * xbytes);
                    const int total = (RO ? 2 : 1) * TT * (int)Nrow;
                    for (int e = threadIdx.x; e < total; e += kScanThreads)
                        cb[e] = __bfloat162float(src[e]);
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&conv[s]);
                    if (!__all_sync(0xffffffffu, mbar_wait(&conv[s], (r / STAGES) & 1u))) {
                        ok = false;
                        break;
                    }
                    Bs = cb + n0;
                    Cs = cb + TT * Nrow + n0;
                } else {
                    Bs = reinterpret_cast<const float *>(p + 2 * xbytes) + n0;
                    Cs = reinterpret_cast<const float *>(p + 2 * xbytes + nbytes) + n0;
                }
                const int64_t rem = nsteps - (int64_t)i * TT;
                const int tc = rem < TT ? (int)rem : TT;

                // Phase 1, breadth first: TT independent softplus evaluations
                // advance together, so their dependent FMAs interleave.
                float dlv[TT], uv[TT];
#pragma unroll
                for (int tt = 0; tt < TT; ++tt)
                    dlv[tt] = smem_val(ds + tt * DPB);
                // Pairs of timesteps share one packed fp32x2 instruction; each
                // lane rounds exactly as the scalar operation would.
                if constexpr (SOFTPLUS) {
                    float2 ev[TT / 2], pv[TT / 2];
#pragma unroll
                    for (int j = 0; j < TT / 2; ++j) {
                        ev[j] = make_float2(ex2(-fabsf(dlv[2 * j]) * kLog2e), ex2(-fabsf(dlv[2 * j + 1]) * kLog2e));
                        pv[j] = make_float2(kLog1pPoly[8], kLog1pPoly[8]);
                    }
#pragma unroll
                    for (int c = 7; c >= 0; --c) {
#pragma unroll
                        for (int j = 0; j < TT / 2; ++j)
                            pv[j] = __ffma2_rn(pv[j], ev[j], make_float2(kLog1pPoly[c], kLog1pPoly[c]));
                    }
#pragma unroll
                    for (int j = 0; j < TT / 2; ++j) {
                        const float2 r = __ffma2_rn(pv[j], ev[j], make_float2(fmaxf(dlv[2 * j], 0.0f), fmaxf(dlv[2 * j + 1], 0.0f)));
                        dlv[2 * j] = r.x;
                        dlv[2 * j + 1] = r.y;
                    }
                }
#pragma unroll
                for (int j = 0; j < TT / 2; ++j) {
                    const float2 u = __fmul2_rn(make_float2(dlv[2 * j], dlv[2 * j + 1]),
                                                make_float2(smem_val(xs + 2 * j * DPB), smem_val(xs + (2 * j + 1) * DPB)));
                    uv[2 * j] = u.x;
                    uv[2 * j + 1] = u.y;
                }
                if constexpr (!RO) {
                    // Stage sum of dl by pairwise halving (rows past the chunk
                    // end do not count), then one compensated add.
                    float part[TT];
#pragma unroll
                    for (int tt = 0; tt < TT; ++tt)
                        part[tt] = tt < tc ? dlv[tt] : 0.0f;
#pragma unroll
                    for (int w = TT / 2; w > 0; w /= 2) {
#pragma unroll
                        for (int tt = 0; tt < w; ++tt)
                            part[tt] += part[tt + w];
                    }
                    const float yk = part[0] - s_err;
                    const float tk = s_sum + yk;
                    s_err = (tk - s_sum) - yk;
                    s_sum = tk;
                }
                if (lane == 0 && rel_stage >= 0 && rel_stage + STAGES < nst && mbar_pending(rel_state) == 1) {
                    const uint32_t rf = ring + rel_stage + STAGES;
                    if (mbar_test_state(&empty[rf % STAGES], rel_state)) {   // acquire the other warps' reads
                        fence_proxy_async_smem();
                        issue(rf, rel_stage + STAGES);
                    }
                }
                rel_stage = -1;

                auto step = [&](int tt) {
                    float Bv[NS];
                    SmemStateLoad<float, NS, VEC>::run(Bs + tt * Nrow, valid, Bv);
                    const float2 dl2 = make_float2(dlv[tt], dlv[tt]);
                    const float2 u2 = make_float2(uv[tt], uv[tt]);
                    const float xt = ZOH ? smem_val(xs + tt * DPB) : 0.0f;
                    auto in_term = [&](int j, float2 e, float2 decay) {
                        if constexpr (ZOH)
                            return zoh_pair(dl2, e, decay, Ainv[j],
                                            __fmul2_rn(make_float2(xt, xt), make_float2(Bv[2 * j], Bv[2 * j + 1])));
                        else
                            return __fmul2_rn(u2, make_float2(Bv[2 * j], Bv[2 * j + 1]));
                    };
                    if constexpr (RO) {
                        float Cv[NS];
                        SmemStateLoad<float, NS, VEC>::run(Cs + tt * Nrow, valid, Cv);
                        float2 acc[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
#pragma unroll
                        for (int j = 0; j < NP; ++j) {
                            const float2 e = __fmul2_rn(dl2, A2[j]);
                            const float2 decay = make_float2(ex2(e.x), ex2(e.y));
                            h[j] = __ffma2_rn(decay, h[j], in_term(j, e, decay));
                            acc[j & 1] = __ffma2_rn(h[j], make_float2(Cv[2 * j], Cv[2 * j + 1]), acc[j & 1]);
                        }
                        const float2 s2 = __fadd2_rn(acc[0], acc[1]);
                        float yv = s2.x + s2.y;
#pragma unroll
                        for (int o = NSPLIT / 2; o > 0; o >>= 1)
                            yv += __shfl_xor_sync(0xffffffffu, yv, o);
                        if constexpr (GATE)
                            yv = block_out(yv, dsk, smem_val(xs + tt * DPB), has_z,
                                           has_z ? smem_val(zs + tt * DPB) : 0.0f);
                        if (active && q == 0)
                            Io<T>::store(yp + tt * D, yv);
                    } else {
#pragma unroll
                        for (int j = 0; j < NP; ++j) {
                            const float2 e = __fmul2_rn(dl2, A2[j]);
                            const float2 decay = make_float2(ex2(e.x), ex2(e.y));
                            h[j] = __ffma2_rn(decay, h[j], in_term(j, e, decay));
                        }
                    }
                };
                if (tc == TT) {
#pragma unroll
                    for (int tt = 0; tt < TT; ++tt)
                        step(tt);
                } else {
                    // The chunk's last, partial stage (at most one per item):
                    // a compact loop, so that the unrolled body above is the
                    // only large copy of the step code in the instruction cache.
#pragma unroll 1
                    for (int tt = 0; tt < tc; ++tt) {
                        float dl = smem_val(ds + tt * DPB);
                        if (SOFTPLUS)
                            dl = softplus(dl);
                        const float2 dl2 = make_float2(dl, dl);
                        const float xt = smem_val(xs + tt * DPB);
                        const float u = dl * xt;
                        const float2 u2 = make_float2(u, u);
                        float Bv[NS], Cv[NS];
                        SmemStateLoad<float, NS, VEC>::run(Bs + tt * Nrow, valid, Bv);
                        if constexpr (RO)
                            SmemStateLoad<float, NS, VEC>::run(Cs + tt * Nrow, valid, Cv);
                        float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
                        for (int j = 0; j < NP; ++j) {
                            const float2 e = __fmul2_rn(dl2, A2[j]);
                            const float2 decay = make_float2(ex2(e.x), ex2(e.y));
                            float2 inp;
                            if constexpr (ZOH)
                                inp = zoh_pair(dl2, e, decay, Ainv[j],
                                               __fmul2_rn(make_float2(xt, xt), make_float2(Bv[2 * j], Bv[2 * j + 1])));
                            else
                                inp = __fmul2_rn(u2, make_float2(Bv[2 * j], Bv[2 * j + 1]));
                            h[j] = __ffma2_rn(decay, h[j], inp);
                            if constexpr (RO)
                                acc = __ffma2_rn(h[j], make_float2(Cv[2 * j], Cv[2 * j + 1]), acc);
                        }
                        if constexpr (RO) {
                            float yv = acc.x + acc.y;
#pragma unroll
                            for (int o = NSPLIT / 2; o > 0; o >>= 1)
                                yv += __shfl_xor_sync(0xffffffffu, yv, o);
                            if constexpr (GATE)
                                yv = block_out(yv, dsk, smem_val(xs + tt * DPB), has_z,
                                               has_z ? smem_val(zs + tt * DPB) : 0.0f);
                            if (active && q == 0)
                                Io<T>::store(yp + tt * D, yv);
                        }
                    }
                }
                yp += (int64_t)TT * D;
                // This warp is done with the buffer.
                __syncwarp();
                if (lane == 0) {
                    rel_state = mbar_arrive_state(&empty[s]);
                    rel_stage = i;
                }
            }
        };
        if (readout)
            run_stages(std::true_type{});
        else
            run_stages(std::false_type{});
        ring += (uint32_t)nst;

        if (!__syncthreads_and(ok)) {   // same answer in every thread
            if (threadIdx.x == 0)
                *s_abort = 1;
            break;
        }

        if (active) {
            if (readout) {
                if (k == a.K - 1 && a.hT) {
                    float *dst = a.hT + (b * D + d) * N + n0;
#pragma unroll
                    for (int j = 0; j < NP; ++j) {
                        if (2 * j < valid) dst[2 * j] = h[j].x;
                        if (2 * j + 1 < valid) dst[2 * j + 1] = h[j].y;
                    }
                }
            } else {
                const int64_t off = ((int64_t)k * a.Bsz * D + b * D + d) * N + n0;
#pragma unroll
                for (int j = 0; j < NP; ++j) {
                    if (2 * j < valid) fa.aggH[off + 2 * j] = h[j].x;
                    if (2 * j + 1 < valid) fa.aggH[off + 2 * j + 1] = h[j].y;
                }
                if (q == 0)
                    fa.aggS[(int64_t)k * a.Bsz * D + b * D + d] = s_sum;
            }
        }
        if (!readout) {
            __syncthreads();   // every thread's pair is written
            if (threadIdx.x == 0) {
                __threadfence();
                if (fa.publish)
                    st_release_u32(fa.ctrl + 1 + idx, 1u);
            }
        }
    }

    // A tile or an aggregate that never arrived: let this CTA's copies in
    // flight land (bounded) before its shared memory goes away.
    if (*s_abort && threadIdx.x == 0) {
        record_fault(fa.fault, kFaultTmaTimeout);
        for (int s = 0; s < STAGES; ++s)
            if (issued[s] > 0)
                mbar_wait(&full[s], (issued[s] - 1) & 1u);
    }
}

inline size_t fused_smem_bytes(size_t es, int TT, int DPB, int64_t Nrow, int stages, bool gate)
{
    const size_t stage = ((gate ? 3 : 2) * (size_t)TT * DPB + 2 * (size_t)TT * (size_t)Nrow) * es;
    const size_t conv = es == 2 ? 2 * (size_t)TT * (size_t)Nrow * 4 : 0;
    return (size_t)stages * (stage + conv) + (size_t)stages * (8 + 8 + 8 + 4) + 16;
}

} // namespace selscan
