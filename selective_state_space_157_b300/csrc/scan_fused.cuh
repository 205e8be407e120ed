// scan_fused.cuh -- the whole forward scan in one persistent kernel.
//
// Work items. The sequence is cut into K chunks and the channels into tiles
// of DPB = THREADS / NSPLIT; G = Bsz * tiles groups. Items are numbered
//     0 .. K*G - 1                 local items      (chunk k,      group g), k-major
//     K*G .. K*G + (K-1)*G - 1     correction items (chunk k >= 1, group g), k-major
// and CTAs take them in that order from an atomic ticket counter.
//
// A local item scans its chunk from a zero state (chunk 0 from h0) and
// writes that scan's read-out to y. It also publishes the chunk's end state
// and sum of dl: the pair (decay[n] = exp(A[d,n] * sum dl), end[n]) of the
// associative composition (a1,b1) o (a2,b2) = (a2 a1, a2 b1 + b2) of the
// parallel scan (booiljung.github.io "3.1 LTI systems ...", section 3.1.5.2).
// The last local item of a group to finish composes the group's pairs in
// chunk order into the true state entering every chunk (chunk 0's end state
// already is one), writes hT, and raises the group's ready flag.
//
// A correction item adds to y what its local item left out: the
// contribution of the state carried into the chunk. With no input that
// state evolves as c_t = exp(dl_t A) c_{t-1} from the carry, and
// y_t += sum_n C_t[n] c_t[n] (the recurrence's linearity in h). With a
// softplus step (dl >= 0) and A <= 0 every |c_t[n]| only shrinks, so once
// it is below fp32 resolution (trunc_tau) for all states of a group of
// four the group is dropped, and the item ends when no group is left:
// the carry's influence fades within a few hundred steps on the
// distributions of the Mamba layers, so the second pass covers a fraction
// of the sequence instead of all of it. States with A > 0 (or any state
// without softplus) are never dropped.
//
// Progress. A correction item waits only on local items of its group,
// whose tickets are all smaller than its own: they were taken by CTAs
// already running, which never wait. So every wait ends, whatever the
// number of resident CTAs. Waits are bounded anyway (tma.cuh).
//
// Inputs arrive as 3-D TMA boxes of TT timesteps (x, delta: TT x DPB; B, C:
// TT x N) into a ring of shared-memory buffers, with "full" mbarriers (TMA
// completion, with the expected byte count). In local items, "empty"
// mbarriers (one arrival per warp when it is done with a buffer) free a
// buffer: the warp whose arrival completes an empty barrier refills that
// buffer with the stage STAGES ahead; it learns that from the arrival's
// result one stage later, so no warp ever waits for another. Correction
// items take delta, C (and z) only, and agree at every stage, with one CTA
// barrier, whether any state is left and the next buffer should be loaded.
// Boxes that run past D or L are zero-filled by the TMA unit; those lanes
// and rows are never stored.
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
    float *aggS;          // (K, Bsz, D): sum of dl over chunk k
    float *aggH;          // (K, Bsz, D, N): end state of chunk k's local scan; once the group's
                          // pairs are composed, slot k holds the state entering chunk k + 1
    unsigned *ctrl;       // [0]: ticket counter; [1 + g]: local items of group g done;
                          // [1 + G + g]: group g's carries ready (all zeroed per call)
    unsigned *fault;      // fault word of the launching stream
    uint64_t wait_ns;     // limit of a correction item's wait for its group's carries
    float trunc_tau;      // correction states below this magnitude are dropped (0: never)
    void *yres;           // bf16 output, chunks >= 1: (Bsz, L, D) bf16 rounding residual of the local
                          // scan's y, so that the corrected y is rounded once in effect (else null)
    int publish;          // 0 only for the timeout test: carries are never announced
    int spread;           // every local item is resident at once: they compose the carries in slices
    int nslices;          // slices of THREADS (chain, state) series per group
    int stages;
    int groups;           // G
    int items_local;      // K * G
    int items_total;      // items_local + (K - 1) * G
};

constexpr unsigned kFaultFlagTimeout = 2;   // a group's chunk carries never appeared
constexpr int kFoldBatch = 4;               // chunk pairs in flight per composition round
// Correction states below this magnitude are dropped: their contribution to
// any later y is below 2^-36 |C|, far under fp32 resolution.
constexpr float kTruncTau = 1.4551915228366852e-11f;   // 2^-36

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

// Four states of a B or C row from the stage tile, from state 4 * gi of
// this thread's slice (zeros past `valid` on the scalar path).
template <bool VEC>
__device__ __forceinline__ void smem_quad(const float *row, int gi, int valid, float (&v)[4])
{
    if constexpr (VEC) {
        const float4 w = *reinterpret_cast<const float4 *>(row + 4 * gi);
        v[0] = w.x; v[1] = w.y; v[2] = w.z; v[3] = w.w;
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            v[i] = 4 * gi + i < valid ? row[4 * gi + i] : 0.0f;
    }
}

// Warp 0 waits until *f >= target (acquire), bounded by wait_ns; on timeout
// it records the fault and raises the CTA's abort flag. Warp-uniform: every
// lane leaves together.
__device__ __forceinline__ void wait_count(const unsigned *f, unsigned target, uint64_t wait_ns, unsigned *fault,
                                           volatile int *s_abort, int lane)
{
    const uint64_t tstart = global_ns();
    bool done = ld_acquire_u32(f) >= target;
    while (!__any_sync(0xffffffffu, done)) {
        __nanosleep(256);
        done = ld_acquire_u32(f) >= target;
        if (__any_sync(0xffffffffu, global_ns() - tstart > wait_ns)) {
            if (lane == 0) {
                record_fault(fault, kFaultFlagTimeout);
                *s_abort = 1;
            }
            break;
        }
    }
}

// Stores NS states from registers (float4 stores on the vector path, which
// write each chain's states in four instructions instead of sixteen).
template <int NS, bool VEC>
__device__ __forceinline__ void store_state(float *p, int valid, const float2 (&v)[NS / 2])
{
    if (VEC) {
#pragma unroll
        for (int j = 0; j < NS / 2; j += 2)
            reinterpret_cast<float4 *>(p)[j / 2] = make_float4(v[j].x, v[j].y, v[j + 1].x, v[j + 1].y);
    } else {
#pragma unroll
        for (int j = 0; j < NS / 2; ++j) {
            if (2 * j < valid) p[2 * j] = v[j].x;
            if (2 * j + 1 < valid) p[2 * j + 1] = v[j].y;
        }
    }
}

// ZOH: the zero-order-hold input term (zoh_pair) in place of dl * B * x.
// GATE: the read-out also applies the block's skip and gate (block_out),
// with z staged beside x in the ring.
// CHUNKED: the sequence is cut into chunks (local and correction items, a
// ticket counter); otherwise one pass, CTA x scanning channel group x.
// THREADS: 128 (up to three CTAs per SM), 256 or 384 (one CTA per SM). SMs
// give their oldest CTA priority, so several CTAs with equal items end far
// apart (on a B300 the youngest of three took 1.6x as long as the oldest);
// the chunked form therefore runs one CTA of twelve warps per SM, and a
// one-pass plan with two threads per chain one CTA of eight warps, whose ring
// keeps every warp within a few stages of the others.
template <typename T, int NS, int NSPLIT, bool VEC, int TT, bool SOFTPLUS, bool GATE, bool ZOH, bool CHUNKED,
          int THREADS = kScanThreads>
// Three CTAs per SM fit the shared-memory ring; the register cap this implies
// (168) is above what the kernel needs, and measured faster than 128.
__global__ void __launch_bounds__(THREADS, THREADS <= 128 ? 3 : 1)
scan_fused_kernel(const __grid_constant__ FusedArgs fa)
{
    static_assert(NS % 4 == 0, "states are processed in pairs of pairs");
    static_assert(TT % 2 == 0, "timesteps are processed in pairs");
    // Launched as a programmatic dependent of the kernel before it on the
    // stream: the CTAs may be resident early, and touch nothing before that
    // kernel has completed; the next kernel may be scheduled once every CTA
    // of this one has started.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    constexpr int DPB = THREADS / NSPLIT;
    // x, delta and z tiles arrive as NB boxes of W channels each (a TMA box
    // spans at most 256 elements), stored [NB][TT][W].
    constexpr int NB = DPB > 256 ? 2 : 1;
    constexpr int W = DPB / NB;
    static_assert(W * NB == DPB && W <= 256, "channel tile splits into equal boxes");
    constexpr int NP = NS / 2;
    constexpr int NG = NS / 4;   // groups of four states (one 16-byte row load each)
    constexpr int kWarps = THREADS / 32;
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
    // Bytes a stage brings: x, delta, B and C (and z) for a local item;
    // delta and C (and z) for a correction item.
    const int local_bytes = 2 * xbytes + 2 * nbytes + (has_z ? xbytes : 0);
    const int corr_bytes = xbytes + nbytes + (has_z ? xbytes : 0);
    constexpr bool kBf16 = sizeof(T) == 2;
    const int cfloats = kBf16 ? 2 * TT * (int)Nrow : 0;   // fp32 copy of a stage's B and C rows
    float *conv_buf = reinterpret_cast<float *>(smem + STAGES * sbytes);
    // With NSPLIT threads per chain, each stage's (dl, dl * x) per channel is
    // computed once, cooperatively, into this buffer (one per ring slot).
    constexpr int kDluFloats = NSPLIT > 1 ? 2 * TT * DPB : 0;
    float2 *dlu = reinterpret_cast<float2 *>(smem + STAGES * (sbytes + cfloats * 4));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * (sbytes + cfloats * 4 + kDluFloats * 4));
    uint64_t *empty = full + STAGES;
    uint64_t *conv = empty + STAGES;   // bf16: every warp converted its share of the stage
    unsigned *issued = reinterpret_cast<unsigned *>(conv + STAGES);
    volatile int *s_item = reinterpret_cast<volatile int *>(issued + STAGES);
    volatile int *s_abort = s_item + 1;
    volatile int *s_last = s_item + 2;

    const int grp = threadIdx.x / NSPLIT;
    const int q = threadIdx.x % NSPLIT;
    const int xcol = (grp / W) * (TT * W) + grp % W;   // this channel's column in an [NB][TT][W] tile
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
    const int64_t bd_all = (int64_t)a.Bsz * D;
    const int64_t slot = bd_all * N;

    for (int round = 0;; ++round) {
        // With a ticket counter CTAs stay resident and take items in order;
        // without one (a single chunk: no dependences) CTA x runs item x.
        if (threadIdx.x == 0)
            *s_item = CHUNKED ? (int)atomicAdd(&fa.ctrl[0], 1u) : (round == 0 ? (int)blockIdx.x : fa.items_total);
        __syncthreads();
        const int item = *s_item;
        if (item >= fa.items_total || *s_abort)
            break;
        const bool local = !CHUNKED || item < fa.items_local;
        const int idx = local ? item : item - fa.items_local;
        const int kq = idx / fa.groups;
        const int g = idx - kq * fa.groups;
        const int k = local ? kq : kq + 1;
        const int64_t b = g / a.dtiles;
        const int d0 = (g % a.dtiles) * DPB;
        const int64_t d_raw = (int64_t)d0 + grp;
        const bool active = d_raw < D;
        const int64_t d = active ? d_raw : D - 1;
        const int64_t t0 = (int64_t)k * a.chunk;
        const int64_t nsteps = min(L, t0 + a.chunk) - t0;
        const int nst = (int)((nsteps + TT - 1) / TT);
        const int64_t off = (b * D + d) * N + n0;   // this thread's states in a (Bsz, D, N) slot

        auto buf = [&](uint32_t r) { return smem + (r % STAGES) * sbytes; };
        auto issue = [&](uint32_t r, int i) {   // stage i of this item into ring slot r
            const int s = (int)(r % STAGES);
            unsigned char *p = buf(r);
            const int t = (int)(t0 + (int64_t)i * TT);
            issued[s] += 1;
            mbar_arrive_expect_tx(&full[s], (uint32_t)(local ? local_bytes : corr_bytes));
            constexpr int sub = TT * W * (int)sizeof(T);   // bytes of one box
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                if (local)
                    tma_load_3d(p + nb * sub, &fa.mx, &full[s], d0 + nb * W, t, (int)b);
                tma_load_3d(p + xbytes + nb * sub, &fa.md, &full[s], d0 + nb * W, t, (int)b);
                if (has_z)
                    tma_load_3d(p + 2 * xbytes + 2 * nbytes + nb * sub, &fa.mz, &full[s], d0 + nb * W, t, (int)b);
            }
            if (local)
                tma_load_3d(p + 2 * xbytes, &fa.mB, &full[s], 0, t, (int)b);
            tma_load_3d(p + 2 * xbytes + nbytes, &fa.mC, &full[s], 0, t, (int)b);
        };

        // Every warp finished the previous item: its buffers may be refilled.
        if (threadIdx.x == 0) {
            fence_proxy_async_smem();
            for (int f = 0; f < STAGES && f < nst; ++f)
                issue(ring + f, f);
        }

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

        T *yp = static_cast<T *>(a.y) + (b * L + t0) * D + d;
        bool ok = true;

        // The B and C rows of a stage in fp32: straight from the tile, or
        // (bf16 input) from this stage's fp32 copy, which the four warps
        // convert together -- every thread needs every row, so converting
        // once per CTA instead of once per thread saves most of the
        // unpacking work. Rows [first, first + rows) of the B|C pair.
        // With several threads per chain (with_dlu), the stage's dl (after
        // softplus) and dl * x are computed once per channel into the slot's
        // dlu buffer by the same cooperative pass. A CTA-wide mbarrier closes
        // the pass (bounded wait), so the warps need no CTA barrier.
        constexpr bool kCoop = kBf16 || NSPLIT > 1;
        auto stage_rows = [&](const unsigned char *p, int s, uint32_t r, int first, int rows, const float **Bs,
                              const float **Cs, bool with_dlu) -> bool {
            if constexpr (kBf16) {
                float *cb = conv_buf + s * cfloats;
                const __nv_bfloat16 *src = reinterpret_cast<const __nv_bfloat16 *>(p + 2 * xbytes);
                const int lo = first * TT * (int)Nrow, hi = (first + rows) * TT * (int)Nrow;
                for (int e = lo + threadIdx.x; e < hi; e += THREADS)
                    cb[e] = __bfloat162float(src[e]);
            }
            if constexpr (NSPLIT > 1) {
                if (with_dlu) {
                    float2 *db = dlu + s * TT * DPB;
                    const T *xt = reinterpret_cast<const T *>(p);
                    const T *dt = reinterpret_cast<const T *>(p + xbytes);
                    static_assert((TT * DPB) % THREADS == 0, "whole rounds of the cooperative pass");
#pragma unroll
                    for (int e0 = 0; e0 < TT * DPB; e0 += THREADS) {
                        const int e = e0 + threadIdx.x;
                        const int tt = e / DPB, c = e % DPB;
                        const int col = (c / W) * (TT * W) + tt * W + c % W;
                        float dl = smem_val(dt + col);
                        if (SOFTPLUS)
                            dl = softplus(dl);
                        db[e] = make_float2(dl, dl * smem_val(xt + col));
                    }
                }
            }
            if constexpr (kCoop) {
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&conv[s]);
                if (!__all_sync(0xffffffffu, mbar_wait(&conv[s], (r / STAGES) & 1u)))
                    return false;
            }
            if constexpr (kBf16) {
                float *cb = conv_buf + s * cfloats;
                *Bs = cb + n0;
                *Cs = cb + TT * Nrow + n0;
            } else {
                *Bs = reinterpret_cast<const float *>(p + 2 * xbytes) + n0;
                *Cs = reinterpret_cast<const float *>(p + 2 * xbytes + nbytes) + n0;
            }
            return true;
        };

        if (local) {
            // ---------------- local item: the chunk's scan from h0 (chunk 0) or zero
            const float dsk = (GATE && a.Dskip) ? __ldg(a.Dskip + d) : 0.0f;
            float2 h[NP];
            if (k == 0 && a.h0) {
                load_state_cg<NS, false>(a.h0 + off, valid, h);
            } else {
#pragma unroll
                for (int j = 0; j < NP; ++j)
                    h[j] = make_float2(0.0f, 0.0f);
            }
            float s_sum = 0.0f, s_err = 0.0f;
            // bf16 output that a correction item will add to: keep what
            // rounding y dropped.
            T *rp = (kBf16 && fa.yres && k > 0) ? static_cast<T *>(fa.yres) + (b * L + t0) * D + d : nullptr;
            // The stage loop, compiled twice: with one chunk (TRACK false)
            // nothing else needs the chunk's sum of dl or rounding residuals,
            // and the loop keeps only what the scan itself needs live.
            auto run_local = [&](auto track) {
            constexpr bool TRACK = decltype(track)::value;
            auto put = [&](int64_t o, float v) {
                if constexpr (kBf16) {
                    const __nv_bfloat16 r = __float2bfloat16_rn(v);
                    yp[o] = r;
                    if (TRACK && rp)
                        rp[o] = __float2bfloat16_rn(v - __bfloat162float(r));
                } else {
                    yp[o] = v;
                }
            };
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
                const T *xs = reinterpret_cast<const T *>(p) + xcol;
                const T *ds = reinterpret_cast<const T *>(p + xbytes) + xcol;
                [[maybe_unused]] const T *zs = reinterpret_cast<const T *>(p + 2 * xbytes + 2 * nbytes) + xcol;
                const float *Bs;
                const float *Cs;
                if (!stage_rows(p, s, r, 0, 2, &Bs, &Cs, true)) {
                    ok = false;
                    break;
                }
                const int64_t rem = nsteps - (int64_t)i * TT;
                const int tc = rem < TT ? (int)rem : TT;

                // Phase 1, breadth first: TT independent softplus evaluations
                // advance together, so their dependent FMAs interleave.
                float dlv[TT], uv[TT];
                if constexpr (NSPLIT > 1) {
                    // Computed once per channel by the cooperative pass.
                    const float2 *db = dlu + s * TT * DPB + grp;
#pragma unroll
                    for (int tt = 0; tt < TT; ++tt) {
                        const float2 v = db[tt * DPB];
                        dlv[tt] = v.x;
                        uv[tt] = v.y;
                    }
                } else {
#pragma unroll
                for (int tt = 0; tt < TT; ++tt)
                    dlv[tt] = smem_val(ds + tt * W);
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
                        const float2 rr = __ffma2_rn(pv[j], ev[j], make_float2(fmaxf(dlv[2 * j], 0.0f), fmaxf(dlv[2 * j + 1], 0.0f)));
                        dlv[2 * j] = rr.x;
                        dlv[2 * j + 1] = rr.y;
                    }
                }
#pragma unroll
                for (int j = 0; j < TT / 2; ++j) {
                    const float2 u = __fmul2_rn(make_float2(dlv[2 * j], dlv[2 * j + 1]),
                                                make_float2(smem_val(xs + 2 * j * W), smem_val(xs + (2 * j + 1) * W)));
                    uv[2 * j] = u.x;
                    uv[2 * j + 1] = u.y;
                }
                }
                if constexpr (TRACK) {
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
                    [[maybe_unused]] const float xt = ZOH ? smem_val(xs + tt * W) : 0.0f;
                    float Cv[NS];
                    SmemStateLoad<float, NS, VEC>::run(Cs + tt * Nrow, valid, Cv);
                    float2 acc[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
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
                        acc[j & 1] = __ffma2_rn(h[j], make_float2(Cv[2 * j], Cv[2 * j + 1]), acc[j & 1]);
                    }
                    const float2 s2 = __fadd2_rn(acc[0], acc[1]);
                    float yv = s2.x + s2.y;
#pragma unroll
                    for (int o = NSPLIT / 2; o > 0; o >>= 1)
                        yv += __shfl_xor_sync(0xffffffffu, yv, o);
                    if constexpr (GATE)
                        yv = block_out(yv, dsk, smem_val(xs + tt * W), has_z,
                                       has_z ? smem_val(zs + tt * W) : 0.0f);
                    if (active && q == 0)
                        put((int64_t)tt * D, yv);
                };
                if (tc == TT) {
#pragma unroll
                    for (int tt = 0; tt < TT; ++tt)
                        step(tt);
                } else {
                    // The chunk's last, partial stage (at most one per item): a
                    // compact loop, so that the unrolled body above is the only
                    // large copy of the step code in the instruction cache.
#pragma unroll 1
                    for (int tt = 0; tt < tc; ++tt) {
                        float dl = smem_val(ds + tt * W);
                        if (SOFTPLUS)
                            dl = softplus(dl);
                        const float2 dl2 = make_float2(dl, dl);
                        const float xt = smem_val(xs + tt * W);
                        const float u = dl * xt;
                        const float2 u2 = make_float2(u, u);
                        float Bv[NS], Cv[NS];
                        SmemStateLoad<float, NS, VEC>::run(Bs + tt * Nrow, valid, Bv);
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
                            acc = __ffma2_rn(h[j], make_float2(Cv[2 * j], Cv[2 * j + 1]), acc);
                        }
                        float yv = acc.x + acc.y;
#pragma unroll
                        for (int o = NSPLIT / 2; o > 0; o >>= 1)
                            yv += __shfl_xor_sync(0xffffffffu, yv, o);
                        if constexpr (GATE)
                            yv = block_out(yv, dsk, xt, has_z, has_z ? smem_val(zs + tt * W) : 0.0f);
                        if (active && q == 0)
                            put((int64_t)tt * D, yv);
                    }
                }
                yp += (int64_t)TT * D;
                if (TRACK && rp)
                    rp += (int64_t)TT * D;
                // This warp is done with the buffer.
                __syncwarp();
                if (lane == 0) {
                    rel_state = mbar_arrive_state(&empty[s]);
                    rel_stage = i;
                }
            }
            };
            if constexpr (CHUNKED)
                run_local(std::true_type{});
            else
                run_local(std::false_type{});
            ring += (uint32_t)nst;
            if (!__syncthreads_and(ok)) {   // same answer in every thread
                if (threadIdx.x == 0)
                    *s_abort = 1;
                break;
            }

            if constexpr (!CHUNKED) {
                if (active && a.hT) {
                    float *dst = a.hT + off;
#pragma unroll
                    for (int j = 0; j < NP; ++j) {
                        if (2 * j < valid) dst[2 * j] = h[j].x;
                        if (2 * j + 1 < valid) dst[2 * j + 1] = h[j].y;
                    }
                }
                continue;
            } else {
            // Publish the chunk's pair; the group's last local item composes.
            if (active) {
                store_state<NS, VEC>(fa.aggH + (int64_t)k * slot + off, valid, h);
                if (q == 0)
                    fa.aggS[(int64_t)k * bd_all + b * D + d] = s_sum;
            }
            __threadfence();   // this thread's y and pair, visible to the GPU
            __syncthreads();
            if (threadIdx.x == 0) {
                *s_last = atomicAdd(&fa.ctrl[1 + g], 1u) == (unsigned)(a.K - 1);
                __threadfence();
            }
            __syncthreads();
            if (fa.spread) {
                // Every local item of the group is resident: the first
                // nslices of them compose one slice each of the group's
                // (chain, state) series, one series per thread, once all the
                // group's pairs are published. c_1 = end_0; c_{j+1} =
                // exp(A * sum dl_j) c_j + end_j, stored in slot j (the state
                // entering chunk j + 1); the last one is hT. A thread's loads
                // of 32 pairs are all in flight at once.
                if (k >= fa.nslices)
                    continue;
                if (threadIdx.x < 32)
                    wait_count(fa.ctrl + 1 + g, (unsigned)a.K, fa.wait_ns, fa.fault, s_abort, lane);
                __syncthreads();
                if (*s_abort)
                    break;
                unsigned done_slices = 0;
                for (int sl = k; sl < fa.nslices; sl += a.K) {
                    ++done_slices;
                    const int64_t i = (int64_t)sl * THREADS + threadIdx.x;
                    const int64_t dc = d0 + i / N;
                    const int64_t n = i % N;
                    if (i / N >= DPB || dc >= D)
                        continue;
                    const float An = __ldg(a.A + dc * N + n) * kLog2e;
                    const int64_t o = (b * D + dc) * N + n;
                    const float *Sq = fa.aggS + b * D + dc;
                    float cs = __ldcg(fa.aggH + o);
                    for (int j0 = 1; j0 < a.K; j0 += 32) {
                        float Sv[32], Ev[32];
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj) {
                            const int64_t j = j0 + jj < a.K ? j0 + jj : a.K - 1;
                            Sv[jj] = __ldcg(Sq + j * bd_all);
                            Ev[jj] = __ldcg(fa.aggH + j * slot + o);
                        }
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj) {
                            const int j = j0 + jj;
                            if (j < a.K) {
                                cs = fmaf(ex2(An * Sv[jj]), cs, Ev[jj]);
                                if (j < a.K - 1)
                                    fa.aggH[(int64_t)j * slot + o] = cs;
                                else if (a.hT)
                                    a.hT[o] = cs;
                            }
                        }
                    }
                }
                __threadfence();
                __syncthreads();   // this item's slices are written
                if (threadIdx.x == 0 && fa.publish)
                    atomicAdd(fa.ctrl + 1 + fa.groups + g, done_slices);
                continue;
            }
            if (!*s_last)
                continue;
            // Compose the group's pairs in chunk order: c_1 = end_0 (chunk 0
            // started from h0); c_{j+1} = exp(A * sum dl_j) c_j + end_j. Slot j
            // receives c_{j+1}, the state entering chunk j + 1; the last one is
            // hT. Loads run kFoldBatch pairs ahead of their use.
            __threadfence();
            // The pairs were written by other CTAs up to a whole item ago and
            // may have left L2: bring them all back at once, so that the
            // batches below wait for L2, not for DRAM, round trip by round trip.
            const float *Sp = fa.aggS + b * D + d;
            for (int j = 1; j < a.K; ++j) {
                prefetch_l2(fa.aggH + (int64_t)j * slot + off);
                if (q == 0)
                    prefetch_l2(Sp + (int64_t)j * bd_all);
            }
            float2 c[NP];
            load_state_cg<NS, VEC>(fa.aggH + off, valid, c);
            for (int j0 = 1; j0 < a.K; j0 += kFoldBatch) {
                float S[kFoldBatch];
                float2 E[kFoldBatch][NP];
#pragma unroll
                for (int jj = 0; jj < kFoldBatch; ++jj) {
                    const int64_t j = j0 + jj < a.K ? j0 + jj : a.K - 1;   // past the end: a repeat, unused
                    S[jj] = __ldcg(Sp + j * bd_all);
                    load_state_cg<NS, VEC>(fa.aggH + j * slot + off, valid, E[jj]);
                }
#pragma unroll
                for (int jj = 0; jj < kFoldBatch; ++jj) {
                    const int j = j0 + jj;
                    if (j < a.K) {
                        const float2 s2 = make_float2(S[jj], S[jj]);
#pragma unroll
                        for (int i = 0; i < NP; ++i) {
                            const float2 e = __fmul2_rn(s2, A2[i]);
                            c[i] = __ffma2_rn(make_float2(ex2(e.x), ex2(e.y)), c[i], E[jj][i]);
                        }
                        if (active && j < a.K - 1)
                            store_state<NS, VEC>(fa.aggH + (int64_t)j * slot + off, valid, c);
                        else if (active && a.hT)
                            store_state<NS, false>(a.hT + off, valid, c);
                    }
                }
            }
            __threadfence();
            __syncthreads();   // every carry is written
            if (threadIdx.x == 0 && fa.publish)
                st_release_u32(fa.ctrl + 1 + fa.groups + g, (unsigned)fa.nslices);
            continue;
            }
        }

        // ---------------- correction item: the carry's contribution to chunk k
        if constexpr (CHUNKED) {
        // Warp 0 waits until every slice of the group's carries is composed.
        if (threadIdx.x < 32)
            wait_count(fa.ctrl + 1 + fa.groups + g, (unsigned)fa.nslices, fa.wait_ns, fa.fault, s_abort, lane);
        __syncthreads();
        if (*s_abort)
            break;
        float2 c[NP];
        load_state_cg<NS, VEC>(fa.aggH + (int64_t)(k - 1) * slot + off, valid, c);
        const float tau = fa.trunc_tau;
        // Group gi stays while any lane holds a state in it that is not
        // below tau (NaN included) or can grow (A > 0).
        auto group_live = [&](int gi) -> bool {
            bool live = false;
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int j = 2 * gi + jj;
                live |= !(fabsf(c[j].x) < tau) || A2[j].x > 0.0f;
                live |= !(fabsf(c[j].y) < tau) || A2[j].y > 0.0f;
            }
            return __any_sync(0xffffffffu, live);
        };
        unsigned alive = 0;
#pragma unroll
        for (int gi = 0; gi < NG; ++gi)
            alive |= group_live(gi) ? 1u << gi : 0u;
        const T *yin = static_cast<const T *>(a.y) + (b * L + t0) * D + d;
        const T *rin = (kBf16 && fa.yres) ? static_cast<const T *>(fa.yres) + (b * L + t0) * D + d : nullptr;
        // Outputs of the local scan for the current stage, with the bf16
        // rounding residuals when kept. Each stage's are loaded when the stage
        // before has finished with its own, so the loads run during that
        // stage's barriers, tile wait and softplus.
        float yl[TT], rl[TT];
#pragma unroll
        for (int tt = 0; tt < TT; ++tt) {
            const bool in = active && q == 0 && tt < nsteps;
            yl[tt] = in ? Io<T>::load_cg(yin + tt * D) : 0.0f;
            rl[tt] = (in && rin) ? Io<T>::load_cg(rin + tt * D) : 0.0f;
        }
        int consumed = 0;
        for (int i = 0; i < nst; ++i) {
            const uint32_t r = ring + i;
            const int s = (int)(r % STAGES);
            // A wait that ran out does not leave the loop at once: every warp
            // meets the stage's CTA barriers below, and they end the item.
            ok = ok && __all_sync(0xffffffffu, mbar_wait(&full[s], (r / STAGES) & 1u));
            consumed = i + 1;
            const unsigned char *p = buf(r);
            const T *ds = reinterpret_cast<const T *>(p + xbytes) + xcol;
            const T *zs = reinterpret_cast<const T *>(p + 2 * xbytes + 2 * nbytes) + xcol;
            const float *Bs = nullptr;
            const float *Cs = nullptr;
            ok = ok && stage_rows(p, s, r, 1, 1, &Bs, &Cs, false);
            const int64_t rem = nsteps - (int64_t)i * TT;
            const int tc = rem < TT ? (int)rem : TT;
            if (alive && ok) {
                // Steps of the stage, breadth first: dl for all of them (0 past
                // the chunk end, so that those steps leave the state as it is).
                float dlv[TT];
#pragma unroll
                for (int tt = 0; tt < TT; ++tt) {
                    float v = smem_val(ds + tt * W);
                    if (SOFTPLUS)
                        v = softplus(v);
                    dlv[tt] = tt < tc ? v : 0.0f;
                }
                float2 accs[TT];
#pragma unroll
                for (int tt = 0; tt < TT; ++tt)
                    accs[tt] = make_float2(0.0f, 0.0f);
                // One warp-uniform branch per group and stage; inside, the
                // stage's steps are straight-line code, so the exponentials of
                // later steps overlap the products of earlier ones.
#pragma unroll
                for (int gi = 0; gi < NG; ++gi) {
                    if (alive & (1u << gi)) {
#pragma unroll
                        for (int tt = 0; tt < TT; ++tt) {
                            float Cq[4];
                            smem_quad<VEC>(Cs + tt * Nrow, gi, valid, Cq);
                            const float2 dl2 = make_float2(dlv[tt], dlv[tt]);
#pragma unroll
                            for (int jj = 0; jj < 2; ++jj) {
                                const int j = 2 * gi + jj;
                                const float2 e = __fmul2_rn(dl2, A2[j]);
                                c[j] = __fmul2_rn(make_float2(ex2(e.x), ex2(e.y)), c[j]);
                                accs[tt] = __ffma2_rn(c[j], make_float2(Cq[2 * jj], Cq[2 * jj + 1]), accs[tt]);
                            }
                        }
                    }
                }
#pragma unroll
                for (int tt = 0; tt < TT; ++tt) {
                    if (tt >= tc)
                        break;
                    float yv = accs[tt].x + accs[tt].y;
#pragma unroll
                    for (int o = NSPLIT / 2; o > 0; o >>= 1)
                        yv += __shfl_xor_sync(0xffffffffu, yv, o);
                    if constexpr (GATE) {
                        // y = (scan + Dskip x) silu(z) is linear in the scan.
                        if (has_z)
                            yv *= silu(smem_val(zs + tt * W));
                    }
                    if (active && q == 0)
                        Io<T>::store(yp + tt * D, yl[tt] + (rin ? rl[tt] : 0.0f) + yv);
                }
#pragma unroll
                for (int gi = 0; gi < NG; ++gi)
                    if ((alive & (1u << gi)) && !group_live(gi))
                        alive &= ~(1u << gi);
                // The next stage's outputs of the local scan.
                const int64_t nrem = nsteps - (int64_t)(i + 1) * TT;
#pragma unroll
                for (int tt = 0; tt < TT; ++tt) {
                    const bool in = alive && active && q == 0 && tt < nrem;
                    yl[tt] = in ? Io<T>::load_cg(yin + (TT + tt) * D) : 0.0f;
                    rl[tt] = (in && rin) ? Io<T>::load_cg(rin + (TT + tt) * D) : 0.0f;
                }
            }
            yp += (int64_t)TT * D;
            yin += (int64_t)TT * D;
            if (rin)
                rin += (int64_t)TT * D;
            // Every warp is done with the buffer; did any wait run out, and
            // is any state left?
            if (__syncthreads_or(!ok))
                break;
            const bool more = __syncthreads_or(alive != 0);
            if (more && threadIdx.x == 0 && i + STAGES < nst) {
                fence_proxy_async_smem();
                issue(ring + i + STAGES, i + STAGES);
            }
            if (!more) {
                // Let the stages already in flight land (each one completes
                // its phase of every barrier, as a consumed stage does).
                const int end = min(nst, i + STAGES);
                for (int i2 = i + 1; i2 < end; ++i2) {
                    const uint32_t r2 = ring + i2;
                    if (!__all_sync(0xffffffffu, mbar_wait(&full[r2 % STAGES], (r2 / STAGES) & 1u)))
                        ok = false;
                    if constexpr (kCoop) {
                        __syncwarp();
                        if (lane == 0)
                            mbar_arrive(&conv[r2 % STAGES]);
                    }
                }
                consumed = end;
                break;
            }
        }
        ring += (uint32_t)consumed;
        if (!__syncthreads_and(ok)) {
            if (threadIdx.x == 0)
                *s_abort = 1;
            break;
        }
        }
    }

    // A tile or a carry that never arrived: let this CTA's copies in flight
    // land (bounded) before its shared memory goes away.
    if (*s_abort && threadIdx.x == 0) {
        record_fault(fa.fault, kFaultTmaTimeout);
        for (int s = 0; s < STAGES; ++s)
            if (issued[s] > 0)
                mbar_wait(&full[s], (issued[s] - 1) & 1u);
    }
}

inline size_t fused_smem_bytes(size_t es, int TT, int DPB, int64_t Nrow, int stages, bool gate, int nsplit)
{
    const size_t stage = ((gate ? 3 : 2) * (size_t)TT * DPB + 2 * (size_t)TT * (size_t)Nrow) * es;
    const size_t conv = es == 2 ? 2 * (size_t)TT * (size_t)Nrow * 4 : 0;
    const size_t dlu = nsplit > 1 ? 2 * (size_t)TT * DPB * 4 : 0;
    return (size_t)stages * (stage + conv + dlu) + (size_t)stages * (8 + 8 + 8 + 4) + 16;
}

} // namespace selscan
