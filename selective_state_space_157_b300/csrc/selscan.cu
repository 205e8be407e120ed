// selscan.cu -- host side of libselscan: argument checks, launch planning,
// the chunk-carry workspace, and the exported C entry points declared in
// include/selscan.h.
#include "selscan.h"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "host_common.h"
#include "launch.h"

namespace selscan {

thread_local char g_err[512];

int fail(int code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char *what)
{
    return fail(SELSCAN_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

long env_long(const char *name, long dflt)
{
    const char *s = getenv(name);
    if (!s || !*s) return dflt;
    char *end = nullptr;
    long v = strtol(s, &end, 10);
    return (end && *end == '\0') ? v : dflt;
}

// ---- per-device state -----------------------------------------------------

namespace {
std::mutex g_mu;
cudaMemPool_t g_pool[kMaxDevices];
int g_sms[kMaxDevices];
} // namespace

int device_info(int *dev, int *sms)
{
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (*dev < 0 || *dev >= kMaxDevices) return fail(SELSCAN_ERR_UNSUPPORTED, "device ordinal %d", *dev);
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_sms[*dev] == 0) {
        int n = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, *dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        g_sms[*dev] = n;
    }
    *sms = g_sms[*dev];
    return SELSCAN_OK;
}

int workspace_pool(int dev, cudaMemPool_t *pool)
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_pool[dev]) {
        cudaMemPoolProps props;
        memset(&props, 0, sizeof props);
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t p;
        cudaError_t e = cudaMemPoolCreate(&p, &props);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemPoolCreate");
        uint64_t keep = UINT64_MAX;   // keep freed blocks for reuse until released
        cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep);
        g_pool[dev] = p;
    }
    *pool = g_pool[dev];
    return SELSCAN_OK;
}

// ---- fault words ----------------------------------------------------------
// Kernels that wait (on a TMA tile or a chunk carry) give up after a time
// limit and record a code in a fault word. Each stream gets its own word, so
// selscan_check_device_error reports a timeout to checks on the stream the
// kernel ran on, and to no other.

constexpr int kFaultSlots = 64;
static __device__ unsigned g_fault_slots[kFaultSlots];

namespace {
struct FaultTable {
    unsigned *base = nullptr;   // device address of g_fault_slots on this device
    cudaStream_t streams[kFaultSlots];
    int used = 0;
};
FaultTable g_faults[kMaxDevices];
std::mutex g_fault_mu;
} // namespace

int fault_word(int dev, cudaStream_t st, unsigned **out)
{
    std::lock_guard<std::mutex> lk(g_fault_mu);
    FaultTable &t = g_faults[dev];
    if (!t.base) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_fault_slots);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the fault words");
        t.base = static_cast<unsigned *>(p);
    }
    int i = 0;
    while (i < t.used && t.streams[i] != st) ++i;
    if (i == t.used) {
        if (t.used < kFaultSlots) t.streams[t.used++] = st;
        else i = kFaultSlots - 1;   // beyond kFaultSlots streams, one shared word
    }
    *out = t.base + i;
    return SELSCAN_OK;
}

namespace {

// ---- fault injection for the failure-detection test -------------------------
// Off unless selscan_test_fault_injection turns it on; nothing in the
// environment can enable it.
std::mutex g_test_mu;
int g_test_withhold = 0;      // chunk carries are never announced
long g_test_wait_ms = 0;      // limit of the waits for them (0: the default)

// ---- forward planning ---------------------------------------------------

// Default buffers in flight per CTA. Two measured fastest on B300 (Bsz=2,
// L=2048, D=1536: 72 us against 79 us with four); no workload measured slower.
constexpr int kStages = 2;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        else
            cudaGetLastError();
    });
    return g_encode;
}

// 3-D map over a row-major (d2, d1, d0) tensor, box (box0, box1, 1).
bool encode_3d(CUtensorMap *m, CUtensorMapDataType dt, size_t es, const void *base, uint64_t d0, uint64_t d1,
               uint64_t d2, uint32_t box0, uint32_t box1)
{
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {d0 * es, d0 * d1 * es};
    cuuint32_t box[3] = {box0, box1, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

struct FwdPlan {
    int ns, nsplit;
    bool vec;
    bool tma;
    int64_t chunk;
    int K;
    int threads;     // CTA size of the fused kernel
    int dtiles;      // channel tiles of threads / nsplit channels
    bool stage_hT;   // hT is h0 and K > 1: the final state goes to the workspace, then to hT
};

// States per thread and threads per chain: the smallest NS in {4, 8, 16}
// covering N / NSPLIT. NSPLIT is 1 up to N = 16 (2 and 4 beyond), unless
// SELSCAN_NSPLIT asks for more threads per chain.
void plan_fwd(int64_t Bsz, int64_t L, int64_t D, int64_t N, size_t es, const void *x, const void *delta,
              const void *B, const void *C, const float *h0, const float *hT, int sms, FwdPlan *p)
{
    int nsplit = N <= 16 ? 1 : (N <= 32 ? 2 : 4);
    long want = env_long("SELSCAN_NSPLIT", 0);
    if ((want == 2 || want == 4) && want > nsplit && N >= 4 * want)
        nsplit = (int)want;
    // (Two threads per chain for one-pass plans with 3 to 6 warps of chains
    // per SM measured slower on B300: Bsz=8 L=2048 D=2048 bf16 took 260 us
    // against 237 with one thread per chain.)
    int64_t per = (N + nsplit - 1) / nsplit;
    int ns = per <= 4 ? 4 : (per <= 8 ? 8 : 16);
    p->ns = ns;
    p->nsplit = nsplit;
    p->vec = (N == (int64_t)ns * nsplit) && ((N * (int64_t)es) % 16 == 0) && aligned(B, 16) &&
             aligned(C, 16);
    const bool bases16 = aligned(x, 16) && aligned(delta, 16) && aligned(B, 16) && aligned(C, 16);
    // TMA needs 16-byte aligned bases and row strides, and 32-bit coordinates.
    p->tma = bases16 && env_long("SELSCAN_NO_TMA", 0) == 0 && (D * (int64_t)es) % 16 == 0 && (N * (int64_t)es) % 16 == 0 &&
             L <= 0x7fffffffLL && D <= 0x7fffffffLL && Bsz <= 0x7fffffffLL;

    // Chunking. One pass whenever the chains alone give three or more warps
    // per SM: on B300 that is the fastest form (Bsz=8, D=2048).
    // Below that, on the TMA path (one persistent kernel), every chunk is
    // scanned once from a zero state by a local item, and chunks 1..K-1 get a
    // correction pass that ends once the carried state has faded. So the
    // sequence is cut into as many chunks as fill the GPU with local items in
    // one wave: K = floor(resident CTAs / channel groups), with one CTA of
    // kFusedChunkedThreads per SM.
    // The plain-load path (aggregate, carry and readout kernels; every chunk
    // but the last is scanned twice) measured best with about 12 warps per
    // SM in flight while chunks stay short, 24 once chunks reach 512 steps.
    auto tiles = [&](int threads) { const int64_t c = threads / nsplit; return (D + c - 1) / c; };
    const int64_t warps1 = Bsz * tiles(kScanThreads) * (kScanThreads / 32);
    const long want_warps = env_long("SELSCAN_TARGET_WARPS", 0);
    auto chunks_for = [&](long warps_per_sm) -> int64_t {
        const int64_t target = (int64_t)warps_per_sm * sms;
        return warps1 >= target ? 1 : (target + warps1 - 1) / warps1;
    };
    int64_t K = 1;
    if (warps1 > 0 && want_warps > 0) {
        K = chunks_for(want_warps);
    } else if (warps1 > 0 && p->tma) {
        if (warps1 < 3 * (int64_t)sms) {
            const int64_t groups = Bsz * tiles(kFusedChunkedThreads);
            const int64_t resident = (int64_t)sms * kFusedChunkedCtasPerSm;
            K = groups >= resident ? 1 : resident / groups;
        }
    } else if (warps1 > 0 && warps1 < 3 * (int64_t)sms) {
        K = chunks_for(12);
        if (K > 1 && L / K >= 512)
            K = chunks_for(24);
    }
    const int64_t min_chunk = 64;
    int64_t maxK = (L + min_chunk - 1) / min_chunk;
    if (K > maxK) K = maxK;
    if (K < 1) K = 1;
    int64_t chunk = L > 0 ? (L + K - 1) / K : 1;
    long force = env_long("SELSCAN_CHUNK", -1);
    if (force == 0) chunk = L > 0 ? L : 1;
    else if (force > 0) chunk = force;
    if (chunk < 1) chunk = 1;
    const int64_t min_for_grid = (L + 65534) / 65535;   // gridDim.y limit
    if (chunk < min_for_grid) chunk = min_for_grid;
    p->chunk = chunk;
    p->K = L > 0 ? (int)((L + chunk - 1) / chunk) : 1;
    // The fused kernel's CTA size (fused_threads); the plain-load kernels run
    // CTAs of kScanThreads.
    p->threads = p->tma ? fused_threads(p->K > 1, nsplit) : kScanThreads;
    p->dtiles = (int)tiles(p->threads);
    // Every chunk's first pass (fused kernel) or readout (plain kernels) may
    // load h0 while the final state is written: in place, that would race.
    p->stage_hT = hT != nullptr && hT == h0 && p->K > 1;
}

// Workspace of a plan, in this order: per chunk and chain the end state
// (N floats, K slots), then the sum of dl (1 float, K slots); the ticket
// counter and two words per channel group (local items done, carries
// ready; the plain-load path uses none of them); then, for in-place resume,
// the staged final state (Bsz * D * N floats).
// With bf16 output on the TMA path, chunks >= 1 also keep the bf16 rounding
// residual of their local y (Bsz * L * D bf16, chunk 0's part unused).
struct WsLayout {
    size_t pairs, flags, res, stage, total;
};

WsLayout fwd_workspace_layout(const FwdPlan &plan, int64_t Bsz, int64_t L, int64_t D, int64_t N, int dtype)
{
    WsLayout w{0, 0, 0, 0, 0};
    if (plan.K > 1) {
        w.pairs = (size_t)plan.K * (size_t)(Bsz * D) * (size_t)(N + 1) * sizeof(float);
        w.flags = (1 + 2 * (size_t)(Bsz * plan.dtiles)) * sizeof(unsigned);
        if (plan.tma && dtype == SELSCAN_BF16) w.res = (size_t)(Bsz * L * D) * 2;
    }
    if (plan.stage_hT) w.stage = (size_t)(Bsz * D * N) * sizeof(float);
    w.total = w.pairs + ((w.flags + 255) & ~(size_t)255) + ((w.res + 15) & ~(size_t)15) + w.stage;
    return w;
}

size_t fwd_workspace_bytes(const FwdPlan &plan, int64_t Bsz, int64_t L, int64_t D, int64_t N, int dtype)
{
    return fwd_workspace_layout(plan, Bsz, L, D, N, dtype).total;
}

// Clears a chunked call's control words, as a programmatic dependent of the
// kernel before it (the previous call, which may still use words at the
// same addresses), so that the fused kernel after it can be one too.
__global__ void __launch_bounds__(256) clear_ctrl_kernel(unsigned *w, int n)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    for (int i = blockIdx.x * 256 + threadIdx.x; i < n; i += gridDim.x * 256)
        w[i] = 0u;
}

cudaError_t launch_dependent(const void *kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st, void **args)
{
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, kernel, args);
}

// TMA path: one persistent kernel (local scans, carry composition and
// corrections together).
// Returns SELSCAN_ERR_UNSUPPORTED when TMA cannot be set up (the caller then
// takes the plain path); nothing has been enqueued in that case.
int launch_fused(const ScanArgs &a, const FwdPlan &plan, int dtype, int sms, float *ws, unsigned *fault,
                 cudaStream_t st)
{
    FusedLaunch fl;
    const bool sp = a.softplus != 0;
    const bool gate = a.Dskip != nullptr || a.z != nullptr;
    if (a.z && !aligned(a.z, 16)) return SELSCAN_ERR_UNSUPPORTED;
    const bool zoh = a.zoh != 0;
    const int stages = (int)env_long("SELSCAN_TMA_STAGES", kStages);
    const bool chunked = plan.K > 1;
    auto pick = dtype == SELSCAN_F32 ? (chunked ? pick_fused_f32_chunked : pick_fused_f32_onepass)
                                     : (chunked ? pick_fused_bf16_chunked : pick_fused_bf16_onepass);
    const bool ok = pick(plan.ns, plan.nsplit, plan.vec, sp, gate, zoh, a.N, stages, &fl);
    if (!ok) return SELSCAN_ERR_UNSUPPORTED;
    FusedArgs fa;
    memset(&fa, 0, sizeof fa);
    const CUtensorMapDataType dt = dtype == SELSCAN_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const size_t es = dtype == SELSCAN_F32 ? 4 : 2;
    if (fl.threads != plan.threads) return SELSCAN_ERR_UNSUPPORTED;
    const uint32_t dpb = (uint32_t)fl.box_w;
    const uint32_t tt = (uint32_t)fl.tt;
    if (!(encode_3d(&fa.mx, dt, es, a.x, a.D, a.L, a.Bsz, dpb, tt) &&
          encode_3d(&fa.md, dt, es, a.delta, a.D, a.L, a.Bsz, dpb, tt) &&
          encode_3d(&fa.mB, dt, es, a.B, a.N, a.L, a.Bsz, (uint32_t)a.N, tt) &&
          encode_3d(&fa.mC, dt, es, a.C, a.N, a.L, a.Bsz, (uint32_t)a.N, tt) &&
          (!a.z || encode_3d(&fa.mz, dt, es, a.z, a.D, a.L, a.Bsz, dpb, tt))))
        return SELSCAN_ERR_UNSUPPORTED;
    fa.s = a;
    fa.stages = fl.stages;
    fa.fault = fault;
    {
        std::lock_guard<std::mutex> lk(g_test_mu);
        fa.publish = g_test_withhold ? 0 : 1;
        const uint64_t limit_ms = g_test_wait_ms > 0 ? (uint64_t)g_test_wait_ms : kWaitLimitNs / 1000000ull;
        fa.wait_ns = limit_ms * 1000000ull;
    }
    // Only with a softplus step is every dl >= 0, so that a state with
    // A <= 0 can only shrink and may be dropped once negligible.
    fa.trunc_tau = a.softplus ? kTruncTau : 0.0f;
    const int64_t groups = a.Bsz * plan.dtiles;
    const int64_t items_local = (int64_t)plan.K * groups;
    const int64_t items_total = items_local + (int64_t)(plan.K - 1) * groups;
    if (items_total > 0x7fffffffLL) return fail(SELSCAN_ERR_UNSUPPORTED, "too many work items");
    fa.groups = (int)groups;
    fa.items_local = (int)items_local;
    fa.items_total = (int)items_total;
    int64_t grid = items_total;
    if (plan.K > 1) {
        // A correction item reads delta (and z) of its chunk after the local
        // item of that chunk wrote y: in place over those, take the plain path.
        if (a.y == a.delta || (a.z && a.y == a.z)) return SELSCAN_ERR_UNSUPPORTED;
        const WsLayout w = fwd_workspace_layout(plan, a.Bsz, a.L, a.D, a.N, dtype);
        const size_t bdn = (size_t)(a.Bsz * a.D * a.N);
        fa.aggH = ws;
        fa.aggS = ws + (size_t)plan.K * bdn;
        fa.ctrl = reinterpret_cast<unsigned *>(reinterpret_cast<unsigned char *>(ws) + w.pairs);
        if (w.res)
            fa.yres = reinterpret_cast<unsigned char *>(ws) + w.pairs + ((w.flags + 255) & ~(size_t)255);
        unsigned *ctrl = fa.ctrl;
        int nwords = (int)(w.flags / sizeof(unsigned));
        void *cargs[] = {&ctrl, &nwords};
        const unsigned cblocks = (unsigned)((nwords + 255) / 256 < 148 ? (nwords + 255) / 256 : 148);
        cudaError_t e = launch_dependent((const void *)clear_ctrl_kernel, dim3(cblocks), dim3(256), 0, st, cargs);
        if (e != cudaSuccess) return cuda_fail(e, "clearing the chunk flags");
        const int64_t resident = (int64_t)sms * fl.ctas_per_sm;
        if (grid > resident) grid = resident;
        // When every local item is resident at once, the group's local items
        // compose its carries in slices (each waits for the group's pairs,
        // which all running items publish); otherwise the group's last local
        // item composes them alone.
        fa.spread = items_local <= grid ? 1 : 0;
        const int64_t dpb = fl.threads / plan.nsplit;
        fa.nslices = (int)((dpb * a.N + fl.threads - 1) / fl.threads);
    }
    void *args[] = {&fa};
    cudaError_t e = launch_dependent(fl.kernel, dim3((unsigned)grid), dim3(fl.threads), fl.smem, st, args);
    return e == cudaSuccess ? SELSCAN_OK : cuda_fail(e, "kernel launch");
}

// Enqueues the kernels of one forward call. `ws` holds fwd_workspace_bytes
// of the plan (null when that is 0).
int launch_fwd_into(const ScanArgs &base, const FwdPlan &plan, int dtype, int dev, int sms, float *ws,
                    cudaStream_t st)
{
    ScanArgs a = base;
    a.chunk = plan.chunk;
    a.K = plan.K;
    a.dtiles = plan.dtiles;
    if (a.Bsz * plan.dtiles > 0x7fffffffLL) return fail(SELSCAN_ERR_UNSUPPORTED, "grid too large");
    const WsLayout w = fwd_workspace_layout(plan, a.Bsz, a.L, a.D, a.N, dtype);
    float *hT_final = a.hT;
    if (plan.stage_hT)
        a.hT = reinterpret_cast<float *>(reinterpret_cast<unsigned char *>(ws) + w.total - w.stage);
    unsigned *fault = nullptr;
    int rc = fault_word(dev, st, &fault);
    if (rc != SELSCAN_OK) return rc;
    rc = SELSCAN_ERR_UNSUPPORTED;
    if (plan.tma) {
        rc = launch_fused(a, plan, dtype, sms, ws, fault, st);
        if (rc == SELSCAN_ERR_UNSUPPORTED) g_err[0] = '\0';
    }
    if (rc == SELSCAN_ERR_UNSUPPORTED) {
        // The plain-load kernels run CTAs of kScanThreads.
        const int64_t cpc = kScanThreads / plan.nsplit;
        a.dtiles = (int)((a.D + cpc - 1) / cpc);
        if (a.Bsz * a.dtiles > 0x7fffffffLL) return fail(SELSCAN_ERR_UNSUPPORTED, "grid too large");
        if (plan.K > 1) {
            const int64_t bd = a.Bsz * a.D;
            a.agg_h = ws;
            a.agg_s = a.agg_h + (size_t)plan.K * (size_t)bd * (size_t)a.N;
        }
        rc = launch_plain_kernels(a, plan.ns, plan.nsplit, plan.vec, dtype, st);
    }
    if (rc == SELSCAN_OK && plan.stage_hT) {
        const cudaError_t e = cudaMemcpyAsync(hT_final, a.hT, w.stage, cudaMemcpyDeviceToDevice, st);
        if (e != cudaSuccess) return cuda_fail(e, "final state copy");
    }
    return rc;
}

// One forward call with its workspace from the library's stream-ordered pool.
int launch_fwd(const ScanArgs &base, const FwdPlan &plan, int dtype, int dev, int sms, cudaStream_t st)
{
    const size_t bytes = fwd_workspace_bytes(plan, base.Bsz, base.L, base.D, base.N, dtype);
    void *ws = nullptr;
    if (bytes > 0) {
        cudaMemPool_t pool = nullptr;
        int rc = workspace_pool(dev, &pool);
        if (rc != SELSCAN_OK) return rc;
        cudaError_t e = cudaMallocFromPoolAsync(&ws, bytes, pool, st);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(SELSCAN_ERR_NO_MEMORY, "chunk workspace of %zu bytes: %s", bytes, cudaGetErrorString(e));
        }
    }
    int rc = launch_fwd_into(base, plan, dtype, dev, sms, static_cast<float *>(ws), st);
    if (ws) cudaFreeAsync(ws, st);
    return rc;
}

// Argument checks shared by the forward entry points (no CUDA call).
// *empty is set when there is nothing to compute (Bsz == 0 or D == 0).
int check_fwd_args(const void *x, const void *delta, const float *A, const void *B, const void *C,
                   const void *y, int64_t Bsz, int64_t L, int64_t D, int64_t N, int dtype, const float *h0,
                   const float *hT, bool *empty, const float *Dskip = nullptr, const void *z = nullptr)
{
    *empty = false;
    if (dtype != SELSCAN_F32 && dtype != SELSCAN_BF16)
        return fail(SELSCAN_ERR_INVALID_ARG, "dtype %d is neither SELSCAN_F32 nor SELSCAN_BF16", dtype);
    if (Bsz < 0 || L < 0 || D < 0)
        return fail(SELSCAN_ERR_INVALID_ARG, "negative size (Bsz=%lld L=%lld D=%lld)",
                    (long long)Bsz, (long long)L, (long long)D);
    if (N < 1)
        return fail(SELSCAN_ERR_INVALID_ARG, "N=%lld must be >= 1", (long long)N);
    if (N > SELSCAN_MAX_N)
        return fail(SELSCAN_ERR_UNSUPPORTED, "N=%lld exceeds SELSCAN_MAX_N=%d", (long long)N, SELSCAN_MAX_N);
    int64_t nld, nln, ndn;
    if (!mul_ok(Bsz, L, D, &nld) || !mul_ok(Bsz, L, N, &nln) || !mul_ok(Bsz, D, N, &ndn))
        return fail(SELSCAN_ERR_INVALID_ARG, "sizes overflow (Bsz=%lld L=%lld D=%lld N=%lld)",
                    (long long)Bsz, (long long)L, (long long)D, (long long)N);
    if (Bsz == 0 || D == 0) {
        *empty = true;
        return SELSCAN_OK;
    }
    if (!A)
        return fail(SELSCAN_ERR_INVALID_ARG, "A is NULL");
    const size_t es = dtype == SELSCAN_F32 ? 4 : 2;
    if (L > 0) {
        if (!x || !delta || !B || !C || !y)
            return fail(SELSCAN_ERR_INVALID_ARG, "x, delta, B, C and y must be non-NULL when L > 0");
        if (!aligned(x, es) || !aligned(delta, es) || !aligned(B, es) || !aligned(C, es) || !aligned(y, es) ||
            !aligned(z, es))
            return fail(SELSCAN_ERR_INVALID_ARG, "x, delta, B, C, y, z must be aligned to their element size");
    }
    if (!aligned(A, 4) || !aligned(h0, 4) || !aligned(hT, 4) || !aligned(Dskip, 4))
        return fail(SELSCAN_ERR_INVALID_ARG, "A, h0, hT, Dskip must be 4-byte aligned");

    const Range ry = range(L > 0 ? y : nullptr, nld * es, "y"), rhT = range(hT, ndn * 4, "hT");
    struct Input {
        Range r;
        bool y_may_equal;    // y may be this buffer exactly (in-place output)
        bool hT_may_equal;   // hT may be this buffer exactly (resume in place)
    };
    const Input ins[] = {
        {range(x, nld * es, "x"), true, false},      {range(delta, nld * es, "delta"), true, false},
        {range(B, nln * es, "B"), false, false},     {range(C, nln * es, "C"), false, false},
        {range(A, D * N * 4, "A"), false, false},    {range(h0, ndn * 4, "h0"), false, true},
        {range(L > 0 ? z : nullptr, nld * es, "z"), true, false}, {range(Dskip, D * 4, "Dskip"), false, false},
    };
    for (const Input &in : ins) {
        if (overlaps(ry, in.r) && !(in.y_may_equal && in.r.lo == ry.lo))
            return fail(SELSCAN_ERR_INVALID_ARG, "y overlaps %s", in.r.name);
        if (overlaps(rhT, in.r) && !(in.hT_may_equal && in.r.lo == rhT.lo))
            return fail(SELSCAN_ERR_INVALID_ARG, "hT overlaps %s", in.r.name);
    }
    if (overlaps(ry, rhT))
        return fail(SELSCAN_ERR_INVALID_ARG, "y overlaps hT");
    return SELSCAN_OK;
}

// L == 0: the final state is the initial state (or zeros); nothing else is written.
int empty_sequence_state(const float *h0, float *hT, int64_t Bsz, int64_t D, int64_t N, cudaStream_t st)
{
    if (!hT || hT == h0) return SELSCAN_OK;
    const size_t bytes = (size_t)(Bsz * D * N) * 4;
    cudaError_t e = h0 ? cudaMemcpyAsync(hT, h0, bytes, cudaMemcpyDeviceToDevice, st) : cudaMemsetAsync(hT, 0, bytes, st);
    return e == cudaSuccess ? SELSCAN_OK : cuda_fail(e, "L == 0 state copy");
}

} // namespace
} // namespace selscan

using namespace selscan;

extern "C" int selscan_fwd(const void *x, const void *delta, const float *A, const void *B,
                           const void *C, void *y, int64_t Bsz, int64_t L, int64_t D, int64_t N,
                           int dtype, int delta_softplus, const float *h0, float *hT, void *stream)
{
    return selscan_fwd_gated(x, delta, A, B, C, nullptr, nullptr, y, Bsz, L, D, N, dtype, delta_softplus,
                             h0, hT, stream);
}

extern "C" int selscan_fwd_gated(const void *x, const void *delta, const float *A, const void *B,
                                 const void *C, const float *Dskip, const void *z, void *y, int64_t Bsz,
                                 int64_t L, int64_t D, int64_t N, int dtype, int delta_softplus,
                                 const float *h0, float *hT, void *stream)
{
    return selscan_fwd_ex(x, delta, A, B, C, Dskip, z, y, Bsz, L, D, N, dtype,
                          delta_softplus ? SELSCAN_FLAG_SOFTPLUS : 0, h0, hT, stream);
}

extern "C" int selscan_fwd_ex(const void *x, const void *delta, const float *A, const void *B,
                              const void *C, const float *Dskip, const void *z, void *y, int64_t Bsz,
                              int64_t L, int64_t D, int64_t N, int dtype, int flags, const float *h0,
                              float *hT, void *stream)
{
    g_err[0] = '\0';
    if (flags & ~(SELSCAN_FLAG_SOFTPLUS | SELSCAN_FLAG_ZOH))
        return fail(SELSCAN_ERR_INVALID_ARG, "unknown flags 0x%x", (unsigned)flags);
    const int delta_softplus = (flags & SELSCAN_FLAG_SOFTPLUS) != 0;
    bool empty = false;
    int rc = check_fwd_args(x, delta, A, B, C, y, Bsz, L, D, N, dtype, h0, hT, &empty, Dskip, z);
    if (rc != SELSCAN_OK || empty) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (L == 0) return empty_sequence_state(h0, hT, Bsz, D, N, st);

    int dev = 0, sms = 0;
    rc = device_info(&dev, &sms);
    if (rc != SELSCAN_OK) return rc;
    const size_t es = dtype == SELSCAN_F32 ? 4 : 2;
    FwdPlan plan;
    plan_fwd(Bsz, L, D, N, es, x, delta, B, C, h0, hT, sms, &plan);
    ScanArgs a;
    memset(&a, 0, sizeof a);
    a.x = x; a.delta = delta; a.B = B; a.C = C; a.A = A; a.y = y; a.h0 = h0; a.hT = hT;
    a.Bsz = Bsz; a.L = L; a.D = D; a.N = N;
    a.Dskip = Dskip; a.z = z;
    a.softplus = delta_softplus ? 1 : 0;
    a.zoh = (flags & SELSCAN_FLAG_ZOH) ? 1 : 0;
    return launch_fwd(a, plan, dtype, dev, sms, st);
}

// ---- allocation-free forward ----------------------------------------------
// Chunk-carry scratch for callers that cannot allocate: a fixed array in the
// library's device image. Host code must not use the name as an address (on
// the host it is only a stand-in); its device address is looked up once per
// device with that device current.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SELSCAN_NOALLOC_SCRATCH_BYTES];

namespace selscan {
namespace {
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices];

int noalloc_scratch(int dev, float **out)
{
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the scratch array");
        g_noalloc_ptr[dev] = p;
    }
    *out = static_cast<float *>(g_noalloc_ptr[dev]);
    return SELSCAN_OK;
}
} // namespace
} // namespace selscan

extern "C" int selscan_fwd_noalloc(const void *x, const void *delta, const float *A, const void *B,
                                   const void *C, void *y, int64_t Bsz, int64_t L, int64_t D, int64_t N,
                                   int dtype, int delta_softplus, const float *h0, float *hT, void *stream)
{
    g_err[0] = '\0';
    bool empty = false;
    int rc = check_fwd_args(x, delta, A, B, C, y, Bsz, L, D, N, dtype, h0, hT, &empty);
    if (rc != SELSCAN_OK || empty) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (L == 0) return empty_sequence_state(h0, hT, Bsz, D, N, st);

    int dev = 0, sms = 0;
    rc = device_info(&dev, &sms);
    if (rc != SELSCAN_OK) return rc;
    const size_t es = dtype == SELSCAN_F32 ? 4 : 2;
    FwdPlan plan;
    plan_fwd(Bsz, L, D, N, es, x, delta, B, C, h0, hT, sms, &plan);
    const size_t need = fwd_workspace_bytes(plan, Bsz, L, D, N, dtype);
    if (need > SELSCAN_NOALLOC_SCRATCH_BYTES)
        return fail(SELSCAN_ERR_UNSUPPORTED,
                    "this problem needs %zu bytes of chunk scratch (%d chunks) but the allocation-free entry "
                    "point has %u; use selscan_fwd or split the sequence",
                    need, plan.K, (unsigned)SELSCAN_NOALLOC_SCRATCH_BYTES);
    float *ws = nullptr;
    if (need > 0) {
        rc = noalloc_scratch(dev, &ws);
        if (rc != SELSCAN_OK) return rc;
    }
    ScanArgs a;
    memset(&a, 0, sizeof a);
    a.x = x; a.delta = delta; a.B = B; a.C = C; a.A = A; a.y = y; a.h0 = h0; a.hT = hT;
    a.Bsz = Bsz; a.L = L; a.D = D; a.N = N;
    a.softplus = delta_softplus ? 1 : 0;
    return launch_fwd_into(a, plan, dtype, dev, sms, ws, st);
}

// ---- forward from host buffers --------------------------------------------
// The sequence is cut into pieces along L. Piece p's inputs are copied in on
// one stream while piece p-1 is scanned on a second and piece p-2's output is
// copied out on a third; the scan of each piece starts from the final state
// of the one before (h0/hT chaining on the device), so pieces compose exactly
// like chunks. Device staging is double-buffered per piece.

namespace selscan {
namespace {

struct HostPipe {
    cudaStream_t in = nullptr, in2 = nullptr, comp = nullptr, out = nullptr;
    cudaEvent_t ev[10] = {};  // start, alloc, in[2], comp[2], out[2], in2[2]
    std::mutex mu;            // one host-buffer call at a time per device
};
HostPipe g_pipe[kMaxDevices];
std::mutex g_pipe_init;

int host_pipe(int dev, HostPipe **out)
{
    std::lock_guard<std::mutex> lk(g_pipe_init);
    HostPipe &hp = g_pipe[dev];
    if (!hp.in) {
        cudaStream_t s[4];
        for (int i = 0; i < 4; ++i) {
            cudaError_t e = cudaStreamCreateWithFlags(&s[i], cudaStreamNonBlocking);
            if (e != cudaSuccess) return cuda_fail(e, "cudaStreamCreateWithFlags");
        }
        for (cudaEvent_t &ev : hp.ev) {
            cudaError_t e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
            if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreateWithFlags");
        }
        hp.in = s[0];
        hp.comp = s[1];
        hp.out = s[2];
        hp.in2 = s[3];
    }
    *out = &hp;
    return SELSCAN_OK;
}

// Rows of `width` bytes, `rows` of them, between pitched buffers.
cudaError_t copy_rows(void *dst, size_t dpitch, const void *src, size_t spitch, size_t width, size_t rows,
                      cudaMemcpyKind kind, cudaStream_t st)
{
    return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, rows, kind, st);
}

} // namespace
} // namespace selscan

extern "C" int selscan_fwd_host(const void *x, const void *delta, const float *A, const void *B,
                                const void *C, void *y, int64_t Bsz, int64_t L, int64_t D, int64_t N,
                                int dtype, int delta_softplus, const float *h0, float *hT, void *stream)
{
    return selscan_fwd_host_ex(x, delta, A, B, C, nullptr, nullptr, y, Bsz, L, D, N, dtype,
                               delta_softplus ? SELSCAN_FLAG_SOFTPLUS : 0, h0, hT, stream);
}

extern "C" int selscan_fwd_host_ex(const void *x, const void *delta, const float *A, const void *B,
                                   const void *C, const float *Dskip, const void *z, void *y, int64_t Bsz,
                                   int64_t L, int64_t D, int64_t N, int dtype, int flags, const float *h0,
                                   float *hT, void *stream)
{
    g_err[0] = '\0';
    if (flags & ~(SELSCAN_FLAG_SOFTPLUS | SELSCAN_FLAG_ZOH))
        return fail(SELSCAN_ERR_INVALID_ARG, "unknown flags 0x%x", (unsigned)flags);
    const int delta_softplus = (flags & SELSCAN_FLAG_SOFTPLUS) != 0;
    bool empty = false;
    int rc = check_fwd_args(x, delta, A, B, C, y, Bsz, L, D, N, dtype, h0, hT, &empty, Dskip, z);
    if (rc != SELSCAN_OK || empty) return rc;
    const size_t es = dtype == SELSCAN_F32 ? 4 : 2;
    const size_t state_bytes = (size_t)(Bsz * D * N) * 4;
    if (L == 0) {   // the final state is the initial state (or zeros)
        if (hT && hT != h0) {
            if (h0) memcpy(hT, h0, state_bytes);
            else memset(hT, 0, state_bytes);
        }
        return SELSCAN_OK;
    }

    int dev = 0, sms = 0;
    rc = device_info(&dev, &sms);
    if (rc != SELSCAN_OK) return rc;
    HostPipe *hp = nullptr;
    rc = host_pipe(dev, &hp);
    if (rc != SELSCAN_OK) return rc;
    std::lock_guard<std::mutex> lk(hp->mu);

    // Piece length: about 32 MB of input per piece, at least 64 steps, and
    // at least two pieces when L >= 128 so that copies overlap. Measured on
    // B300 (pinned buffers): Bsz=2 L=2048 D=1536 takes 1.40 ms per call in
    // two pieces against 1.54 ms in seven; Bsz=1 L=131072 37 ms in pieces of
    // 2700 or 4096 steps against 43 ms in pieces of 676 (fewer, larger
    // copies and launches per call).
    // SELSCAN_HOST_PIECE overrides it, for tests.
    const size_t step_in = (size_t)Bsz * (size_t)((z ? 3 : 2) * D + 2 * N) * es;
    int64_t lp = (int64_t)((32u << 20) / (step_in ? step_in : 1));
    if (lp < 64) lp = 64;
    if (lp >= L && L >= 128) lp = (L + 1) / 2;
    const long force = env_long("SELSCAN_HOST_PIECE", 0);
    if (force > 0) lp = force;
    if (lp > L) lp = L;
    const int64_t pieces = (L + lp - 1) / lp;
    const bool chain = pieces > 1 || h0 || hT;

    // Device staging: per slot x, delta, y (and z) (Bsz, lp, D) and B, C
    // (Bsz, lp, N); then A, Dskip, and two states (piece p reads one and
    // writes the other, so no scan updates its state in place). Every part
    // starts on a 256-byte boundary.
    auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
    const size_t bx = up((size_t)(Bsz * lp * D) * es), bn = up((size_t)(Bsz * lp * N) * es);
    const size_t slot_bytes = (z ? 4 : 3) * bx + 2 * bn;
    const size_t a_bytes = up((size_t)(D * N) * 4), dsk_bytes = Dskip ? up((size_t)D * 4) : 0;
    const size_t total = 2 * slot_bytes + a_bytes + dsk_bytes + (chain ? 2 * up(state_bytes) : 0);
    cudaMemPool_t pool = nullptr;
    rc = workspace_pool(dev, &pool);
    if (rc != SELSCAN_OK) return rc;

    cudaStream_t caller = static_cast<cudaStream_t>(stream);
    cudaEvent_t ev_start = hp->ev[0], ev_alloc = hp->ev[1];
    cudaEvent_t *ev_in = hp->ev + 2, *ev_comp = hp->ev + 4, *ev_out = hp->ev + 6, *ev_in2 = hp->ev + 8;
    // Inputs over two copy streams (x and B on one, delta and C on the other)
    // unless SELSCAN_HOST_COPY_STREAMS=1.
    const bool two_in = env_long("SELSCAN_HOST_COPY_STREAMS", 2) != 1;
    cudaStream_t in2 = two_in ? hp->in2 : hp->in;
    cudaError_t e = cudaEventRecord(ev_start, caller);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    cudaStreamWaitEvent(hp->comp, ev_start, 0);
    unsigned char *ws = nullptr;
    e = cudaMallocFromPoolAsync(reinterpret_cast<void **>(&ws), total, pool, hp->comp);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(SELSCAN_ERR_NO_MEMORY, "host staging of %zu bytes: %s", total, cudaGetErrorString(e));
    }
    cudaEventRecord(ev_alloc, hp->comp);
    cudaStreamWaitEvent(hp->in, ev_alloc, 0);
    cudaStreamWaitEvent(hp->in2, ev_alloc, 0);
    cudaStreamWaitEvent(hp->out, ev_alloc, 0);
    float *A_d = reinterpret_cast<float *>(ws + 2 * slot_bytes);
    float *Dskip_d = Dskip ? reinterpret_cast<float *>(ws + 2 * slot_bytes + a_bytes) : nullptr;
    float *state_d[2] = {nullptr, nullptr};
    if (chain) {
        state_d[0] = reinterpret_cast<float *>(ws + 2 * slot_bytes + a_bytes + dsk_bytes);
        state_d[1] = reinterpret_cast<float *>(reinterpret_cast<unsigned char *>(state_d[0]) + up(state_bytes));
    }

    e = cudaMemcpyAsync(A_d, A, (size_t)(D * N) * 4, cudaMemcpyHostToDevice, hp->in);
    if (e == cudaSuccess && Dskip)
        e = cudaMemcpyAsync(Dskip_d, Dskip, (size_t)D * 4, cudaMemcpyHostToDevice, hp->in);
    if (e == cudaSuccess && h0)
        e = cudaMemcpyAsync(state_d[0], h0, state_bytes, cudaMemcpyHostToDevice, hp->in);

    const size_t rows = (size_t)Bsz;
    const size_t xpitch = (size_t)(L * D) * es, npitch = (size_t)(L * N) * es;
    for (int64_t p = 0; p < pieces && e == cudaSuccess && rc == SELSCAN_OK; ++p) {
        const int slot = (int)(p & 1);
        unsigned char *base = ws + slot * slot_bytes;
        void *x_d = base, *dl_d = base + bx, *y_d = base + 2 * bx, *B_d = base + 3 * bx, *C_d = base + 3 * bx + bn;
        void *z_d = z ? base + 3 * bx + 2 * bn : nullptr;
        const int64_t l0 = p * lp;
        const int64_t n = L - l0 < lp ? L - l0 : lp;
        const size_t wx = (size_t)(n * D) * es, wn = (size_t)(n * N) * es;
        const size_t ox = (size_t)(l0 * D) * es, on = (size_t)(l0 * N) * es;

        // In: the slot's inputs are free once the scan of piece p-2 is done.
        if (p >= 2) {
            cudaStreamWaitEvent(hp->in, ev_comp[slot], 0);
            if (two_in) cudaStreamWaitEvent(in2, ev_comp[slot], 0);
        }
        e = copy_rows(x_d, wx, static_cast<const unsigned char *>(x) + ox, xpitch, wx, rows, cudaMemcpyHostToDevice, hp->in);
        if (e == cudaSuccess)
            e = copy_rows(dl_d, wx, static_cast<const unsigned char *>(delta) + ox, xpitch, wx, rows, cudaMemcpyHostToDevice, in2);
        if (e == cudaSuccess)
            e = copy_rows(B_d, wn, static_cast<const unsigned char *>(B) + on, npitch, wn, rows, cudaMemcpyHostToDevice, hp->in);
        if (e == cudaSuccess)
            e = copy_rows(C_d, wn, static_cast<const unsigned char *>(C) + on, npitch, wn, rows, cudaMemcpyHostToDevice, in2);
        if (e == cudaSuccess && z)
            e = copy_rows(z_d, wx, static_cast<const unsigned char *>(z) + ox, xpitch, wx, rows, cudaMemcpyHostToDevice, in2);
        if (e != cudaSuccess) break;
        cudaEventRecord(ev_in[slot], hp->in);
        if (two_in) cudaEventRecord(ev_in2[slot], in2);

        // Scan: after the inputs landed and piece p-2's output left the slot.
        cudaStreamWaitEvent(hp->comp, ev_in[slot], 0);
        if (two_in) cudaStreamWaitEvent(hp->comp, ev_in2[slot], 0);
        if (p >= 2) cudaStreamWaitEvent(hp->comp, ev_out[slot], 0);
        FwdPlan plan;
        const float *h_in = (p == 0 && !h0) ? nullptr : state_d[p & 1];
        float *h_out = state_d[(p + 1) & 1];
        plan_fwd(Bsz, n, D, N, es, x_d, dl_d, B_d, C_d, h_in, h_out, sms, &plan);
        ScanArgs a;
        memset(&a, 0, sizeof a);
        a.x = x_d; a.delta = dl_d; a.B = B_d; a.C = C_d; a.A = A_d; a.y = y_d;
        a.h0 = h_in;
        a.hT = h_out;
        a.Bsz = Bsz; a.L = n; a.D = D; a.N = N;
        a.Dskip = Dskip_d; a.z = z_d;
        a.softplus = delta_softplus ? 1 : 0;
        a.zoh = (flags & SELSCAN_FLAG_ZOH) ? 1 : 0;
        rc = launch_fwd(a, plan, dtype, dev, sms, hp->comp);
        if (rc != SELSCAN_OK) break;
        cudaEventRecord(ev_comp[slot], hp->comp);

        // Out.
        cudaStreamWaitEvent(hp->out, ev_comp[slot], 0);
        e = copy_rows(static_cast<unsigned char *>(y) + ox, xpitch, y_d, wx, wx, rows, cudaMemcpyDeviceToHost, hp->out);
        if (e != cudaSuccess) break;
        cudaEventRecord(ev_out[slot], hp->out);
    }
    if (e == cudaSuccess && rc == SELSCAN_OK && hT)
        e = cudaMemcpyAsync(hT, state_d[pieces & 1], state_bytes, cudaMemcpyDeviceToHost, hp->out);

    // Drain every stream, then give the staging back and let the caller's
    // stream continue after this call.
    cudaError_t e2 = cudaStreamSynchronize(hp->in);
    cudaError_t e5 = cudaStreamSynchronize(hp->in2);
    cudaError_t e3 = cudaStreamSynchronize(hp->out);
    cudaFreeAsync(ws, hp->comp);
    cudaError_t e4 = cudaStreamSynchronize(hp->comp);
    if (rc != SELSCAN_OK) return rc;
    if (e == cudaSuccess) e = e2;
    if (e == cudaSuccess) e = e5;
    if (e == cudaSuccess) e = e3;
    if (e == cudaSuccess) e = e4;
    if (e != cudaSuccess) return cuda_fail(e, "host-buffer pipeline");
    return SELSCAN_OK;
}

extern "C" int selscan_step(float *state, const float *x, const float *delta, const float *A,
                            const float *B, const float *C, float *y, int64_t Bsz, int64_t D,
                            int64_t N, void *stream)
{
    return selscan_step_gated(state, x, delta, A, B, C, nullptr, nullptr, y, Bsz, D, N, stream);
}

extern "C" int selscan_step_gated(float *state, const float *x, const float *delta, const float *A,
                                  const float *B, const float *C, const float *Dskip, const float *z,
                                  float *y, int64_t Bsz, int64_t D, int64_t N, void *stream)
{
    return selscan_step_ex(state, x, delta, A, B, C, Dskip, z, y, Bsz, D, N, 0, stream);
}

extern "C" int selscan_step_ex(float *state, const float *x, const float *delta, const float *A,
                               const float *B, const float *C, const float *Dskip, const float *z,
                               float *y, int64_t Bsz, int64_t D, int64_t N, int flags, void *stream)
{
    g_err[0] = '\0';
    if (flags & ~SELSCAN_FLAG_ZOH)
        return fail(SELSCAN_ERR_INVALID_ARG, "unknown flags 0x%x (the decode step takes SELSCAN_FLAG_ZOH only)",
                    (unsigned)flags);
    if (Bsz < 0 || D < 0)
        return fail(SELSCAN_ERR_INVALID_ARG, "negative size (Bsz=%lld D=%lld)", (long long)Bsz, (long long)D);
    if (N < 1)
        return fail(SELSCAN_ERR_INVALID_ARG, "N=%lld must be >= 1", (long long)N);
    if (N > SELSCAN_MAX_N)
        return fail(SELSCAN_ERR_UNSUPPORTED, "N=%lld exceeds SELSCAN_MAX_N=%d", (long long)N, SELSCAN_MAX_N);
    int64_t ndn, nd1;
    if (!mul_ok(Bsz, D, N, &ndn) || !mul_ok(Bsz, D, 1, &nd1))
        return fail(SELSCAN_ERR_INVALID_ARG, "sizes overflow");
    if (Bsz == 0 || D == 0)
        return SELSCAN_OK;
    if (!state || !x || !delta || !A || !B || !C || !y)
        return fail(SELSCAN_ERR_INVALID_ARG, "state, x, delta, A, B, C and y must be non-NULL");
    const void *ptrs[] = {state, x, delta, A, B, C, y, Dskip, z};
    for (const void *p : ptrs)
        if (!aligned(p, 4))
            return fail(SELSCAN_ERR_INVALID_ARG, "every pointer must be 4-byte aligned");
    const Range rs = range(state, ndn * 4, "state"), ry = range(y, nd1 * 4, "y");
    const Range ins[] = {range(x, nd1 * 4, "x"), range(delta, nd1 * 4, "delta"), range(A, D * N * 4, "A"),
                         range(B, Bsz * N * 4, "B"), range(C, Bsz * N * 4, "C"),
                         range(Dskip, D * 4, "Dskip"), range(z, nd1 * 4, "z")};
    for (const Range &r : ins) {
        if (overlaps(rs, r)) return fail(SELSCAN_ERR_INVALID_ARG, "state overlaps %s", r.name);
        if (overlaps(ry, r)) return fail(SELSCAN_ERR_INVALID_ARG, "y overlaps %s", r.name);
    }
    if (overlaps(rs, ry))
        return fail(SELSCAN_ERR_INVALID_ARG, "y overlaps state");

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    StepArgs a{state, x, delta, A, B, C, y, Dskip, z, Bsz, D, N};
    const bool zoh = (flags & SELSCAN_FLAG_ZOH) != 0;
    // 4V states per lane (V 16-byte groups), G = N / (4V) lanes per chain; G
    // must divide the warp so that a chain's lanes never straddle two warps.
    // V = 1 measured fastest on B300 (Bsz=256, D=2560, N=16, state from HBM:
    // 17.3 us per step against 18.7 with V = 2 and 24.4 with V = 4);
    // SELSCAN_STEP_V selects another.
    long V = env_long("SELSCAN_STEP_V", 1);
    if (V != 1 && V != 2 && V != 4) V = 1;
    while (V > 1 && N % (4 * V) != 0) V /= 2;
    const int G = (int)(N / (4 * V));
    const bool vec = (N % 4 == 0) && (G == 1 || G == 2 || G == 4 || G == 8 || G == 16) &&
                     aligned(state, 16) && aligned(A, 16) && aligned(B, 16) && aligned(C, 16);
    return launch_step_kernel(a, G, (int)V, vec, zoh, st);
}

// ---- causal depthwise convolution before the scan ------------------------

extern "C" int selscan_conv1d(const void *x, const float *w, const float *bias, void *out, int64_t Bsz,
                              int64_t L, int64_t D, int64_t K, int dtype, int silu, const float *state_in,
                              float *state_out, void *stream)
{
    g_err[0] = '\0';
    if (dtype != SELSCAN_F32 && dtype != SELSCAN_BF16)
        return fail(SELSCAN_ERR_INVALID_ARG, "dtype %d is neither SELSCAN_F32 nor SELSCAN_BF16", dtype);
    if (Bsz < 0 || L < 0 || D < 0)
        return fail(SELSCAN_ERR_INVALID_ARG, "negative size (Bsz=%lld L=%lld D=%lld)", (long long)Bsz,
                    (long long)L, (long long)D);
    if (K < 1 || K > kConvMaxK)
        return fail(K < 1 ? SELSCAN_ERR_INVALID_ARG : SELSCAN_ERR_UNSUPPORTED, "K=%lld must be in 1..%d",
                    (long long)K, kConvMaxK);
    int64_t nld, nds;
    if (!mul_ok(Bsz, L, D, &nld) || !mul_ok(Bsz, D, K - 1, &nds))
        return fail(SELSCAN_ERR_INVALID_ARG, "sizes overflow");
    if (Bsz == 0 || D == 0)
        return SELSCAN_OK;
    if (Bsz > 65535 || (L + kConvT - 1) / kConvT > 65535 || (D + kConvThreads - 1) / kConvThreads > 0x7fffffffLL)
        return fail(SELSCAN_ERR_UNSUPPORTED, "grid too large (Bsz <= 65535, L <= %lld)", 65535LL * kConvT);
    const size_t es = dtype == SELSCAN_F32 ? 4 : 2;
    if (!w || (L > 0 && (!x || !out)))
        return fail(SELSCAN_ERR_INVALID_ARG, "w, and x and out when L > 0, must be non-NULL");
    if (!aligned(x, es) || !aligned(out, es) || !aligned(w, 4) || !aligned(bias, 4) || !aligned(state_in, 4) ||
        !aligned(state_out, 4))
        return fail(SELSCAN_ERR_INVALID_ARG, "x and out must be aligned to their element size, the rest to 4 bytes");
    const Range ro = range(L > 0 ? out : nullptr, nld * (int64_t)es, "out"), rs = range(state_out, nds * 4, "state_out");
    const Range ins[] = {range(L > 0 ? x : nullptr, nld * (int64_t)es, "x"), range(w, D * K * 4, "w"),
                         range(bias, D * 4, "bias"), range(state_in, nds * 4, "state_in")};
    for (const Range &r : ins) {
        if (overlaps(ro, r)) return fail(SELSCAN_ERR_INVALID_ARG, "out overlaps %s", r.name);
        if (overlaps(rs, r)) return fail(SELSCAN_ERR_INVALID_ARG, "state_out overlaps %s", r.name);
    }
    if (overlaps(ro, rs))
        return fail(SELSCAN_ERR_INVALID_ARG, "out overlaps state_out");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (L == 0) {   // the carried state passes through unchanged
        if (!state_out || nds == 0) return SELSCAN_OK;
        cudaError_t e = state_in ? cudaMemcpyAsync(state_out, state_in, (size_t)nds * 4, cudaMemcpyDeviceToDevice, st)
                                 : cudaMemsetAsync(state_out, 0, (size_t)nds * 4, st);
        return e == cudaSuccess ? SELSCAN_OK : cuda_fail(e, "L == 0 state copy");
    }
    ConvArgs a{x, w, bias, out, state_in, state_out, Bsz, L, D, silu ? 1 : 0};
    // Four channels per thread when rows allow vector access (D % 4 == 0,
    // x and out aligned to 4 elements, bias to 16 bytes).
    const bool vec = D % 4 == 0 && aligned(x, 4 * es) && aligned(out, 4 * es) && aligned(bias, 16) &&
                     env_long("SELSCAN_CONV_VEC", 1) != 0;
    return launch_conv1d_kernel(a, K, dtype, vec, st);
}

extern "C" int selscan_conv1d_step(float *conv_state, const float *x, const float *w, const float *bias,
                                   float *out, int64_t Bsz, int64_t D, int64_t K, int silu, void *stream)
{
    g_err[0] = '\0';
    if (Bsz < 0 || D < 0)
        return fail(SELSCAN_ERR_INVALID_ARG, "negative size (Bsz=%lld D=%lld)", (long long)Bsz, (long long)D);
    if (K < 1 || K > kConvMaxK)
        return fail(K < 1 ? SELSCAN_ERR_INVALID_ARG : SELSCAN_ERR_UNSUPPORTED, "K=%lld must be in 1..%d",
                    (long long)K, kConvMaxK);
    int64_t nd, nds;
    if (!mul_ok(Bsz, D, 1, &nd) || !mul_ok(Bsz, D, K - 1, &nds))
        return fail(SELSCAN_ERR_INVALID_ARG, "sizes overflow");
    if (Bsz == 0 || D == 0)
        return SELSCAN_OK;
    if (!x || !w || !out || (K > 1 && !conv_state))
        return fail(SELSCAN_ERR_INVALID_ARG, "x, w, out (and conv_state when K > 1) must be non-NULL");
    const void *ptrs[] = {conv_state, x, w, bias, out};
    for (const void *p : ptrs)
        if (!aligned(p, 4))
            return fail(SELSCAN_ERR_INVALID_ARG, "every pointer must be 4-byte aligned");
    const Range rs = range(K > 1 ? conv_state : nullptr, nds * 4, "conv_state"), ro = range(out, nd * 4, "out");
    const Range ins[] = {range(x, nd * 4, "x"), range(w, D * K * 4, "w"), range(bias, D * 4, "bias")};
    for (const Range &r : ins) {
        if (overlaps(rs, r)) return fail(SELSCAN_ERR_INVALID_ARG, "conv_state overlaps %s", r.name);
        if (overlaps(ro, r)) return fail(SELSCAN_ERR_INVALID_ARG, "out overlaps %s", r.name);
    }
    if (overlaps(rs, ro))
        return fail(SELSCAN_ERR_INVALID_ARG, "out overlaps conv_state");
    ConvStepArgs a{conv_state, x, w, bias, out, Bsz, D, silu ? 1 : 0};
    return launch_conv1d_step_kernel(a, K, static_cast<cudaStream_t>(stream));
}

extern "C" int selscan_fwd_plan(int64_t Bsz, int64_t L, int64_t D, int64_t N, int dtype, int *chunks,
                                int64_t *chunk_len, int *launches, int64_t *workspace_bytes)
{
    g_err[0] = '\0';
    if (dtype != SELSCAN_F32 && dtype != SELSCAN_BF16)
        return fail(SELSCAN_ERR_INVALID_ARG, "dtype %d is neither SELSCAN_F32 nor SELSCAN_BF16", dtype);
    if (Bsz < 0 || L < 0 || D < 0 || N < 1)
        return fail(SELSCAN_ERR_INVALID_ARG, "bad sizes");
    if (N > SELSCAN_MAX_N)
        return fail(SELSCAN_ERR_UNSUPPORTED, "N=%lld exceeds SELSCAN_MAX_N=%d", (long long)N, SELSCAN_MAX_N);
    int dev = 0, sms = 0;
    int rc = device_info(&dev, &sms);
    if (rc != SELSCAN_OK) return rc;
    FwdPlan plan;
    const size_t es = dtype == SELSCAN_F32 ? 4 : 2;
    // Alignment does not change the chunking; pass 16-byte aligned stand-ins.
    const void *al = reinterpret_cast<const void *>(uintptr_t(256));
    plan_fwd(Bsz, L, D, N, es, al, al, al, al, nullptr, nullptr, sms, &plan);
    const bool empty = Bsz == 0 || D == 0 || L == 0;
    if (chunks) *chunks = empty ? 0 : plan.K;
    if (chunk_len) *chunk_len = empty ? 0 : plan.chunk;
    // The TMA path runs as one kernel (plus a flag reset when chunked); the
    // plain path as aggregate + carry + readout kernels.
    // TMA path: the fused kernel, after the kernel that clears the control
    // words of a chunked plan; plain path: aggregate, carry and readout.
    if (launches) *launches = empty ? 0 : (plan.K > 1 ? (plan.tma ? 2 : 3) : 1);
    if (workspace_bytes) *workspace_bytes = empty ? 0 : (int64_t)fwd_workspace_bytes(plan, Bsz, L, D, N, dtype);
    return SELSCAN_OK;
}

extern "C" const char *selscan_last_error(void) { return g_err; }

extern "C" int selscan_check_device_error(void *stream)
{
    g_err[0] = '\0';
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "device work");
    int dev = 0, sms = 0;
    int rc = device_info(&dev, &sms);
    if (rc != SELSCAN_OK) return rc;
    unsigned *word = nullptr;
    rc = fault_word(dev, st, &word);
    if (rc != SELSCAN_OK) return rc;
    unsigned fault = 0;
    e = cudaMemcpyAsync(&fault, word, sizeof fault, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "reading the stream's fault word");
    if (fault != 0) {
        e = cudaMemsetAsync(word, 0, sizeof fault, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) return cuda_fail(e, "clearing the stream's fault word");
        const char *what = fault == kFaultTmaTimeout    ? "an input tile never arrived"
                           : fault == kFaultFlagTimeout ? "a chunk carry never appeared"
                           : fault == 3                 ? "a tensor-core product never completed"
                                                        : "unknown";
        return fail(SELSCAN_ERR_TIMEOUT, "a kernel gave up waiting (fault code %u: %s)", fault, what);
    }
    return SELSCAN_OK;
}

extern "C" int selscan_test_fault_injection(int withhold_carries, int wait_limit_ms)
{
    g_err[0] = '\0';
    if (withhold_carries < 0 || wait_limit_ms < 0 || (uint64_t)wait_limit_ms > kWaitLimitNs / 1000000ull)
        return fail(SELSCAN_ERR_INVALID_ARG, "withhold_carries must be 0 or 1 and wait_limit_ms in 0..%llu",
                    (unsigned long long)(kWaitLimitNs / 1000000ull));
    std::lock_guard<std::mutex> lk(g_test_mu);
    g_test_withhold = withhold_carries ? 1 : 0;
    g_test_wait_ms = wait_limit_ms;
    return SELSCAN_OK;
}

extern "C" void selscan_release_workspace(void)
{
    std::lock_guard<std::mutex> lk(g_mu);
    for (int i = 0; i < kMaxDevices; ++i)
        if (g_pool[i]) cudaMemPoolTrimTo(g_pool[i], 0);
}

extern "C" const char *selscan_version(void) { return "libselscan 0.1.0 (sm_103a)"; }
