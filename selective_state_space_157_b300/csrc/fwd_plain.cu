// fwd_plain.cu -- the plain-load forward path: scan_chunk_kernel (aggregate
// and readout roles, scan_fwd.cuh) and the carry composition between them.
// Used when TMA's alignment rules do not hold for a call's tensors.
#include "host_common.h"
#include "launch.h"

namespace selscan {
namespace {

// Step 2: compose chunk pairs in order. One thread per (b, d, n); the K-1
// aggregates are replaced in place by the incoming states of chunks 1..K-1.
struct CarryArgs {
    const float *A;
    const float *h0;   // (Bsz, D, N) or null
    float *agg_h;      // (K-1, Bsz, D, N) in: end states from zero; out: incoming states
    const float *agg_s;
    int64_t Bsz, D, N;
    int K;
};

__global__ void __launch_bounds__(256) scan_carry_kernel(const CarryArgs a)
{
    const int64_t total = a.Bsz * a.D * a.N;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= total)
        return;
    const int64_t bd = i / a.N;
    const int64_t n = i - bd * a.N;
    const int64_t d = bd % a.D;
    const float A2 = __ldg(a.A + d * a.N + n) * kLog2e;
    float c = a.h0 ? a.h0[i] : 0.0f;
    const int64_t bdn = total, bdsz = a.Bsz * a.D;
    for (int k = 0; k + 1 < a.K; ++k) {
        const float decay = ex2(A2 * a.agg_s[(int64_t)k * bdsz + bd]);
        float *slot = a.agg_h + (int64_t)k * bdn + i;
        c = fmaf(decay, c, *slot);   // (decay, end) o carry
        *slot = c;                   // incoming state of chunk k+1
    }
}

using ScanKernel = void (*)(ScanArgs);

struct ScanKernels {
    ScanKernel readout, aggregate;
};

template <typename T, int NS, int NSPLIT>
ScanKernels pick_vec(bool vec)
{
    if (vec)
        return {scan_chunk_kernel<T, NS, NSPLIT, true, true>, scan_chunk_kernel<T, NS, NSPLIT, false, true>};
    return {scan_chunk_kernel<T, NS, NSPLIT, true, false>, scan_chunk_kernel<T, NS, NSPLIT, false, false>};
}

template <typename T>
bool pick_shape(int ns, int nsplit, bool vec, ScanKernels *out)
{
    switch (ns * 100 + nsplit) {
    case 401: *out = pick_vec<T, 4, 1>(vec); return true;
    case 801: *out = pick_vec<T, 8, 1>(vec); return true;
    case 1601: *out = pick_vec<T, 16, 1>(vec); return true;
    case 402: *out = pick_vec<T, 4, 2>(vec); return true;
    case 802: *out = pick_vec<T, 8, 2>(vec); return true;
    case 1602: *out = pick_vec<T, 16, 2>(vec); return true;
    case 404: *out = pick_vec<T, 4, 4>(vec); return true;
    case 804: *out = pick_vec<T, 8, 4>(vec); return true;
    case 1604: *out = pick_vec<T, 16, 4>(vec); return true;
    default: return false;
    }
}

} // namespace

int launch_plain_kernels(const ScanArgs &base, int ns, int nsplit, bool vec, int dtype, cudaStream_t st)
{
    ScanKernels ks{};
    const bool ok = dtype == SELSCAN_F32 ? pick_shape<float>(ns, nsplit, vec, &ks)
                                         : pick_shape<__nv_bfloat16>(ns, nsplit, vec, &ks);
    if (!ok) return fail(SELSCAN_ERR_UNSUPPORTED, "no kernel for NS=%d NSPLIT=%d", ns, nsplit);
    const ScanArgs &a = base;
    const int64_t gx = a.Bsz * a.dtiles;
    if (a.K > 1) {
        ks.aggregate<<<dim3((unsigned)gx, (unsigned)(a.K - 1)), kScanThreads, 0, st>>>(a);
        CarryArgs c{a.A, a.h0, a.agg_h, a.agg_s, a.Bsz, a.D, a.N, a.K};
        const int64_t total = a.Bsz * a.D * a.N;
        scan_carry_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(c);
    }
    ks.readout<<<dim3((unsigned)gx, (unsigned)a.K), kScanThreads, 0, st>>>(a);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SELSCAN_OK : cuda_fail(e, "kernel launch");
}

} // namespace selscan
