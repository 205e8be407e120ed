// conv1d.cu -- the causal depthwise convolution kernels (conv1d.cuh) and
// their launchers.
#include "host_common.h"
#include "launch.h"

namespace selscan {
namespace {

template <typename T>
int launch_conv1d_ring(const ConvArgs &a, int64_t K, cudaStream_t st)
{
    int dev = 0, sms = 0;
    const int rc = device_info(&dev, &sms);
    if (rc != SELSCAN_OK) return rc;
    // Segments of equal length, enough for about kConvRingPerSm CTAs on
    // every SM.
    const int64_t cols = (a.D / 4 + kConvThreads - 1) / kConvThreads;
    const int64_t want = (int64_t)sms * kConvRingPerSm;
    const int64_t nseg0 = (want + cols * a.Bsz - 1) / (cols * a.Bsz);
    int64_t seg = (a.L + nseg0 - 1) / nseg0;
    if (seg < (a.L + 65534) / 65535) seg = (a.L + 65534) / 65535;
    // A programmatic dependent of the kernel before it on the stream (the
    // kernel waits for it first thing).
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cols, (unsigned)a.Bsz, (unsigned)((a.L + seg - 1) / seg));
    cfg.blockDim = dim3(kConvThreads);
    cfg.stream = st;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    cudaError_t e;
    switch (K) {
    case 1: e = cudaLaunchKernelEx(&cfg, conv1d_ring_kernel<T, 1>, a, seg); break;
    case 2: e = cudaLaunchKernelEx(&cfg, conv1d_ring_kernel<T, 2>, a, seg); break;
    case 3: e = cudaLaunchKernelEx(&cfg, conv1d_ring_kernel<T, 3>, a, seg); break;
    case 4: e = cudaLaunchKernelEx(&cfg, conv1d_ring_kernel<T, 4>, a, seg); break;
    case 5: e = cudaLaunchKernelEx(&cfg, conv1d_ring_kernel<T, 5>, a, seg); break;
    case 6: e = cudaLaunchKernelEx(&cfg, conv1d_ring_kernel<T, 6>, a, seg); break;
    case 7: e = cudaLaunchKernelEx(&cfg, conv1d_ring_kernel<T, 7>, a, seg); break;
    default: e = cudaLaunchKernelEx(&cfg, conv1d_ring_kernel<T, 8>, a, seg); break;
    }
    return e == cudaSuccess ? SELSCAN_OK : cuda_fail(e, "kernel launch");
}

template <typename T>
int launch_conv1d_t(const ConvArgs &a, int64_t K, bool vec, cudaStream_t st)
{
    if (vec) {
        const int rc = launch_conv1d_ring<T>(a, K, st);
        if (rc != SELSCAN_OK) return rc;
    } else {
        const dim3 grid((unsigned)((a.D + kConvThreads - 1) / kConvThreads), (unsigned)a.Bsz,
                        (unsigned)((a.L + kConvT - 1) / kConvT));
        switch (K) {
        case 1: conv1d_kernel<T, 1><<<grid, kConvThreads, 0, st>>>(a); break;
        case 2: conv1d_kernel<T, 2><<<grid, kConvThreads, 0, st>>>(a); break;
        case 3: conv1d_kernel<T, 3><<<grid, kConvThreads, 0, st>>>(a); break;
        case 4: conv1d_kernel<T, 4><<<grid, kConvThreads, 0, st>>>(a); break;
        case 5: conv1d_kernel<T, 5><<<grid, kConvThreads, 0, st>>>(a); break;
        case 6: conv1d_kernel<T, 6><<<grid, kConvThreads, 0, st>>>(a); break;
        case 7: conv1d_kernel<T, 7><<<grid, kConvThreads, 0, st>>>(a); break;
        default: conv1d_kernel<T, 8><<<grid, kConvThreads, 0, st>>>(a); break;
        }
    }
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SELSCAN_OK : cuda_fail(e, "kernel launch");
}

} // namespace

int launch_conv1d_kernel(const ConvArgs &a, int64_t K, int dtype, bool vec, cudaStream_t st)
{
    return dtype == SELSCAN_F32 ? launch_conv1d_t<float>(a, K, vec, st)
                                : launch_conv1d_t<__nv_bfloat16>(a, K, vec, st);
}

int launch_conv1d_step_kernel(const ConvStepArgs &a, int64_t K, cudaStream_t st)
{
    const int64_t blocks = (a.Bsz * a.D + kConvThreads - 1) / kConvThreads;
    if (blocks > 0x7fffffffLL) return fail(SELSCAN_ERR_UNSUPPORTED, "grid too large");
    const unsigned nb = (unsigned)blocks;
    switch (K) {
    case 1: conv1d_step_kernel<1><<<nb, kConvThreads, 0, st>>>(a); break;
    case 2: conv1d_step_kernel<2><<<nb, kConvThreads, 0, st>>>(a); break;
    case 3: conv1d_step_kernel<3><<<nb, kConvThreads, 0, st>>>(a); break;
    case 4: conv1d_step_kernel<4><<<nb, kConvThreads, 0, st>>>(a); break;
    case 5: conv1d_step_kernel<5><<<nb, kConvThreads, 0, st>>>(a); break;
    case 6: conv1d_step_kernel<6><<<nb, kConvThreads, 0, st>>>(a); break;
    case 7: conv1d_step_kernel<7><<<nb, kConvThreads, 0, st>>>(a); break;
    default: conv1d_step_kernel<8><<<nb, kConvThreads, 0, st>>>(a); break;
    }
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SELSCAN_OK : cuda_fail(e, "kernel launch");
}

} // namespace selscan
