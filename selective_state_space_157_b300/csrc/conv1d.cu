// conv1d.cu -- the causal depthwise convolution kernels (conv1d.cuh) and
// their launchers.
#include "host_common.h"
#include "launch.h"

namespace selscan {
namespace {

template <typename T, int RUN>
void launch_conv1d_vec(const ConvArgs &a, int64_t K, cudaStream_t st)
{
    const dim3 grid((unsigned)((a.D / 4 + kConvThreads - 1) / kConvThreads), (unsigned)a.Bsz,
                    (unsigned)((a.L + RUN - 1) / RUN));
    switch (K) {
    case 1: conv1d_vec_kernel<T, 1, RUN><<<grid, kConvThreads, 0, st>>>(a); break;
    case 2: conv1d_vec_kernel<T, 2, RUN><<<grid, kConvThreads, 0, st>>>(a); break;
    case 3: conv1d_vec_kernel<T, 3, RUN><<<grid, kConvThreads, 0, st>>>(a); break;
    case 4: conv1d_vec_kernel<T, 4, RUN><<<grid, kConvThreads, 0, st>>>(a); break;
    case 5: conv1d_vec_kernel<T, 5, RUN><<<grid, kConvThreads, 0, st>>>(a); break;
    case 6: conv1d_vec_kernel<T, 6, RUN><<<grid, kConvThreads, 0, st>>>(a); break;
    case 7: conv1d_vec_kernel<T, 7, RUN><<<grid, kConvThreads, 0, st>>>(a); break;
    default: conv1d_vec_kernel<T, 8, RUN><<<grid, kConvThreads, 0, st>>>(a); break;
    }
}

template <typename T>
int launch_conv1d_t(const ConvArgs &a, int64_t K, bool vec, cudaStream_t st)
{
    if (vec) {
        launch_conv1d_vec<T, kConvVecRun>(a, K, st);
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
