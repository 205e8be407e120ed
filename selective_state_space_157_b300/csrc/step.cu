// step.cu -- the decode step kernels (scan_step.cuh) and their launcher.
#include "host_common.h"
#include "launch.h"

namespace selscan {
namespace {

// A launch that may start while the kernel before it on the stream drains
// (the kernel waits for it in its first instruction).
template <typename K>
cudaError_t launch_dependent(K kernel, unsigned blocks, cudaStream_t st, const StepArgs &a)
{
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(kStepThreads);
    cfg.stream = st;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

} // namespace

int launch_step_kernel(const StepArgs &a, int G, int V, bool vec, bool zoh, cudaStream_t st)
{
    const int64_t chains = a.Bsz * a.D;
    if (vec) {
        const int64_t blocks = (chains * G + kStepThreads - 1) / kStepThreads;
        if (blocks > 0x7fffffffLL) return fail(SELSCAN_ERR_UNSUPPORTED, "grid too large");
        const unsigned nb = (unsigned)blocks;
        cudaError_t le = cudaSuccess;
#define SELSCAN_STEP_CASE(g, v) \
        if (G == g && V == v) { \
            le = zoh ? launch_dependent(step_vec_kernel<g, v, true>, nb, st, a) \
                     : launch_dependent(step_vec_kernel<g, v, false>, nb, st, a); \
        }
        SELSCAN_STEP_CASE(1, 1) else SELSCAN_STEP_CASE(2, 1) else SELSCAN_STEP_CASE(4, 1)
        else SELSCAN_STEP_CASE(8, 1) else SELSCAN_STEP_CASE(16, 1)
        else SELSCAN_STEP_CASE(1, 2) else SELSCAN_STEP_CASE(2, 2) else SELSCAN_STEP_CASE(4, 2)
        else SELSCAN_STEP_CASE(8, 2) else SELSCAN_STEP_CASE(1, 4) else SELSCAN_STEP_CASE(2, 4)
        else SELSCAN_STEP_CASE(4, 4)
        else return fail(SELSCAN_ERR_UNSUPPORTED, "no decode kernel for G=%d V=%d", G, V);
#undef SELSCAN_STEP_CASE
        if (le != cudaSuccess) return cuda_fail(le, "kernel launch");
    } else {
        const int64_t blocks = (chains + kStepThreads - 1) / kStepThreads;
        if (blocks > 0x7fffffffLL) return fail(SELSCAN_ERR_UNSUPPORTED, "grid too large");
        if (zoh) step_scalar_kernel<true><<<(unsigned)blocks, kStepThreads, 0, st>>>(a);
        else step_scalar_kernel<false><<<(unsigned)blocks, kStepThreads, 0, st>>>(a);
    }
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SELSCAN_OK : cuda_fail(e, "kernel launch");
}

} // namespace selscan
