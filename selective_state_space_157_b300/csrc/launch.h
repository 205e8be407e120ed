// launch.h -- what the kernel translation units export to the host code in
// selscan.cu: the forward kernels' launch descriptions and the launchers of
// the plain-load forward, the decode step and the convolution. Each kernel
// family is compiled in its own translation unit (fwd_fused_f32.cu,
// fwd_fused_bf16.cu, fwd_plain.cu, step.cu, conv1d.cu) so the library builds
// in parallel.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "conv1d.cuh"
#include "scan_fused.cuh"
#include "scan_step.cuh"

namespace selscan {

// CTA size of the persistent forward kernel: one pass runs CTAs of 128
// threads (128 / NSPLIT channels each, up to three per SM); the chunked form
// runs one CTA of 384 threads per SM (its launch bounds), so that no item
// waits behind an older CTA on its SM. The planner sizes the chunking by it.
constexpr int kFusedChunkedThreads = 384;
constexpr int kFusedChunkedCtasPerSm = 1;

// CTA size of the fused kernel: chunked plans kFusedChunkedThreads; one pass
// 256 threads (one CTA per SM, 128 channels) with two threads per chain,
// else kScanThreads.
constexpr int fused_threads(bool chunked, int nsplit)
{
    return chunked ? kFusedChunkedThreads : (nsplit == 2 ? 2 * kScanThreads : kScanThreads);
}

// The persistent forward kernel chosen for a problem: launched by the host
// with cudaLaunchKernel(kernel, grid, threads, {&FusedArgs}, smem).
struct FusedLaunch {
    const void *kernel;
    size_t smem;        // dynamic shared memory per CTA
    int ctas_per_sm;    // resident CTAs per SM at that shared-memory size
    int tt, stages;     // timesteps per pipeline stage, ring buffers
    int threads;        // CTA size
    int box_w;          // channels per TMA box of x, delta and z (at most 256)
};

// False when no fused variant fits (the caller then takes the plain path).
// The one-pass form serves plans with one chunk, the chunked form the rest.
bool pick_fused_f32_onepass(int ns, int nsplit, bool vec, bool softplus, bool gate, bool zoh, int64_t N,
                            int stages, FusedLaunch *out);
bool pick_fused_f32_chunked(int ns, int nsplit, bool vec, bool softplus, bool gate, bool zoh, int64_t N,
                            int stages, FusedLaunch *out);
bool pick_fused_bf16_onepass(int ns, int nsplit, bool vec, bool softplus, bool gate, bool zoh, int64_t N,
                             int stages, FusedLaunch *out);
bool pick_fused_bf16_chunked(int ns, int nsplit, bool vec, bool softplus, bool gate, bool zoh, int64_t N,
                             int stages, FusedLaunch *out);

// Plain-load forward: aggregate, carry and readout launches (K > 1), or one
// readout launch. a.chunk, a.K, a.dtiles and, for K > 1, a.agg_h / a.agg_s
// are set by the caller. Returns a selscan_status.
int launch_plain_kernels(const ScanArgs &a, int ns, int nsplit, bool vec, int dtype, cudaStream_t st);

// Decode step: G lanes per chain with V 16-byte groups each (vec), or one
// thread per chain.
int launch_step_kernel(const StepArgs &a, int G, int V, bool vec, bool zoh, cudaStream_t st);

// Causal depthwise convolution (+ SiLU) over a sequence, and its decode step.
int launch_conv1d_kernel(const ConvArgs &a, int64_t K, int dtype, bool vec, cudaStream_t st);
int launch_conv1d_step_kernel(const ConvStepArgs &a, int64_t K, cudaStream_t st);

} // namespace selscan
