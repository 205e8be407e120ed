// alu_peaks.cu -- measures the arithmetic throughputs the selective scan's
// roofline is stated in: base-2 exponentials on the special-function unit
// (ex2.approx.ftz.f32, one per state update) and FP32 fused multiply-adds,
// scalar (fma.rn.f32) and packed (fma.rn.f32x2, two lanes per instruction).
//
// Each kernel runs many independent dependency chains per thread at full
// occupancy, so the pipe, not latency, limits it; the second of two launches
// is timed with CUDA events. Built as its own library (libselscan_probe.so)
// for the benchmark; the scan library does not contain it.
#include <cuda_runtime.h>

#include <cstdint>

namespace {

constexpr int kThreads = 256;
constexpr int kChains = 16;

__device__ __forceinline__ float ex2_neg(float v)
{
    float r;
    asm volatile("{\n\t.reg .f32 t;\n\tneg.f32 t, %1;\n\tex2.approx.ftz.f32 %0, t;\n\t}" : "=f"(r) : "f"(v));
    return r;
}

// v <- 2^-v converges to about 0.64, so the chains stay finite.
__global__ void __launch_bounds__(kThreads) ex2_kernel(float *sink, int iters)
{
    float v[kChains];
#pragma unroll
    for (int i = 0; i < kChains; ++i)
        v[i] = 0.5f + 1e-3f * (float)(threadIdx.x & 31) + 0.01f * (float)i;
    for (int k = 0; k < iters; ++k) {
#pragma unroll
        for (int i = 0; i < kChains; ++i)
            v[i] = ex2_neg(v[i]);
    }
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < kChains; ++i)
        s += v[i];
    if (s == -1.0f)   // never true: keeps the chains live
        sink[blockIdx.x] = s;
}

// v <- v * a + b with |a| < 1 converges, so the chains stay finite.
__global__ void __launch_bounds__(kThreads) ffma_kernel(float *sink, int iters, float a, float b)
{
    float v[kChains];
#pragma unroll
    for (int i = 0; i < kChains; ++i)
        v[i] = 1.0f + 1e-3f * (float)(threadIdx.x & 31) + 0.01f * (float)i;
    for (int k = 0; k < iters; ++k) {
#pragma unroll
        for (int i = 0; i < kChains; ++i)
            v[i] = fmaf(v[i], a, b);
    }
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < kChains; ++i)
        s += v[i];
    if (s == -1.0f)
        sink[blockIdx.x] = s;
}

__global__ void __launch_bounds__(kThreads) ffma2_kernel(float *sink, int iters, float a, float b)
{
    float2 v[kChains / 2];
#pragma unroll
    for (int i = 0; i < kChains / 2; ++i)
        v[i] = make_float2(1.0f + 1e-3f * (float)(threadIdx.x & 31), 1.0f + 0.01f * (float)i);
    const float2 a2 = make_float2(a, a), b2 = make_float2(b, b);
    for (int k = 0; k < iters; ++k) {
#pragma unroll
        for (int i = 0; i < kChains / 2; ++i)
            v[i] = __ffma2_rn(v[i], a2, b2);
    }
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < kChains / 2; ++i)
        s += v[i].x + v[i].y;
    if (s == -1.0f)
        sink[blockIdx.x] = s;
}

template <typename Launch>
int timed(Launch launch, float *ms)
{
    cudaEvent_t e0, e1;
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) return 1;
    launch();   // warm-up (clocks, instruction cache)
    cudaEventRecord(e0);
    launch();
    cudaEventRecord(e1);
    const cudaError_t e = cudaEventSynchronize(e1);
    if (e == cudaSuccess) cudaEventElapsedTime(ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? 0 : 1;
}

} // namespace

// Operations per second on the current device: ex2 results, scalar FMA
// lane-operations and packed FMA lane-operations (two per instruction).
// Returns 0 on success. Takes well under a second on a B300.
extern "C" int selscan_probe_alu_peaks(double *ex2_per_s, double *ffma_per_s, double *ffma2_per_s)
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 1;
    float *sink = nullptr;
    const int blocks = sms * 8;   // 2048 threads per SM
    if (cudaMalloc(&sink, (size_t)blocks * sizeof(float)) != cudaSuccess) return 1;
    const double threads = (double)blocks * kThreads;
    const int it_ex2 = 4096, it_fma = 16384;
    float ms = 0.0f;
    int rc = timed([&] { ex2_kernel<<<blocks, kThreads>>>(sink, it_ex2); }, &ms);
    if (!rc) *ex2_per_s = threads * it_ex2 * kChains / (ms * 1e-3);
    if (!rc) rc = timed([&] { ffma_kernel<<<blocks, kThreads>>>(sink, it_fma, 0.9999f, 1e-4f); }, &ms);
    if (!rc) *ffma_per_s = threads * it_fma * kChains / (ms * 1e-3);
    if (!rc) rc = timed([&] { ffma2_kernel<<<blocks, kThreads>>>(sink, it_fma, 0.9999f, 1e-4f); }, &ms);
    if (!rc) *ffma2_per_s = threads * it_fma * kChains / (ms * 1e-3);
    cudaFree(sink);
    return rc;
}
