// selscan_bwd.cu -- the backward pass: scan_bwd_kernel (scan_bwd.cuh), its
// argument checks, checkpoint workspace and launch.
#include <cstring>

#include "host_common.h"
#include "scan_bwd.cuh"

using namespace selscan;

extern "C" int selscan_bwd(const float *x, const float *delta, const float *A, const float *B,
                           const float *C, const float *h0, const float *dy, const float *dhT,
                           float *dx, float *ddelta, float *dA, float *dB, float *dC, float *dh0,
                           int64_t Bsz, int64_t L, int64_t D, int64_t N, int delta_softplus,
                           void *stream)
{
    g_err[0] = '\0';
    if (Bsz < 0 || L < 0 || D < 0)
        return fail(SELSCAN_ERR_INVALID_ARG, "negative size (Bsz=%lld L=%lld D=%lld)",
                    (long long)Bsz, (long long)L, (long long)D);
    if (N < 1)
        return fail(SELSCAN_ERR_INVALID_ARG, "N=%lld must be >= 1", (long long)N);
    if (N > 32)
        return fail(SELSCAN_ERR_UNSUPPORTED, "N=%lld: the backward pass takes N <= 32", (long long)N);
    if (Bsz > 65535)
        return fail(SELSCAN_ERR_UNSUPPORTED, "Bsz=%lld exceeds 65535", (long long)Bsz);
    int64_t nld, nln, ndn;
    if (!mul_ok(Bsz, L, D, &nld) || !mul_ok(Bsz, L, N, &nln) || !mul_ok(Bsz, D, N, &ndn))
        return fail(SELSCAN_ERR_INVALID_ARG, "sizes overflow (Bsz=%lld L=%lld D=%lld N=%lld)",
                    (long long)Bsz, (long long)L, (long long)D, (long long)N);
    if (D == 0)
        return SELSCAN_OK;
    if (!A || !dA)
        return fail(SELSCAN_ERR_INVALID_ARG, "A and dA must be non-NULL");
    if (Bsz > 0 && L > 0 && (!x || !delta || !B || !C || !dy || !dx || !ddelta || !dB || !dC))
        return fail(SELSCAN_ERR_INVALID_ARG, "x, delta, B, C, dy, dx, ddelta, dB, dC must be non-NULL when L > 0");
    const void *ptrs[] = {x, delta, A, B, C, h0, dy, dhT, dx, ddelta, dA, dB, dC, dh0};
    for (const void *p : ptrs)
        if (!aligned(p, 4))
            return fail(SELSCAN_ERR_INVALID_ARG, "every pointer must be 4-byte aligned");
    const int64_t lb = L > 0 ? nld * 4 : 0, ln = L > 0 ? nln * 4 : 0;
    const Range ins[] = {range(x, lb, "x"), range(delta, lb, "delta"), range(A, D * N * 4, "A"),
                         range(B, ln, "B"), range(C, ln, "C"), range(h0, ndn * 4, "h0"),
                         range(dy, lb, "dy"), range(dhT, ndn * 4, "dhT")};
    const Range outs[] = {range(dx, lb, "dx"), range(ddelta, lb, "ddelta"), range(dA, D * N * 4, "dA"),
                          range(dB, ln, "dB"), range(dC, ln, "dC"), range(dh0, ndn * 4, "dh0")};
    for (size_t i = 0; i < sizeof outs / sizeof outs[0]; ++i) {
        for (const Range &r : ins)
            if (overlaps(outs[i], r))
                return fail(SELSCAN_ERR_INVALID_ARG, "%s overlaps %s", outs[i].name, r.name);
        for (size_t j = 0; j < i; ++j)
            if (overlaps(outs[i], outs[j]))
                return fail(SELSCAN_ERR_INVALID_ARG, "%s overlaps %s", outs[i].name, outs[j].name);
    }

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(dA, 0, (size_t)(D * N) * 4, st);
    if (e != cudaSuccess) return cuda_fail(e, "dA zero fill");
    if (Bsz == 0) return SELSCAN_OK;
    if (L == 0) {
        if (!dh0) return SELSCAN_OK;
        e = dhT ? cudaMemcpyAsync(dh0, dhT, (size_t)ndn * 4, cudaMemcpyDeviceToDevice, st)
                : cudaMemsetAsync(dh0, 0, (size_t)ndn * 4, st);
        return e == cudaSuccess ? SELSCAN_OK : cuda_fail(e, "L == 0 state gradient");
    }
    if ((e = cudaMemsetAsync(dB, 0, (size_t)nln * 4, st)) != cudaSuccess ||
        (e = cudaMemsetAsync(dC, 0, (size_t)nln * 4, st)) != cudaSuccess)
        return cuda_fail(e, "dB, dC zero fill");

    const BwdShape shape = bwd_shape(L, D, N);
    int64_t ckpt_floats;
    if (!mul_ok(Bsz * shape.nch, D, shape.P, &ckpt_floats))
        return fail(SELSCAN_ERR_INVALID_ARG, "checkpoint workspace size overflows");
    if (shape.gx > 0x7fffffffLL) return fail(SELSCAN_ERR_UNSUPPORTED, "grid too large");

    int dev = 0, sms = 0;
    int rc = device_info(&dev, &sms);
    if (rc != SELSCAN_OK) return rc;
    cudaMemPool_t pool = nullptr;
    rc = workspace_pool(dev, &pool);
    if (rc != SELSCAN_OK) return rc;
    void *ws = nullptr;
    e = cudaMallocFromPoolAsync(&ws, (size_t)ckpt_floats * 4, pool, st);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(SELSCAN_ERR_NO_MEMORY, "checkpoint workspace of %lld bytes: %s", (long long)ckpt_floats * 4,
                    cudaGetErrorString(e));
    }
    BwdArgs a;
    memset(&a, 0, sizeof a);
    a.x = x; a.delta = delta; a.A = A; a.B = B; a.C = C; a.h0 = h0; a.gy = dy; a.ghT = dhT;
    a.dx = dx; a.ddelta = ddelta; a.dA = dA; a.dB = dB; a.dC = dC; a.dh0 = dh0;
    a.ckpt = static_cast<float *>(ws);
    a.Bsz = Bsz; a.L = L; a.D = D; a.N = N;
    a.softplus = delta_softplus ? 1 : 0;
    e = launch_scan_bwd(a, shape, st);
    cudaFreeAsync(ws, st);
    return e == cudaSuccess ? SELSCAN_OK : cuda_fail(e, "backward kernel launch");
}
