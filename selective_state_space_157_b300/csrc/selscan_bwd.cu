// selscan_bwd.cu -- the backward pass: the kernels of scan_bwd.cuh, their
// argument checks, workspace and launches.
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
    return selscan_bwd_gated(x, delta, A, B, C, nullptr, nullptr, h0, dy, dhT, dx, ddelta, dA, dB, dC, nullptr,
                             nullptr, dh0, Bsz, L, D, N, delta_softplus, stream);
}

extern "C" int selscan_bwd_gated(const float *x, const float *delta, const float *A, const float *B,
                                 const float *C, const float *Dskip, const float *z, const float *h0,
                                 const float *dy, const float *dhT, float *dx, float *ddelta, float *dA,
                                 float *dB, float *dC, float *dDskip, float *dz, float *dh0, int64_t Bsz,
                                 int64_t L, int64_t D, int64_t N, int delta_softplus, void *stream)
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
    if ((Dskip && !dDskip) || (!Dskip && dDskip) || (z && !dz) || (!z && dz))
        return fail(SELSCAN_ERR_INVALID_ARG, "dDskip goes with Dskip and dz with z: both or neither");
    if (Bsz > 0 && L > 0 && (!x || !delta || !B || !C || !dy || !dx || !ddelta || !dB || !dC))
        return fail(SELSCAN_ERR_INVALID_ARG, "x, delta, B, C, dy, dx, ddelta, dB, dC must be non-NULL when L > 0");
    const void *ptrs[] = {x, delta, A, B, C, h0, dy, dhT, dx, ddelta, dA, dB, dC, dh0, Dskip, z, dDskip, dz};
    for (const void *p : ptrs)
        if (!aligned(p, 4))
            return fail(SELSCAN_ERR_INVALID_ARG, "every pointer must be 4-byte aligned");
    const int64_t lb = L > 0 ? nld * 4 : 0, ln = L > 0 ? nln * 4 : 0;
    const Range ins[] = {range(x, lb, "x"), range(delta, lb, "delta"), range(A, D * N * 4, "A"),
                         range(B, ln, "B"), range(C, ln, "C"), range(h0, ndn * 4, "h0"),
                         range(dy, lb, "dy"), range(dhT, ndn * 4, "dhT"), range(Dskip, D * 4, "Dskip"),
                         range(z, lb, "z")};
    const Range outs[] = {range(dx, lb, "dx"), range(ddelta, lb, "ddelta"), range(dA, D * N * 4, "dA"),
                          range(dB, ln, "dB"), range(dC, ln, "dC"), range(dh0, ndn * 4, "dh0"),
                          range(dDskip, D * 4, "dDskip"), range(dz, lb, "dz")};
    for (size_t i = 0; i < sizeof outs / sizeof outs[0]; ++i) {
        for (const Range &r : ins)
            if (overlaps(outs[i], r))
                return fail(SELSCAN_ERR_INVALID_ARG, "%s overlaps %s", outs[i].name, r.name);
        for (size_t j = 0; j < i; ++j)
            if (overlaps(outs[i], outs[j]))
                return fail(SELSCAN_ERR_INVALID_ARG, "%s overlaps %s", outs[i].name, outs[j].name);
    }

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (Bsz == 0 || L == 0) {   // no kernel runs: dA (and dDskip) are zero
        e = cudaMemsetAsync(dA, 0, (size_t)(D * N) * 4, st);
        if (e == cudaSuccess && dDskip) e = cudaMemsetAsync(dDskip, 0, (size_t)D * 4, st);
        if (e != cudaSuccess) return cuda_fail(e, "dA zero fill");
    }
    if (Bsz == 0) return SELSCAN_OK;
    if (L == 0) {
        if (!dh0) return SELSCAN_OK;
        e = dhT ? cudaMemcpyAsync(dh0, dhT, (size_t)ndn * 4, cudaMemcpyDeviceToDevice, st)
                : cudaMemsetAsync(dh0, 0, (size_t)ndn * 4, st);
        return e == cudaSuccess ? SELSCAN_OK : cuda_fail(e, "L == 0 state gradient");
    }
    // With L > 0 the local kernel zeroes dA, dB, dC (and dDskip) itself.

    int dev = 0, sms = 0;
    int rc = device_info(&dev, &sms);
    if (rc != SELSCAN_OK) return rc;
    int P = 1;
    while (P * kBwdS < N) P <<= 1;
    const int per_sm = bwd_prepare(P, Dskip != nullptr || z != nullptr);
    if (per_sm <= 0) {
        cudaGetLastError();
        return fail(SELSCAN_ERR_CUDA, "backward kernels: shared-memory limit or occupancy query failed");
    }
    const BwdShape shape = bwd_shape(Bsz, L, D, N, sms * per_sm);
    if (shape.gx > 0x7fffffffLL) return fail(SELSCAN_ERR_UNSUPPORTED, "grid too large");

    // Workspace: checkpoints (Bsz, nch, D, NP) and their sums of dl
    // (Bsz, nch, D); per segment hl, gl (Bsz, K, D, NP) and the sum of dl
    // (Bsz, K, D). Each array starts on a 256-byte boundary.
    int64_t ck, sp, seg, sdl;
    if (!mul_ok(Bsz * shape.nch, D, shape.NP, &ck) || !mul_ok(Bsz, shape.nch, D, &sp) ||
        !mul_ok(Bsz * shape.K, D, shape.NP, &seg) || !mul_ok(Bsz, shape.K, D, &sdl))
        return fail(SELSCAN_ERR_INVALID_ARG, "backward workspace size overflows");
    auto up = [](int64_t floats) { return ((size_t)floats * 4 + 255) & ~(size_t)255; };
    const size_t total = up(ck) + up(sp) + 2 * up(seg) + up(sdl);
    cudaMemPool_t pool = nullptr;
    rc = workspace_pool(dev, &pool);
    if (rc != SELSCAN_OK) return rc;
    void *ws = nullptr;
    e = cudaMallocFromPoolAsync(&ws, total, pool, st);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(SELSCAN_ERR_NO_MEMORY, "backward workspace of %zu bytes: %s", total, cudaGetErrorString(e));
    }
    BwdArgs a;
    memset(&a, 0, sizeof a);
    a.x = x; a.delta = delta; a.A = A; a.B = B; a.C = C; a.h0 = h0; a.gy = dy; a.ghT = dhT;
    a.dx = dx; a.ddelta = ddelta; a.dA = dA; a.dB = dB; a.dC = dC; a.dh0 = dh0;
    a.Dskip = Dskip; a.z = z; a.dDskip = dDskip; a.dz = dz;
    char *w = static_cast<char *>(ws);
    a.ckpt = reinterpret_cast<float *>(w); w += up(ck);
    a.spre = reinterpret_cast<float *>(w); w += up(sp);
    a.hl = reinterpret_cast<float *>(w); w += up(seg);
    a.gl = reinterpret_cast<float *>(w); w += up(seg);
    a.sdl = reinterpret_cast<float *>(w);
    a.Bsz = Bsz; a.L = L; a.D = D; a.N = N;
    a.softplus = delta_softplus ? 1 : 0;
    e = launch_scan_bwd(a, shape, st);
    cudaFreeAsync(ws, st);
    return e == cudaSuccess ? SELSCAN_OK : cuda_fail(e, "backward kernel launch");
}
