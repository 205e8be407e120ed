// host_common.h -- host-side helpers shared by the library's translation
// units: the thread-local error message, argument-check helpers, per-device
// information, the stream-ordered workspace pool and the per-stream device
// fault words. Defined in selscan.cu.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "selscan.h"

namespace selscan {

extern thread_local char g_err[512];

// Records a message for selscan_last_error() and returns `code`.
int fail(int code, const char *fmt, ...);
// SELSCAN_ERR_CUDA with the CUDA error's name and text.
int cuda_fail(cudaError_t e, const char *what);

constexpr int64_t kMaxElems = int64_t(1) << 60;
constexpr int kMaxDevices = 64;

// a * b * c without overflow (false if the product exceeds kMaxElems).
inline bool mul_ok(int64_t a, int64_t b, int64_t c, int64_t *out)
{
    if (a == 0 || b == 0 || c == 0) { *out = 0; return true; }
    if (a > kMaxElems / b) return false;
    const int64_t ab = a * b;
    if (ab > kMaxElems / c) return false;
    *out = ab * c;
    return true;
}

struct Range {
    uintptr_t lo, hi;   // [lo, hi)
    const char *name;
};

inline Range range(const void *p, int64_t bytes, const char *name)
{
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Range{lo, p ? lo + (uintptr_t)bytes : lo, name};
}

inline bool overlaps(const Range &a, const Range &b)
{
    if (a.lo == a.hi || b.lo == b.hi) return false;
    return a.lo < b.hi && b.lo < a.hi;
}

inline bool aligned(const void *p, size_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

// Integer value of an environment variable (tuning knobs), or dflt.
long env_long(const char *name, long dflt);

// The current device and its SM count.
int device_info(int *dev, int *sms);

// The library's stream-ordered workspace pool of a device.
int workspace_pool(int dev, cudaMemPool_t *pool);

// The device fault word that kernels enqueued on `st` record their waits'
// timeouts in (one word per stream, up to kFaultSlots streams per device;
// further streams share the last word). Looked up with the device current.
int fault_word(int dev, cudaStream_t st, unsigned **out);

} // namespace selscan
