// host_mem.cu -- page-locked host buffers for the host-buffer entry points
// (selscan_fwd_host and friends): anonymous mappings aligned to 2 MB (with
// transparent huge pages asked for), registered with the CUDA driver.
#include "selscan.h"

#include <cuda_runtime.h>
#include <sys/mman.h>

#include <map>
#include <mutex>
#include <utility>

#include "host_common.h"

using namespace selscan;

namespace {
constexpr size_t kHostAlign = (size_t)2 << 20;
std::mutex g_host_mu;
std::map<void *, std::pair<void *, size_t>> g_host_blocks;   // aligned start -> (mapping, length)
} // namespace

extern "C" void *selscan_host_alloc(size_t bytes)
{
    g_err[0] = '\0';
    if (bytes == 0 || bytes > ((size_t)1 << 46)) {
        fail(SELSCAN_ERR_INVALID_ARG, "selscan_host_alloc: %zu bytes", bytes);
        return nullptr;
    }
    const size_t len = (bytes + kHostAlign - 1) / kHostAlign * kHostAlign;
    const size_t total = len + kHostAlign;
    void *raw = mmap(nullptr, total, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS, -1, 0);
    if (raw == MAP_FAILED) {
        fail(SELSCAN_ERR_NO_MEMORY, "selscan_host_alloc: mapping %zu bytes failed", total);
        return nullptr;
    }
    void *p = reinterpret_cast<void *>((reinterpret_cast<uintptr_t>(raw) + kHostAlign - 1) & ~(uintptr_t)(kHostAlign - 1));
    madvise(p, len, MADV_HUGEPAGE);   // best effort: fewer pages for the DMA engines to translate
    const cudaError_t e = cudaHostRegister(p, len, cudaHostRegisterPortable);
    if (e != cudaSuccess) {
        cudaGetLastError();
        munmap(raw, total);
        cuda_fail(e, "selscan_host_alloc: cudaHostRegister");
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(g_host_mu);
    g_host_blocks[p] = {raw, total};
    return p;
}

extern "C" int selscan_host_free(void *p)
{
    g_err[0] = '\0';
    if (!p) return SELSCAN_OK;
    std::pair<void *, size_t> m;
    {
        std::lock_guard<std::mutex> lk(g_host_mu);
        auto it = g_host_blocks.find(p);
        if (it == g_host_blocks.end())
            return fail(SELSCAN_ERR_INVALID_ARG, "selscan_host_free: %p did not come from selscan_host_alloc", p);
        m = it->second;
        g_host_blocks.erase(it);
    }
    const cudaError_t e = cudaHostUnregister(p);
    munmap(m.first, m.second);
    return e == cudaSuccess ? SELSCAN_OK : cuda_fail(e, "selscan_host_free: cudaHostUnregister");
}
