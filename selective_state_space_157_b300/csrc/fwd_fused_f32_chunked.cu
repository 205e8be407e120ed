// fwd_fused_f32_chunked.cu -- the persistent forward kernel for fp32 tensors,
// chunked form (local and correction items).
#include "fwd_fused_impl.cuh"

namespace selscan {

bool pick_fused_f32_chunked(int ns, int nsplit, bool vec, bool softplus, bool gate, bool zoh, int64_t N, int stages,
                            FusedLaunch *out)
{
    return pick_fused<float, true>(ns, nsplit, vec, softplus, gate, zoh, N, stages, out);
}

} // namespace selscan
