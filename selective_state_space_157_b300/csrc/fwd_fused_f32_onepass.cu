// fwd_fused_f32_onepass.cu -- the persistent forward kernel for fp32 tensors,
// one-pass form.
#include "fwd_fused_impl.cuh"

namespace selscan {

bool pick_fused_f32_onepass(int ns, int nsplit, bool vec, bool softplus, bool gate, bool zoh, int64_t N, int stages,
                            FusedLaunch *out)
{
    return pick_fused<float, false>(ns, nsplit, vec, softplus, gate, zoh, N, stages, out);
}

} // namespace selscan
