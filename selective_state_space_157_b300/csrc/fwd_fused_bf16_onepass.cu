// fwd_fused_bf16_onepass.cu -- the persistent forward kernel for bfloat16
// tensors (fp32 state and arithmetic), one-pass form.
#include "fwd_fused_impl.cuh"

namespace selscan {

bool pick_fused_bf16_onepass(int ns, int nsplit, bool vec, bool softplus, bool gate, bool zoh, int64_t N, int stages,
                             FusedLaunch *out)
{
    return pick_fused<__nv_bfloat16, false>(ns, nsplit, vec, softplus, gate, zoh, N, stages, out);
}

} // namespace selscan
