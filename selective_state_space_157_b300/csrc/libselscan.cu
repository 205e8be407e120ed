// libselscan.cu -- the library's one translation unit: the forward, decode
// and conv1d entry points with the shared argument checks, error state and
// workspace pool (selscan.cu), then the backward pass (selscan_bwd.cu).
#include "selscan.cu"
#include "selscan_bwd.cu"
