// Phase-aligned LayerNorm / RMSNorm backward variants for f32 storage.
#include "rr_lnx.cuh"

namespace rr {
LnxKernels lnx_bwd_kernels_f32() { return make_lnx_bwd_set<kF32, 4>(); }
}  // namespace rr
