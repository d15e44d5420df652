// Phase-aligned LayerNorm / RMSNorm forward variants for f32 storage (one
// translation unit per direction and storage type so they compile in parallel).
#include "rr_lnx.cuh"

namespace rr {
LnxKernels lnx_fwd_kernels_f32() { return make_lnx_fwd_set<kF32, 16>(); }
}  // namespace rr
