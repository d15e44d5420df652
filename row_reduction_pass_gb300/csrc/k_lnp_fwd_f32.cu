// Pipelined long-row LayerNorm / RMSNorm forward variants for f32 storage
// (one translation unit per direction and storage type so they compile in
// parallel).
#include "rr_lnp.cuh"

namespace rr {
LnpKernels lnp_fwd_kernels_f32() { return make_lnp_fwd_set<kF32>(); }
}  // namespace rr
