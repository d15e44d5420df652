// Pipelined long-row LayerNorm / RMSNorm forward variants for bf16 storage
// (one translation unit per direction and storage type so they compile in
// parallel).
#include "rr_lnp.cuh"

namespace rr {
LnpKernels lnp_fwd_kernels_bf16() { return make_lnp_fwd_set<kBF16>(); }
}  // namespace rr
