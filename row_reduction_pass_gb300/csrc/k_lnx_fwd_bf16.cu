// Phase-aligned LayerNorm / RMSNorm forward variants for bf16 storage (one
// translation unit per direction and storage type so they compile in parallel).
#include "rr_lnx.cuh"

namespace rr {
LnxKernels lnx_fwd_kernels_bf16() { return make_lnx_fwd_set<kBF16, 8>(); }
}  // namespace rr
