// Phase-aligned LayerNorm / RMSNorm backward variants for bf16 storage.
#include "rr_lnx.cuh"

namespace rr {
LnxKernels lnx_bwd_kernels_bf16() { return make_lnx_bwd_set<kBF16, 2>(); }
}  // namespace rr
