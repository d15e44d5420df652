// Row-group RMSNorm bwd variants for bf16 storage (one translation unit per
// operation and storage type so they compile in parallel).
#include "rr_ln.cuh"

namespace rr {
LnKernelSet rms_bwd_rowgroup_kernels_bf16() { return make_ln_set<kBF16, false, 2, 16, true, 8>(); }
}  // namespace rr
