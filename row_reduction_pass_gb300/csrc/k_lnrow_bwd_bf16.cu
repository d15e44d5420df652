// Row-group LayerNorm bwd variants for bf16 storage (one translation unit per
// operation and storage type so they compile in parallel).
#include "rr_ln.cuh"

namespace rr {
LnKernelSet ln_bwd_rowgroup_kernels_bf16() { return make_ln_set<kBF16, false, 2, 8, false, 8>(); }
}  // namespace rr
