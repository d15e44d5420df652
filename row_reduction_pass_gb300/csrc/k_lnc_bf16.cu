// Column-block long-row LayerNorm / RMSNorm variants for bf16 storage (one
// translation unit per storage type so they compile in parallel).
#include "rr_lnc.cuh"

namespace rr {
LncKernels lnc_kernels_bf16() { return make_lnc_set<kBF16>(); }
}  // namespace rr
