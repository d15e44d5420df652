// Column-block long-row LayerNorm / RMSNorm variants for f32 storage (one
// translation unit per storage type so they compile in parallel).
#include "rr_lnc.cuh"

namespace rr {
LncKernels lnc_kernels_f32() { return make_lnc_set<kF32>(); }
}  // namespace rr
