// Row-group RMSNorm bwd variants for f32 storage (one translation unit per
// operation and storage type so they compile in parallel).
#include "rr_ln.cuh"

namespace rr {
LnKernelSet rms_bwd_rowgroup_kernels_f32() { return make_ln_set<kF32, false, 4, 16, true, 8>(); }
}  // namespace rr
