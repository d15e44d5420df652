// Phase-aligned softmax / log-softmax / cross-entropy variants for f32
// storage (one translation unit per storage type so they compile in parallel).
#include "rr_smx.cuh"

namespace rr {
SmxKernels smx_kernels_f32() { return make_smx_set<kF32, 12>(); }
}  // namespace rr
