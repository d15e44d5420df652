// Phase-aligned softmax / log-softmax / cross-entropy variants for bf16
// storage (one translation unit per storage type so they compile in parallel).
#include "rr_smx.cuh"

namespace rr {
SmxKernels smx_kernels_bf16() { return make_smx_set<kBF16, 12>(); }
}  // namespace rr
