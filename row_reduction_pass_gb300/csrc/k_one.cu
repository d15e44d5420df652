// Rows of one column: the softmax family and the LayerNorm / RMSNorm forward
// and backward as elementwise streams (fp32 and bf16 storage).
#include "rr_one.cuh"

namespace rr {
OneKernels one_kernels_f32() { return make_one_set<kF32>(); }
OneKernels one_kernels_bf16() { return make_one_set<kBF16>(); }
}  // namespace rr
