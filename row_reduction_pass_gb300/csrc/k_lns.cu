// LayerNorm / RMSNorm backward of short misaligned rows by phase class (fp32
// and bf16 storage).
#include "rr_lns.cuh"

namespace rr {
LnsKernels lns_kernels_f32() { return make_lns_set<kF32>(); }
LnsKernels lns_kernels_bf16() { return make_lns_set<kBF16>(); }
}  // namespace rr
