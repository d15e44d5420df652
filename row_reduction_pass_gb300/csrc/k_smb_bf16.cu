// Long-row softmax / log-softmax backward variants for bf16 storage (one
// translation unit per storage type so they compile in parallel).
#include "rr_smb.cuh"

namespace rr {
SmbKernels smb_kernels_bf16() { return make_smb_set<kBF16>(); }
}  // namespace rr
