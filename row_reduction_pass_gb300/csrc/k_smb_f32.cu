// Long-row softmax / log-softmax backward variants for f32 storage (one
// translation unit per storage type so they compile in parallel).
#include "rr_smb.cuh"

namespace rr {
SmbKernels smb_kernels_f32() { return make_smb_set<kF32>(); }
}  // namespace rr
