// Staged (long-row) variants of OpLnFwd for f32 storage (one translation unit per
// operation and storage type so they compile in parallel).
#include "rr_instantiate.cuh"

namespace rr {
KernelSet lnfwd_kernels_f32() { return make_kernel_set<OpLnFwd, kF32, 6, 8, 256, 8, 18, 512, false>(); }
}  // namespace rr
