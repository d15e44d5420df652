// Staged (long-row) variants of OpLnBwd for f32 storage (one translation unit per
// operation and storage type so they compile in parallel).
#include "rr_instantiate.cuh"

namespace rr {
KernelSet lnbwd_kernels_f32() { return make_kernel_set<OpLnBwd, kF32, 3, 8, 512, 5, 18, 512, false>(); }
const void* col_reduce_kernel_ptr_f32() { return (const void*)col_reduce_kernel<kF32>; }
}  // namespace rr
