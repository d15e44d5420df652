// Kernel variants of OpLnBwd for f32 storage (one translation unit per
// operation and storage type so they compile in parallel).
#include "rr_instantiate.cuh"

namespace rr {
KernelSet lnbwd_kernels_f32() { return make_kernel_set<OpLnBwd, kF32, 2, 8, 512, 2, 18, 512>(); }
const void* col_reduce_kernel_ptr_f32() { return (const void*)col_reduce_kernel<kF32>; }
}  // namespace rr
