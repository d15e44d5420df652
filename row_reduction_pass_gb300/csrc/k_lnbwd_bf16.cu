// Staged (long-row) variants of OpLnBwd for bf16 storage (one translation unit per
// operation and storage type so they compile in parallel).
#include "rr_instantiate.cuh"

namespace rr {
KernelSet lnbwd_kernels_bf16() { return make_kernel_set<OpLnBwd, kBF16, 2, 8, 512, 5, 18, 512, false>(); }
const void* col_reduce_kernel_ptr_bf16() { return (const void*)col_reduce_kernel<kBF16>; }
}  // namespace rr
