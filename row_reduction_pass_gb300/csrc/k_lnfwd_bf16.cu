// Staged (long-row) variants of OpLnFwd for bf16 storage (one translation unit per
// operation and storage type so they compile in parallel).
#include "rr_instantiate.cuh"

namespace rr {
KernelSet lnfwd_kernels_bf16() { return make_kernel_set<OpLnFwd, kBF16, 4, 8, 256, 8, 18, 512, false>(); }
}  // namespace rr
