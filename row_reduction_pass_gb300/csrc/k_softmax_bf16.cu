// Kernel variants of OpSoftmaxXent for bf16 storage (one translation unit per
// operation and storage type so they compile in parallel).
#include "rr_instantiate.cuh"

namespace rr {
KernelSet softmax_kernels_bf16() { return make_kernel_set<OpSoftmaxXent, kBF16, 2, 8, 256, 8, 16, 1024>(); }
}  // namespace rr
