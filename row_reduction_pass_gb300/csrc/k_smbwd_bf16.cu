// Kernel variants of OpSoftmaxBwd (softmax and log-softmax backward) for bf16
// storage (one translation unit per operation and storage type so they compile
// in parallel).
#include "rr_instantiate.cuh"

namespace rr {
KernelSet softmax_bwd_kernels_bf16() { return make_kernel_set<OpSoftmaxBwd, kBF16, 2, 8, 256, 4, 8, 1024>(); }
}  // namespace rr
