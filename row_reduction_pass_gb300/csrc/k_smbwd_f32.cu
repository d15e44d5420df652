// Kernel variants of OpSoftmaxBwd (softmax and log-softmax backward) for f32
// storage (one translation unit per operation and storage type so they compile
// in parallel).
#include "rr_instantiate.cuh"

namespace rr {
KernelSet softmax_bwd_kernels_f32() { return make_kernel_set<OpSoftmaxBwd, kF32, 2, 8, 256, 4, 8, 1024>(); }
}  // namespace rr
