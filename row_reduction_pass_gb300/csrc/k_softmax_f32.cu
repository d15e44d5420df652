// Kernel variants of OpSoftmaxXent for f32 storage (one translation unit per
// operation and storage type so they compile in parallel).
#include "rr_instantiate.cuh"

namespace rr {
KernelSet softmax_kernels_f32() { return make_kernel_set<OpSoftmaxXent, kF32, 2, 8, 256, 8, 16, 1024>(); }
}  // namespace rr
