// Pipelined long-row LayerNorm / RMSNorm backward variants for f32 storage
// (4 chunks a thread at most: the column partials stay in registers).
#include "rr_lnp.cuh"

namespace rr {
LnpKernels lnp_bwd_kernels_f32() { return make_lnp_bwd_set<kF32, 4>(); }
}  // namespace rr
