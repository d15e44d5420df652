// Pipelined long-row LayerNorm / RMSNorm backward variants for bf16 storage
// (2 chunks a thread at most: the column partials stay in registers).
#include "rr_lnp.cuh"

namespace rr {
LnpKernels lnp_bwd_kernels_bf16() { return make_lnp_bwd_set<kBF16, 2>(); }
}  // namespace rr
