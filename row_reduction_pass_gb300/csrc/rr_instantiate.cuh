// rr_instantiate.cuh -- builds the KernelSet of one operation / storage type.
#pragma once

#include "rr_kernels.h"
#include "rr_ops.cuh"

namespace rr {

// DIRECT = false: staged variants only (the operation's direct rows go to
// other kernels); the direct table is left empty.
template <template <int, int, int> class OpT, int DT, int NQC, int NQE, int MAXT_D, int NQSC,
          int NQSE, int MAXT_S, bool DIRECT = true>
KernelSet make_kernel_set() {
  constexpr int V = DType<DT>::V;
  using OC = OpT<DT, V, NQC>;
  using OE = OpT<DT, 1, NQE>;
  KernelSet k{};
  if constexpr (DIRECT) {
  k.direct[0][0] = (const void*)row_kernel<OC, 1, NQC, MAXT_D, false>;
  k.direct[0][1] = (const void*)row_kernel<OC, 2, NQC, MAXT_D, false>;
  k.direct[0][2] = (const void*)row_kernel<OC, 4, NQC, MAXT_D, false>;
  k.direct[0][3] = (const void*)row_kernel<OC, 8, NQC, MAXT_D, false>;
  k.direct[0][4] = (const void*)row_kernel<OC, 16, NQC, MAXT_D, false>;
  k.direct[0][5] = (const void*)row_kernel<OC, 32, NQC, MAXT_D, false>;
  k.direct[0][6] = (const void*)row_kernel<OC, 64, NQC, MAXT_D, false>;
  k.direct[0][7] = (const void*)row_kernel<OC, 128, NQC, MAXT_D, false>;
  k.direct[0][8] = (const void*)row_kernel<OC, 256, NQC, MAXT_D, false>;
  k.direct[1][0] = (const void*)row_kernel<OE, 1, NQE, MAXT_D, false>;
  k.direct[1][1] = (const void*)row_kernel<OE, 2, NQE, MAXT_D, false>;
  k.direct[1][2] = (const void*)row_kernel<OE, 4, NQE, MAXT_D, false>;
  k.direct[1][3] = (const void*)row_kernel<OE, 8, NQE, MAXT_D, false>;
  k.direct[1][4] = (const void*)row_kernel<OE, 16, NQE, MAXT_D, false>;
  k.direct[1][5] = (const void*)row_kernel<OE, 32, NQE, MAXT_D, false>;
  k.direct[1][6] = (const void*)row_kernel<OE, 64, NQE, MAXT_D, false>;
  k.direct[1][7] = (const void*)row_kernel<OE, 128, NQE, MAXT_D, false>;
  k.direct[1][8] = (const void*)row_kernel<OE, 256, NQE, MAXT_D, false>;
  // one row per block for the widest groups (the block grows to the group)
  constexpr int T512 = MAXT_D > 512 ? MAXT_D : 512;
  k.direct[0][9] = (const void*)row_kernel<OC, 512, NQC, T512, false>;
  k.direct[0][10] = (const void*)row_kernel<OC, 1024, NQC, 1024, false>;
  k.direct[1][9] = (const void*)row_kernel<OE, 512, NQE, T512, false>;
  k.direct[1][10] = (const void*)row_kernel<OE, 1024, NQE, 1024, false>;
  }
  k.staged[0] = (const void*)row_kernel<OpT<DT, V, NQSC>, MAXT_S, NQSC, MAXT_S, true>;
  k.staged[1] = (const void*)row_kernel<OpT<DT, 1, NQSE>, MAXT_S, NQSE, MAXT_S, true>;
  k.nq_direct[0] = NQC;
  k.nq_direct[1] = NQE;
  k.nq_staged[0] = NQSC;
  k.nq_staged[1] = NQSE;
  k.maxt_direct = MAXT_D;
  k.maxt_staged = MAXT_S;
  return k;
}

}  // namespace rr
