// Short-row span variants of softmax, log-softmax, cross-entropy and the
// softmax / log-softmax backward, and the LayerNorm / RMSNorm forward and
// backward (fp32 and bf16 storage).
#include "rr_span.cuh"

namespace rr {
SpanKernelSet span_kernels() {
  SpanKernelSet s{};
  s.k[0][0] = (const void*)span_softmax_kernel<kF32, 0>;
  s.k[0][1] = (const void*)span_softmax_kernel<kF32, 1>;
  s.k[0][2] = (const void*)span_softmax_kernel<kF32, 2>;
  s.k[1][0] = (const void*)span_softmax_kernel<kBF16, 0>;
  s.k[1][1] = (const void*)span_softmax_kernel<kBF16, 1>;
  s.k[1][2] = (const void*)span_softmax_kernel<kBF16, 2>;
  s.k[0][3] = (const void*)span_softmax_bwd_kernel<kF32, false>;
  s.k[0][4] = (const void*)span_softmax_bwd_kernel<kF32, true>;
  s.k[1][3] = (const void*)span_softmax_bwd_kernel<kBF16, false>;
  s.k[1][4] = (const void*)span_softmax_bwd_kernel<kBF16, true>;
  s.k[0][5] = (const void*)span_ln_fwd_kernel<kF32, false>;
  s.k[0][6] = (const void*)span_ln_fwd_kernel<kF32, true>;
  s.k[1][5] = (const void*)span_ln_fwd_kernel<kBF16, false>;
  s.k[1][6] = (const void*)span_ln_fwd_kernel<kBF16, true>;
  s.k[0][7] = (const void*)span_ln_bwd_kernel<kF32, false>;
  s.k[0][8] = (const void*)span_ln_bwd_kernel<kF32, true>;
  s.k[1][7] = (const void*)span_ln_bwd_kernel<kBF16, false>;
  s.k[1][8] = (const void*)span_ln_bwd_kernel<kBF16, true>;
  return s;
}
}  // namespace rr
