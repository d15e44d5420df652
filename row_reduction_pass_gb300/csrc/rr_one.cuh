// rr_one.cuh -- the row operations on rows of one column (C = 1), as plain
// streams over the rows.  A row of one element is its own maximum, sum and
// moments, so every per-row reduction of the softmax family ("Engineering a
// CUDA Machine Learning Framework from Scratch", sec. 3.1) and of the norms
// (sec. 3.2, sec. 2.2) becomes elementwise; the general kernels' per-row
// machinery (row geometry, staging, merges over lanes) cost ~190 thread
// instructions for such a row.  A block takes tiles of kOneThreads x U rows
// (U = 16 bytes / element size; 4 in the norm backward, which reads four
// tensors a row), tiles b, b + grid, ...; thread t of a tile
// takes rows t, t + kOneThreads, ..., its U loads of each tensor issued
// together, so every warp access covers consecutive rows.  Masked rows,
// labels out of range, ignored rows and non-finite values come out as in the
// general kernels:
//   softmax forward family, with m = x the row's maximum (a NaN is not a
//     maximum: a row of -inf or NaN is masked) and d = e^(x - m) = 1, so
//     exactly: softmax y = 1, log-softmax z = (x - m) - ln 1 = 0, and
//     cross-entropy loss = (m - x) + ln 1 = 0 with dlogits = p - 1 = 0 for
//     label 0, loss NaN (counted) and dlogits = p = 1 for a label out of
//     range; written as x - x (+ 1), which is NaN for x = +inf as
//     (x - m) is; masked or ignored rows give 0 everywhere;
//   softmax backward: S = y dy, dx = y (dy - S); log-softmax: S = dz,
//     dx = dz - 2^(z log2 e) S;
//   LayerNorm: mean = x, M2 = 0, rstd = 1 / sqrt(eps), y = ((x - mean) rstd)
//     gamma + beta; a non-finite x masks the row (y = mean = rstd = 0);
//     RMSNorm: rstd = 1 / sqrt(x^2 + eps), y = (x rstd) gamma;
//   norm backward: xhat = (x - mean) rstd, g = dy gamma, dx = rstd ((g - g) -
//     xhat (g xhat)) (RMSNorm: rstd (g - xhat (g xhat))), a row with rstd = 0
//     gives dx = 0; each block sums its rows' dy xhat (and dy) in a fixed order
//     into its partial, which col_reduce_kernel adds up.
#pragma once

#include "rr_kernels.h"
#include "rr_ops.cuh"

namespace rr {

// The rows of the tiles a block takes: for (t0 ...) { rows t0 + u * kOneThreads + tid }.
#define RR_ONE_TILES(U)                                                              \
  const int64_t tile_ = (int64_t)kOneThreads * (U);                                  \
  for (int64_t t0 = (int64_t)blockIdx.x * tile_ + threadIdx.x; t0 < rows;            \
       t0 += (int64_t)gridDim.x * tile_)

// Softmax family forward, MODE 0 softmax, 1 log-softmax, 2 cross-entropy.
template <int DT, int MODE>
__global__ void __launch_bounds__(kOneThreads) one_softmax_kernel(const SoftmaxParams p,
                                                                  int64_t rows) {
  constexpr int E = DType<DT>::E;
  constexpr int U = 16 / E;
  int bad = 0;
  RR_ONE_TILES(U) {
    float x[U];
    int32_t lab[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t r = t0 + u * kOneThreads;
      x[u] = r < rows ? ld_elem<DT>(p.x + r * E) : 0.f;
      if constexpr (MODE == 2) lab[u] = r < rows ? __ldcs(p.labels + r) : 0;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t r = t0 + u * kOneThreads;
      if (r >= rows) break;
      const bool masked = !(x[u] > -INFINITY);  // -inf or NaN
      const float z = x[u] - x[u];               // 0, or NaN for +inf
      float out;
      if constexpr (MODE == 0) {
        out = masked ? 0.f : z + 1.0f;
      } else if constexpr (MODE == 1) {
        out = masked ? 0.f : z;
      } else {
        const bool skip = lab[u] == p.ignore;
        const bool in_range = lab[u] == 0;
        if (!skip && !in_range) ++bad;
        const bool dead = skip || masked;
        out = dead ? 0.f : (in_range ? z : z + 1.0f);
        __stcs(p.loss + r, dead ? 0.f : (in_range ? z : __int_as_float(0x7fc00000)));
      }
      st_elem<DT>(p.y + r * E, out);
    }
  }
  if constexpr (MODE == 2) {
    // labels out of range: one atomic per warp
    const unsigned total = __reduce_add_sync(0xffffffffu, static_cast<unsigned>(bad));
    if ((threadIdx.x & 31) == 0 && total != 0 && p.bad != nullptr) atomicAdd(p.bad, (int)total);
  }
}

// Softmax / log-softmax backward.
template <int DT, bool LOG>
__global__ void __launch_bounds__(kOneThreads) one_softmax_bwd_kernel(const SoftmaxBwdParams p,
                                                                      int64_t rows) {
  constexpr int E = DType<DT>::E;
  constexpr int U = 16 / E;
  RR_ONE_TILES(U) {
    float y[U], dy[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t r = t0 + u * kOneThreads;
      y[u] = r < rows ? ld_elem<DT>(p.y + r * E) : 0.f;
      dy[u] = r < rows ? ld_elem<DT>(p.dy + r * E) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t r = t0 + u * kOneThreads;
      if (r >= rows) break;
      float dx;
      if constexpr (LOG) {
        const float S = 0.f + dy[u];
        dx = fmaf(ex2(y[u] * kLog2e), -S, dy[u]);
      } else {
        const float S = fmaf(y[u], dy[u], 0.f);
        dx = y[u] * (dy[u] - S);
      }
      st_elem<DT>(p.dx + r * E, dx);
    }
  }
}

// LayerNorm / RMSNorm forward (gamma, beta: one element each).
template <int DT, bool RMS>
__global__ void __launch_bounds__(kOneThreads) one_norm_fwd_kernel(const LnFwdParams p,
                                                                   int64_t rows) {
  constexpr int E = DType<DT>::E;
  constexpr int U = 16 / E;
  const float gm = ld_elem<DT>(p.gamma);
  const float bt = RMS ? 0.f : ld_elem<DT>(p.beta);
  RR_ONE_TILES(U) {
    float x[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t r = t0 + u * kOneThreads;
      x[u] = r < rows ? ld_elem<DT>(p.x + r * E) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t r = t0 + u * kOneThreads;
      if (r >= rows) break;
      float y;
      if constexpr (RMS) {
        const float ms = fmaf(x[u], x[u], 0.f) * p.inv_cols;
        const bool masked = !isfinite(ms);
        const float rstd = masked ? 0.f : rsqrtf(ms + p.eps);
        __stcs(p.rstd + r, rstd);
        y = masked ? 0.f : (x[u] * rstd) * gm;
      } else {
        const bool masked = !isfinite(x[u]);
        const float rstd = masked ? 0.f : rsqrtf(0.f * p.inv_cols + p.eps);
        __stcs(p.mean + r, masked ? 0.f : x[u] + 0.f);
        __stcs(p.rstd + r, rstd);
        y = masked ? 0.f : fmaf((x[u] - x[u]) * rstd, gm, bt);
      }
      st_elem<DT>(p.y + r * E, y);
    }
  }
}

// LayerNorm / RMSNorm backward: dx, and the block's partial sums of dy xhat
// (and dy) at p.ws + blockIdx.x * planes.
template <int DT, bool RMS>
__global__ void __launch_bounds__(kOneThreads) one_norm_bwd_kernel(const LnBwdParams p,
                                                                   int64_t rows) {
  constexpr int E = DType<DT>::E;
  constexpr int kPlanes = RMS ? 1 : 2;
  __shared__ float red[kOneThreads / 32][2];
  constexpr int U = 4;  // rows a thread takes per tile (four tensors in flight per row)
  const float gm = ld_elem<DT>(p.gamma);
  float ag = 0.f, ab = 0.f;  // this thread's sums of dy xhat, dy (its rows in order)
  RR_ONE_TILES(U) {
    float x[U], dy[U], mean[U], rstd[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t r = t0 + u * kOneThreads;
      const bool in = r < rows;
      x[u] = in ? ld_elem<DT>(p.x + r * E) : 0.f;
      dy[u] = in ? ld_elem<DT>(p.dy + r * E) : 0.f;
      mean[u] = (in && !RMS) ? __ldcs(p.mean + r) : 0.f;
      rstd[u] = in ? __ldcs(p.rstd + r) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t r = t0 + u * kOneThreads;
      if (r >= rows) break;
      float dx = 0.f;
      if (rstd[u] != 0.f) {  // a masked row adds nothing
        const float h = RMS ? x[u] * rstd[u] : (x[u] - mean[u]) * rstd[u];
        const float g = __fmul_rn(dy[u], gm);
        const float b = fmaf(g, h, 0.f) * p.inv_cols;
        float t = RMS ? g : g - g * p.inv_cols;
        t = fmaf(h, -b, t);
        dx = t * rstd[u];
        ag = fmaf(dy[u], h, ag);
        if constexpr (!RMS) ab += dy[u];
      }
      st_elem<DT>(p.dx + r * E, dx);
    }
  }
  // the block's partial: warps' sums in lane order, then the warps in order
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const float og = __shfl_xor_sync(0xffffffffu, ag, off);
    const float ob = __shfl_xor_sync(0xffffffffu, ab, off);
    const bool lo = ((threadIdx.x & 31) & off) == 0;
    ag = lo ? ag + og : og + ag;
    ab = lo ? ab + ob : ob + ab;
  }
  if ((threadIdx.x & 31) == 0) {
    red[threadIdx.x >> 5][0] = ag;
    red[threadIdx.x >> 5][1] = ab;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float sg = 0.f, sb = 0.f;
    for (int w = 0; w < kOneThreads / 32; ++w) {
      sg += red[w][0];
      sb += red[w][1];
    }
    p.ws[(int64_t)blockIdx.x * kPlanes] = sg;
    if constexpr (!RMS) p.ws[(int64_t)blockIdx.x * kPlanes + 1] = sb;
  }
}

template <int DT>
OneKernels make_one_set() {
  OneKernels s{};
  s.fwd[0] = (const void*)one_softmax_kernel<DT, 0>;
  s.fwd[1] = (const void*)one_softmax_kernel<DT, 1>;
  s.fwd[2] = (const void*)one_softmax_kernel<DT, 2>;
  s.bwd[0] = (const void*)one_softmax_bwd_kernel<DT, false>;
  s.bwd[1] = (const void*)one_softmax_bwd_kernel<DT, true>;
  s.norm_fwd[0] = (const void*)one_norm_fwd_kernel<DT, false>;
  s.norm_fwd[1] = (const void*)one_norm_fwd_kernel<DT, true>;
  s.norm_bwd[0] = (const void*)one_norm_bwd_kernel<DT, false>;
  s.norm_bwd[1] = (const void*)one_norm_bwd_kernel<DT, true>;
  return s;
}

}  // namespace rr
