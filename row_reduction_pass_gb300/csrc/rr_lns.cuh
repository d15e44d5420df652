// rr_lns.cuh -- LayerNorm / RMSNorm backward of short rows whose byte length
// is not a multiple of 16 (65 bytes to 1 KB), by phase class.
//
// The backward of "Engineering a CUDA Machine Learning Framework from
// Scratch", sec. 2.2 (pre-derived analytic gradients), per row:
//   xhat = (x - mean) rstd (RMSNorm: x rstd),  g = dy gamma,
//   S1 = sum g,  S2 = sum g xhat,
//   dx = rstd (g - S1 / C - xhat S2 / C)      (RMSNorm: without S1),
// and over rows, per column: dgamma = sum dy xhat, dbeta = sum dy.
//
// A row of rb bytes starts at byte h = (base + r rb) mod 16 of its first
// 16-byte block, and h repeats every P = 16 / gcd(16, rb mod 16) rows (x, dy
// and dx share their address modulo 16).  A warp takes the rows of one phase
// class only, so its lanes own fixed aligned 16-byte chunks of every row it
// sees -- chunk j holds columns W j - h / E .. W j - h / E + W - 1 -- and
// their column partials stay in registers, with gamma read once per launch.
// SUB lanes hold a row (SUB = 8, 16 or 32: a warp takes 4, 2 or 1 rows at a
// time), NQ chunks each, and the next row's chunks while they compute one.
// Full chunks are single 16-byte loads and stores; the head and tail chunk of
// a row move element by element (nothing outside the row is read or written).
// Element pairs use packed f32x2 arithmetic, but g = dy gamma stays a scalar
// round-to-nearest product.  Columns outside the row hold dy = 0 and
// xhat = 0 and add nothing.  A row
// with rstd = 0 (masked by the forward) gets dx = 0 and adds nothing.  At the
// end each block adds its warps' column partials in a fixed order (warp 0..7)
// into its row of the workspace, [gridDim.x][planes][cols] floats, which
// col_reduce_kernel sums: the result does not depend on timing.
#pragma once

#include "rr_kernels.h"
#include "rr_ops.cuh"

namespace rr {

template <int DT, bool RMS, int SUB, int NQ>
__global__ void __launch_bounds__(32 * kLnsWarps)
    lns_bwd_kernel(const LnBwdParams p, const LnsGeo geo) {
  constexpr int E = DType<DT>::E;
  constexpr int W = 16 / E;
  constexpr int kPlanes = RMS ? 1 : 2;
  constexpr int RPW = 32 / SUB;  // rows a warp holds at once
  extern __shared__ __align__(16) float lns_part[];  // [warps][planes][cols]
  const int C = geo.cols;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sl = lane % SUB, sr = lane / SUB;
  const int64_t gw = (int64_t)blockIdx.x * kLnsWarps + warp;
  const int P = geo.P;
  const int cls = (int)(gw % P);            // P divides kLnsWarps
  const int64_t wi = gw / P;                // this warp among its class's warps
  const int64_t wpc = (int64_t)gridDim.x * kLnsWarps / P;
  const int h = (int)(((int64_t)geo.hb0 + (int64_t)cls * geo.rb) & 15);  // head bytes
  const int hc = h / E;                     // elements of chunk 0 before column 0
  const int nch = (h + geo.rb + 15) / 16;   // chunks a row touches
  const int64_t nrows = geo.rows > cls ? (geo.rows - cls + P - 1) / P : 0;  // rows of the class

  // this lane's chunks: column of element e of chunk q, whole-chunk flags,
  // gamma there (0 outside the row), and the column partials
  bool has[NQ], full[NQ];
  float gm[NQ][W], ag[NQ][W], ab[NQ][W];
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    const int j = sl + SUB * q;
    has[q] = j < nch;
    full[q] = has[q] && 16 * j >= h && 16 * j + 16 <= h + geo.rb;
#pragma unroll
    for (int e = 0; e < W; ++e) {
      const int col = W * j + e - hc;
      gm[q][e] = (has[q] && col >= 0 && col < C) ? ld_elem_cached<DT>(p.gamma + (int64_t)col * E)
                                                  : 0.f;
      ag[q][e] = 0.f;
      ab[q][e] = 0.f;
    }
  }

  // A row's raw chunks (and statistics) in registers; the next row's are
  // loaded before the current one is processed (register double buffer), so
  // each warp keeps a row's loads in flight while it computes.
  struct Raw {
    uint4 x[NQ], dy[NQ];
    float rs, mu;
  };
  auto fetch = [&](int64_t t, Raw& v) {
    v.rs = 0.f;
    v.mu = 0.f;
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      v.x[q] = make_uint4(0, 0, 0, 0);
      v.dy[q] = make_uint4(0, 0, 0, 0);
    }
    if (t >= nrows) return;
    const int64_t r = cls + (int64_t)P * t;
    v.rs = __ldg(p.rstd + r);
    if constexpr (!RMS) v.mu = __ldg(p.mean + r);
    const int64_t rowoff = r * (int64_t)geo.rb - h;  // byte of chunk 0 from each tensor's base
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      if (!has[q]) continue;
      const int j = sl + SUB * q;
      const int64_t off = rowoff + 16 * (int64_t)j;
      if (full[q]) {
        v.x[q] = ld_chunk_stream(p.x + off);
        v.dy[q] = ld_chunk_stream(p.dy + off);
      } else {
#pragma unroll
        for (int e = 0; e < W; ++e) {
          const int col = W * j + e - hc;
          if (col >= 0 && col < C) {
            chunk_set_bits<DT>(v.x[q], e, ld_elem_bits<DT>(p.x + off + e * E));
            chunk_set_bits<DT>(v.dy[q], e, ld_elem_bits<DT>(p.dy + off + e * E));
          }
        }
      }
    }
  };

  Raw cur;
  fetch(wi * RPW + sr, cur);
  for (int64_t t0 = wi * RPW; t0 < nrows; t0 += wpc * RPW) {
    const int64_t t = t0 + sr;
    Raw nxt;
    fetch(t + wpc * RPW, nxt);
    const bool act = t < nrows;
    const int64_t r = cls + (int64_t)P * t;
    const float rs = cur.rs, mu = cur.mu;
    const bool live = act && rs != 0.f;
    const int64_t rowoff = r * (int64_t)geo.rb - h;
    // element pairs in packed f32x2 arithmetic; g = dy gamma stays a scalar
    // round-to-nearest product
    float xh[NQ][W], dv[NQ][W];
    float s1a = 0.f, s1b = 0.f, s2a = 0.f, s2b = 0.f;
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      const int j = sl + SUB * q;
      float xv[W];
#pragma unroll
      for (int e = 0; e < W; ++e) {
        const int col = W * j + e - hc;
        // columns outside the row: x = mean (xhat = 0), dy = 0
        const bool in = live && has[q] && col >= 0 && col < C;
        xv[e] = in ? chunk_get<DT>(cur.x[q], e) : mu;
        dv[q][e] = in ? chunk_get<DT>(cur.dy[q], e) : 0.f;
      }
#pragma unroll
      for (int e = 0; e < W; e += 2) {
        if constexpr (RMS) {
          mul2(xh[q][e], xh[q][e + 1], xv[e], xv[e + 1], rs, rs);
        } else {
          float t0, t1;
          add2(t0, t1, xv[e], xv[e + 1], -mu, -mu);
          mul2(xh[q][e], xh[q][e + 1], t0, t1, rs, rs);
        }
        const float g0 = __fmul_rn(dv[q][e], gm[q][e]);
        const float g1 = __fmul_rn(dv[q][e + 1], gm[q][e + 1]);
        if constexpr (!RMS) add2(s1a, s1b, s1a, s1b, g0, g1);
        fma2(s2a, s2b, g0, g1, xh[q][e], xh[q][e + 1], s2a, s2b);
      }
    }
    float s1 = s1a + s1b, s2 = s2a + s2b;
    // the row's sums over its SUB lanes (every lane ends with the same bits)
#pragma unroll
    for (int o = SUB / 2; o >= 1; o >>= 1) {
      if constexpr (!RMS) s1 += __shfl_xor_sync(0xffffffffu, s1, o);
      s2 += __shfl_xor_sync(0xffffffffu, s2, o);
    }
    cur = nxt;
    if (!act) continue;
    const float a = RMS ? 0.f : s1 * p.inv_cols;
    const float b = s2 * p.inv_cols;
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      if (!has[q]) continue;
      const int j = sl + SUB * q;
      float f[W];
#pragma unroll
      for (int e = 0; e < W; e += 2) {
        const float g0 = __fmul_rn(dv[q][e], gm[q][e]);
        const float g1 = __fmul_rn(dv[q][e + 1], gm[q][e + 1]);
        float t0, t1;
        add2(t0, t1, g0, g1, -a, -a);
        fma2(t0, t1, xh[q][e], xh[q][e + 1], -b, -b, t0, t1);
        mul2(f[e], f[e + 1], t0, t1, rs, rs);
        if (!live) f[e] = f[e + 1] = 0.f;  // a masked row: dx = 0
        fma2(ag[q][e], ag[q][e + 1], dv[q][e], dv[q][e + 1], xh[q][e], xh[q][e + 1], ag[q][e],
             ag[q][e + 1]);
        if constexpr (!RMS)
          add2(ab[q][e], ab[q][e + 1], ab[q][e], ab[q][e + 1], dv[q][e], dv[q][e + 1]);
      }
      const int64_t off = rowoff + 16 * (int64_t)j;
      if (full[q]) {
        st_chunk_stream(p.dx + off, chunk_pack<DT>(f));
      } else {
#pragma unroll
        for (int e = 0; e < W; ++e) {
          const int col = W * j + e - hc;
          if (col >= 0 && col < C) st_elem<DT>(p.dx + off + e * E, f[e]);
        }
      }
    }
  }

  // the warp's column partials: the rows it held side by side added (SUB <
  // 32), then each column written once into the warp's shared-memory row
  float* mine = lns_part + (size_t)warp * kPlanes * C;
  for (int i = lane; i < kPlanes * C; i += 32) mine[i] = 0.f;
  __syncwarp();
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
#pragma unroll
    for (int e = 0; e < W; ++e) {
#pragma unroll
      for (int o = 16; o >= SUB; o >>= 1) {  // the warp's rows, lower lanes first
        const float og = __shfl_xor_sync(0xffffffffu, ag[q][e], o);
        const float ob = __shfl_xor_sync(0xffffffffu, ab[q][e], o);
        const bool lo = (lane & o) == 0;
        ag[q][e] = lo ? ag[q][e] + og : og + ag[q][e];
        ab[q][e] = lo ? ab[q][e] + ob : ob + ab[q][e];
      }
      const int col = W * (sl + SUB * q) + e - hc;
      if (sr == 0 && has[q] && col >= 0 && col < C) {
        mine[col] = ag[q][e];
        if constexpr (!RMS) mine[C + col] = ab[q][e];
      }
    }
  }
  __syncthreads();
  float* out = p.ws + (int64_t)blockIdx.x * kPlanes * C;
  for (int i = threadIdx.x; i < kPlanes * C; i += blockDim.x) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kLnsWarps; ++w) s += lns_part[(size_t)w * kPlanes * C + i];
    out[i] = s;
  }
}

// Variants (SUB lanes a row, NQ chunks a lane): 0 (8, 1), 1 (16, 1), 2 (32, 1)
// and, fp32 only, 3 (32, 2).  Two chunks a lane at 8 or 16 lanes a row were
// slower for the LayerNorm (fp32 31 columns 69.0 against 75.4 us), and
// two-chunk bf16 variants need ~170 registers and were slower than the row
// groups.
template <int DT>
LnsKernels make_lns_set() {
  LnsKernels k{};
  k.bwd[0][0] = (const void*)lns_bwd_kernel<DT, false, 8, 1>;
  k.bwd[0][1] = (const void*)lns_bwd_kernel<DT, false, 16, 1>;
  k.bwd[0][2] = (const void*)lns_bwd_kernel<DT, false, 32, 1>;
  k.bwd[1][0] = (const void*)lns_bwd_kernel<DT, true, 8, 1>;
  k.bwd[1][1] = (const void*)lns_bwd_kernel<DT, true, 16, 1>;
  k.bwd[1][2] = (const void*)lns_bwd_kernel<DT, true, 32, 1>;
  if constexpr (DT == kF32) {
    k.bwd[0][3] = (const void*)lns_bwd_kernel<DT, false, 32, 2>;
    k.bwd[1][3] = (const void*)lns_bwd_kernel<DT, true, 32, 2>;
  }
  return k;
}

}  // namespace rr
