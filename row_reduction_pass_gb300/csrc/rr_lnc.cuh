// rr_lnc.cuh -- LayerNorm / RMSNorm forward and backward for very long rows,
// by column blocks: the row statistics in one launch, the outputs in the next
// ("Engineering a CUDA Machine Learning Framework from Scratch", sec. 3.2 for
// the moments and their pairwise (Chan / Welford) merge, sec. 2.2 for the
// analytic backward, sec. 2.3 for the 128-bit accesses).
//
// Rows fall into P phase classes as in rr_lnx.cuh (the rows of a class all
// start at the same offset phi within their first aligned 16-byte chunk), so
// chunk k of a row of class c is an aligned 16-byte block whose lane e is
// column k * W + e - phi.  A work item is (class, column block b, row group):
// chunks [b * CB, b * CB + CB) of the rows of the class in the group.  Warp w
// of the block takes chunks b * CB + 32 * CPL * w + lane + 32 * j (j < CPL) of
// each of the item's rows in turn: the warps stream different columns of the
// same rows, and no thread ever waits for another block -- the launches order
// the phases.  Rows of a few hundred thousand bytes then keep every SM busy
// (a row per block or per cluster leaves most SMs idle or waiting), and the
// second launch reads its inputs again from L2, where the first left them.
//
// Forward, three launches:
//   1. lnc_stats: per row and column block, the moments of the block's values
//      (count n, sum S as a double-float, M2 about the mean), per warp in the
//      corrected two-pass form -- a first sum gives a provisional mean m0, the
//      deviations d = x - m0 then give S = n m0 + sum d (exact product,
//      TwoSum) and M2 = sum d^2 - (sum d)^2 / n -- and the block's warps
//      merged with the Chan / Golub / LeVeque update in warp order.  RMSNorm:
//      sum x^2.  The records go to scratch inside y, which launch 3 overwrites.
//   2. lnc_merge: per row, the column blocks' records merged in block order:
//      mean, rstd (a row whose moments are not finite is masked: 0, 0).
//   3. lnc_norm: y = (x - mean) * rstd * gamma + beta (RMSNorm: x * rstd *
//      gamma), gamma / beta of the item's columns held in registers for all
//      of its rows.
// Backward, two launches and the column reduce:
//   1. lnc_bwd_part: per row and column block, S1 = sum g and S2 = sum g xhat
//      (g = dy * gamma rounded once, xhat = (x - mean) * rstd), per warp and
//      then over the warps in order, to records in the workspace; each lane's
//      column partials sum dy xhat and sum dy over the item's rows go to the
//      item's partial row (class, row group) of the workspace.
//   2. lnc_bwd_dx: per row, S1 and S2 summed over the blocks (a lane per
//      record, ordered butterfly: the same bits in every block of the row) and
//      dx = rstd * ((g - S1 / C) - xhat * S2 / C).
// The copies read whole aligned 16-byte chunks, so the first (last) row of a
// tensor whose base (end) is not 16-byte aligned reads up to 15 bytes before
// (after) it, in a 16-byte block that holds a byte of the tensor; those lanes
// are zeroed before use and never written.
#pragma once

#include "rr_kernels.h"
#include "rr_ops.cuh"

namespace rr {

// Chunks per lane of one row and the chunks a block covers per row.
template <int CPL>
struct LncShape {
  static constexpr int kCB = 32 * CPL * kLncWarps;
};

// A block's work item and its view of the rows.
template <int W, int CPL>
struct LncItem {
  int cls, b, grp;
  int phi;          // row start offset within its first chunk, in elements
  int64_t nch;      // chunks covering a row of the class
  int tail_lanes;   // valid lanes of the row's last chunk (1 .. W)
  int64_t r0;       // first row of the item; rows r0 + i * P (i < nr)
  int nr;
  int64_t k[CPL];   // this lane's chunks of the row
  int lo[CPL], hi[CPL];  // their valid lanes [lo, hi) (empty outside the row)
  int64_t rowb;     // bytes per row

  __device__ __forceinline__ void init(const LncGeo& g, const char* base, int E) {
    const int64_t it = blockIdx.x;
    cls = static_cast<int>(it % g.P);
    const int64_t rest = it / g.P;
    b = static_cast<int>(rest % g.nb);
    grp = static_cast<int>(rest / g.nb);
    rowb = g.cols * E;
    phi = static_cast<int>(((reinterpret_cast<uintptr_t>(base) + (uint64_t)cls * rowb) & 15) / E);
    nch = (phi + g.cols + W - 1) / W;
    tail_lanes = static_cast<int>(phi + g.cols - (int64_t)W * (nch - 1));
    // rows of the class: cls, cls + P, ...; this group's: [grp * rg, grp * rg + rg)
    const int64_t first = (int64_t)grp * g.rg;
    const int64_t in_class = g.rows > cls ? (g.rows - cls + g.P - 1) / g.P : 0;
    r0 = cls + (int64_t)g.P * first;
    nr = static_cast<int>(first < in_class ? (in_class - first < g.rg ? in_class - first : g.rg) : 0);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
      k[j] = (int64_t)b * LncShape<CPL>::kCB + 32 * CPL * warp + lane + 32 * j;
      lo[j] = 0;
      hi[j] = W;
      if (k[j] >= nch) lo[j] = hi[j] = 0;
      else {
        if (k[j] == 0) lo[j] = phi;
        if (k[j] == nch - 1) hi[j] = tail_lanes;
      }
    }
  }
  // Aligned address of chunk j of row r.
  __device__ __forceinline__ const char* chunk(const char* base, int64_t r, int j, int E) const {
    return base + r * rowb - (int64_t)phi * E + k[j] * 16;
  }
  __device__ __forceinline__ int64_t row(int i, const LncGeo& g) const { return r0 + (int64_t)i * g.P; }
};

// The W values src[col0, col0 + W) of a [cols] vector as fp32, 0 outside
// [0, cols): the funnel shift of the (up to) two aligned 16-byte blocks that
// hold them; a block wholly outside the vector is not read.
template <int DT, int W>
__device__ __forceinline__ void lnc_vec_chunk(const char* src, int64_t cols, int64_t col0,
                                              float (&f)[W]) {
  constexpr int E = DType<DT>::E;
  const intptr_t v0 = reinterpret_cast<intptr_t>(src), v1 = v0 + (intptr_t)cols * E;
  const intptr_t a = v0 + (intptr_t)col0 * E;
  const intptr_t bl = a & ~intptr_t(15);
  uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
  if (bl + 16 > v0 && bl < v1) lo = ld_chunk_cached(reinterpret_cast<const char*>(bl));
  if ((a & 15) != 0 && bl + 32 > v0 && bl + 16 < v1)
    hi = ld_chunk_cached(reinterpret_cast<const char*>(bl + 16));
  const uint4 c = funnel16(lo, hi, static_cast<int>(a & 15));
#pragma unroll
  for (int e = 0; e < W; ++e) {
    const int64_t col = col0 + e;
    f[e] = (col >= 0 && col < cols) ? chunk_get<DT>(c, e) : 0.f;
  }
}

// Unpacks chunk c (all W lanes).
template <int DT, int W>
__device__ __forceinline__ void lnc_unpack(const uint4& c, float (&f)[W]) {
#pragma unroll
  for (int e = 0; e < W; ++e) f[e] = chunk_get<DT>(c, e);
}
// Zeroes the lanes outside [lo, hi): only a row's first and last chunk have
// any (other rows' values, or past the row), so interior chunks skip this.
template <int W>
__device__ __forceinline__ void lnc_clip(float (&f)[W], int lo, int hi) {
  if (lo != 0 || hi != W) {
#pragma unroll
    for (int e = 0; e < W; ++e)
      if (e < lo || e >= hi) f[e] = 0.f;
  }
}

// Stores chunk j of a row: one aligned 128-bit store for an interior chunk,
// the row's own lanes one by one for its first / last chunk.
template <int DT, int W>
__device__ __forceinline__ void lnc_store(char* a, int lo, int hi, const float (&f)[W]) {
  constexpr int E = DType<DT>::E;
  if (lo == 0 && hi == W) {
    st_chunk_stream(a, chunk_pack<DT>(f));
  } else {
#pragma unroll
    for (int e = 0; e < W; ++e)
      if (e >= lo && e < hi) st_elem<DT>(a + e * E, f[e]);
  }
}

// Sum over the warp, the same bits in every lane (an ordered butterfly of a
// commutative add).
__device__ __forceinline__ float lnc_warp_sum(float v) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// Rows are streamed two at a time, the next two rows' chunks loaded before
// the current two are used (double-buffered in registers), so every warp
// keeps 2 x 2 x CPL (forward) or 2 x 2 x 2 x CPL (backward) 16-byte loads in
// flight while it computes.
constexpr int kLncRB = 2;

// T tensors' chunks of rows i .. i + kLncRB - 1 of the item (zeros past nr or
// outside the row).
template <int T, int W, int CPL, bool STREAM>
__device__ __forceinline__ void lnc_load(uint4 (&c)[kLncRB][T][CPL], const LncItem<W, CPL>& it,
                                         const LncGeo& g, const char* const (&src)[T], int i,
                                         int E) {
#pragma unroll
  for (int u = 0; u < kLncRB; ++u)
#pragma unroll
    for (int t = 0; t < T; ++t)
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        c[u][t][j] = make_uint4(0u, 0u, 0u, 0u);
        if (i + u < it.nr && it.hi[j] > it.lo[j]) {
          const char* a = it.chunk(src[t], it.row(i + u, g), j, E);
          c[u][t][j] = STREAM ? ld_chunk_stream(a) : ld_chunk_cached(a);
        }
      }
}

// ------------------------------------------------------------- forward ----

// Launch 1: per (row, column block) records -- Moments (LayerNorm) or the sum
// of squares (RMSNorm) -- into the scratch at p.y rounded up to 16 bytes.
template <int DT, bool RMS, int CPL>
__global__ void __launch_bounds__(32 * kLncWarps, 3) lnc_stats_kernel(const LnFwdParams p,
                                                                      const LncGeo g) {
  constexpr int E = DType<DT>::E, W = DType<DT>::V;
  constexpr int RS = 32;  // rows whose warp records are merged together
  __shared__ Moments part[RS][kLncWarps];
  LncItem<W, CPL> it;
  it.init(g, p.x, E);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  char* recs = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(p.y) + 15) & ~uintptr_t(15));
  // valid values of this warp's slice of a row (the same for every row)
  int cnt = 0;
#pragma unroll
  for (int j = 0; j < CPL; ++j) cnt += it.hi[j] - it.lo[j];
  const float nw = lnc_warp_sum(static_cast<float>(cnt));
  const float inv_nw = nw > 0.f ? 1.f / nw : 0.f;
  const char* const src[1] = {p.x};

  uint4 nxt[kLncRB][1][CPL];
  lnc_load<1, W, CPL, false>(nxt, it, g, src, 0, E);
  for (int i = 0; i < it.nr; i += kLncRB) {
    uint4 cur[kLncRB][1][CPL];
#pragma unroll
    for (int u = 0; u < kLncRB; ++u)
#pragma unroll
      for (int j = 0; j < CPL; ++j) cur[u][0][j] = nxt[u][0][j];
    if (i + kLncRB < it.nr) lnc_load<1, W, CPL, false>(nxt, it, g, src, i + kLncRB, E);
#pragma unroll
    for (int u = 0; u < kLncRB; ++u) {
      if (i + u >= it.nr) break;
      float v[CPL][W];
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        lnc_unpack<DT, W>(cur[u][0][j], v[j]);
        lnc_clip<W>(v[j], it.lo[j], it.hi[j]);
      }
      Moments m;
      if constexpr (RMS) {
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int j = 0; j < CPL; ++j)
#pragma unroll
          for (int e = 0; e < W; e += 2) fma2(a0, a1, v[j][e], v[j][e + 1], v[j][e], v[j][e + 1], a0, a1);
        m = {0.f, lnc_warp_sum(a0 + a1), 0.f, 0.f};
      } else {
        // provisional mean, then the deviations about it
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int j = 0; j < CPL; ++j)
#pragma unroll
          for (int e = 0; e < W; e += 2) add2(s0, s1, s0, s1, v[j][e], v[j][e + 1]);
        const float m0 = lnc_warp_sum(s0 + s1) * inv_nw;
        float d0 = 0.f, d1 = 0.f, q0 = 0.f, q1 = 0.f;
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
          float d[W];
#pragma unroll
          for (int e = 0; e < W; e += 2) add2(d[e], d[e + 1], v[j][e], v[j][e + 1], -m0, -m0);
          lnc_clip<W>(d, it.lo[j], it.hi[j]);
#pragma unroll
          for (int e = 0; e < W; e += 2) {
            add2(d0, d1, d0, d1, d[e], d[e + 1]);
            fma2(q0, q1, d[e], d[e + 1], d[e], d[e + 1], q0, q1);
          }
        }
        const float sd = lnc_warp_sum(d0 + d1), q = lnc_warp_sum(q0 + q1);
        // S = nw m0 + sd as a double-float (the product's error exact in one FMA)
        const float pr = __fmul_rn(nw, m0), pe = fmaf(nw, m0, -pr);
        float h, l;
        two_sum(pr, sd, h, l);
        l += pe;
        float sh, sl;
        two_sum(h, l, sh, sl);
        const float t = q - (nw > 0.f ? sd * sd * inv_nw : 0.f);
        m = {nw, nw > 0.f ? sh : 0.f, nw > 0.f ? sl : 0.f, t < 0.f ? 0.f : t};
      }
      if (lane == 0) part[(i + u) % RS][warp] = m;
    }
    // every RS rows (and at the end): the block's record of each row, its
    // warps' records merged in warp order
    const int done = min(i + kLncRB, it.nr);
    if (done % RS == 0 || done == it.nr) {
      __syncthreads();
      const int base = (done - 1) / RS * RS, ns = done - base;
      if (threadIdx.x < ns) {
        const int ri = threadIdx.x;
        Moments m = part[ri][0];
        for (int w = 1; w < kLncWarps; ++w) {
          if constexpr (RMS) m.sh += part[ri][w].sh;
          else m = MergeMoments()(m, part[ri][w]);
        }
        const int64_t r = it.row(base + ri, g);
        if constexpr (RMS)
          reinterpret_cast<float*>(recs)[r * g.nb + it.b] = m.sh;
        else
          reinterpret_cast<float4*>(recs)[r * g.nb + it.b] = make_float4(m.n, m.sh, m.sl, m.m2);
      }
      __syncthreads();
    }
  }
}

// Launch 2: a warp per row merges the row's records (lane l: records l,
// l + 32, ... in order, then an ordered butterfly) and writes mean (LayerNorm)
// and rstd.
template <bool RMS>
__global__ void __launch_bounds__(256) lnc_merge_kernel(const LnFwdParams p, const LncGeo g) {
  const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= g.rows) return;  // whole warps
  const char* recs =
      reinterpret_cast<const char*>((reinterpret_cast<uintptr_t>(p.y) + 15) & ~uintptr_t(15));
  if constexpr (RMS) {
    const float* s = reinterpret_cast<const float*>(recs) + r * g.nb;
    float t = 0.f;
    for (int b = lane; b < g.nb; b += 32) t += s[b];
    const float ms = lnc_warp_sum(t) * p.inv_cols;
    if (lane == 0) p.rstd[r] = isfinite(ms) ? rsqrtf(ms + p.eps) : 0.f;
  } else {
    const float4* s = reinterpret_cast<const float4*>(recs) + r * g.nb;
    Moments m = Moments::identity();
    for (int b = lane; b < g.nb; b += 32) {
      const float4 f = s[b];
      m = MergeMoments()(m, Moments{f.x, f.y, f.z, f.w});
    }
    m = group_reduce<Moments, MergeMoments, 32>(m, MergeMoments());
    if (lane == 0) {
      float mh, ml;
      df_mean(m.sh, m.sl, static_cast<float>(g.cols), p.inv_cols, mh, ml);
      const float var = m.m2 * p.inv_cols;
      const bool masked = !(isfinite(mh) && isfinite(ml) && isfinite(var));
      p.mean[r] = masked ? 0.f : mh + ml;
      p.rstd[r] = masked ? 0.f : rsqrtf(var + p.eps);
    }
  }
}

// Launch 3: y from x (read again), the saved mean / rstd and gamma / beta.
template <int DT, bool RMS, int CPL>
__global__ void __launch_bounds__(32 * kLncWarps, RMS ? 3 : 2) lnc_norm_kernel(const LnFwdParams p,
                                                                     const LncGeo g) {
  constexpr int E = DType<DT>::E, W = DType<DT>::V;
  LncItem<W, CPL> it;
  it.init(g, p.x, E);
  const char* const src[1] = {p.x};
  uint4 nxt[kLncRB][1][CPL];
  lnc_load<1, W, CPL, true>(nxt, it, g, src, 0, E);
  float gm[CPL][W], bt[CPL][W];
#pragma unroll
  for (int j = 0; j < CPL; ++j) {
    const int64_t col0 = it.k[j] * W - it.phi;
#pragma unroll
    for (int e = 0; e < W; ++e) gm[j][e] = bt[j][e] = 0.f;
    if (it.hi[j] > it.lo[j]) {
      lnc_vec_chunk<DT, W>(p.gamma, g.cols, col0, gm[j]);
      if constexpr (!RMS) lnc_vec_chunk<DT, W>(p.beta, g.cols, col0, bt[j]);
    }
  }
  for (int i = 0; i < it.nr; i += kLncRB) {
    uint4 cur[kLncRB][1][CPL];
    float mean[kLncRB], rstd[kLncRB];
#pragma unroll
    for (int u = 0; u < kLncRB; ++u) {
      mean[u] = rstd[u] = 0.f;
      if (i + u < it.nr) {
        const int64_t r = it.row(i + u, g);
        if constexpr (!RMS) mean[u] = __ldg(p.mean + r);
        rstd[u] = __ldg(p.rstd + r);
      }
#pragma unroll
      for (int j = 0; j < CPL; ++j) cur[u][0][j] = nxt[u][0][j];
    }
    if (i + kLncRB < it.nr) lnc_load<1, W, CPL, true>(nxt, it, g, src, i + kLncRB, E);
#pragma unroll
    for (int u = 0; u < kLncRB; ++u) {
      if (i + u >= it.nr) break;
      const int64_t r = it.row(i + u, g);
      const bool masked = rstd[u] == 0.f;
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        if (it.hi[j] <= it.lo[j]) continue;
        float v[W], y[W];
        lnc_unpack<DT, W>(cur[u][0][j], v);
        if (masked) {
#pragma unroll
          for (int e = 0; e < W; ++e) y[e] = 0.f;
        } else {
#pragma unroll
          for (int e = 0; e < W; e += 2) {
            float t0, t1;
            if constexpr (RMS) {
              mul2(t0, t1, v[e], v[e + 1], rstd[u], rstd[u]);
              mul2(y[e], y[e + 1], t0, t1, gm[j][e], gm[j][e + 1]);
            } else {
              add2(t0, t1, v[e], v[e + 1], -mean[u], -mean[u]);
              mul2(t0, t1, t0, t1, rstd[u], rstd[u]);
              fma2(y[e], y[e + 1], t0, t1, gm[j][e], gm[j][e + 1], bt[j][e], bt[j][e + 1]);
            }
          }
        }
        lnc_store<DT, W>(const_cast<char*>(it.chunk(p.y, r, j, E)), it.lo[j], it.hi[j], y);
      }
    }
  }
}

// ------------------------------------------------------------ backward ----

// Launch 1: per (row, column block) records (S1, S2) at p.ws + g.rec_off
// floats, and the item's column partials (sum dy xhat, sum dy) in its partial
// row (class, row group) of p.ws: [partial][planes][cols].
template <int DT, bool RMS, int CPL>
__global__ void __launch_bounds__(32 * kLncWarps, 2) lnc_bwd_part_kernel(const LnBwdParams p,
                                                                         const LncGeo g) {
  constexpr int E = DType<DT>::E, W = DType<DT>::V;
  constexpr int kPlanes = RMS ? 1 : 2;
  constexpr int RS = 32;
  __shared__ float2 part[RS][kLncWarps];
  LncItem<W, CPL> it;
  it.init(g, p.x, E);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float2* recs = reinterpret_cast<float2*>(p.ws + g.rec_off);
  const char* const src[2] = {p.dy, p.x};
  uint4 nxt[kLncRB][2][CPL];
  lnc_load<2, W, CPL, false>(nxt, it, g, src, 0, E);
  float gm[CPL][W], ag[CPL][W], ab[CPL][W];
#pragma unroll
  for (int j = 0; j < CPL; ++j) {
#pragma unroll
    for (int e = 0; e < W; ++e) gm[j][e] = ag[j][e] = ab[j][e] = 0.f;
    if (it.hi[j] > it.lo[j]) lnc_vec_chunk<DT, W>(p.gamma, g.cols, it.k[j] * W - it.phi, gm[j]);
  }
  for (int i = 0; i < it.nr; i += kLncRB) {
    uint4 cur[kLncRB][2][CPL];
    float mean[kLncRB], rstd[kLncRB];
#pragma unroll
    for (int u = 0; u < kLncRB; ++u) {
      mean[u] = rstd[u] = 0.f;
      if (i + u < it.nr) {
        const int64_t r = it.row(i + u, g);
        if constexpr (!RMS) mean[u] = __ldg(p.mean + r);
        rstd[u] = __ldg(p.rstd + r);
      }
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int j = 0; j < CPL; ++j) cur[u][t][j] = nxt[u][t][j];
    }
    if (i + kLncRB < it.nr) lnc_load<2, W, CPL, false>(nxt, it, g, src, i + kLncRB, E);
#pragma unroll
    for (int u = 0; u < kLncRB; ++u) {
      if (i + u >= it.nr) break;
      float s1a = 0.f, s1b = 0.f, s2a = 0.f, s2b = 0.f;
      if (rstd[u] != 0.f) {  // a masked row adds nothing
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
          float dv[W], xv[W];
          lnc_unpack<DT, W>(cur[u][0][j], dv);
          lnc_unpack<DT, W>(cur[u][1][j], xv);
          lnc_clip<W>(dv, it.lo[j], it.hi[j]);
          lnc_clip<W>(xv, it.lo[j], it.hi[j]);
#pragma unroll
          for (int e = 0; e < W; e += 2) {
            float h0, h1;
            if constexpr (RMS) {
              mul2(h0, h1, xv[e], xv[e + 1], rstd[u], rstd[u]);
            } else {
              add2(h0, h1, xv[e], xv[e + 1], -mean[u], -mean[u]);
              mul2(h0, h1, h0, h1, rstd[u], rstd[u]);
            }
            // g rounded once (a product that must not fuse into the sums)
            const float g0 = __fmul_rn(dv[e], gm[j][e]), g1 = __fmul_rn(dv[e + 1], gm[j][e + 1]);
            if constexpr (!RMS) add2(s1a, s1b, s1a, s1b, g0, g1);
            fma2(s2a, s2b, g0, g1, h0, h1, s2a, s2b);
            fma2(ag[j][e], ag[j][e + 1], dv[e], dv[e + 1], h0, h1, ag[j][e], ag[j][e + 1]);
            if constexpr (!RMS) add2(ab[j][e], ab[j][e + 1], ab[j][e], ab[j][e + 1], dv[e], dv[e + 1]);
          }
        }
      }
      const float s1 = RMS ? 0.f : lnc_warp_sum(s1a + s1b), s2 = lnc_warp_sum(s2a + s2b);
      if (lane == 0) part[(i + u) % RS][warp] = make_float2(s1, s2);
    }
    const int done = min(i + kLncRB, it.nr);
    if (done % RS == 0 || done == it.nr) {
      __syncthreads();
      const int base = (done - 1) / RS * RS, ns = done - base;
      if (threadIdx.x < ns) {
        const int ri = threadIdx.x;
        float2 t = part[ri][0];
        for (int w = 1; w < kLncWarps; ++w) {
          t.x += part[ri][w].x;
          t.y += part[ri][w].y;
        }
        recs[it.row(base + ri, g) * g.nb + it.b] = t;
      }
      __syncthreads();
    }
  }
  // the item's column partials: every column of the block, zeros included
  float* out = p.ws + ((int64_t)it.cls * g.ng + it.grp) * kPlanes * g.cols;
#pragma unroll
  for (int j = 0; j < CPL; ++j) {
    if (it.hi[j] <= it.lo[j]) continue;
    const int64_t col0 = it.k[j] * W - it.phi;
#pragma unroll
    for (int e = 0; e < W; ++e) {
      if (e < it.lo[j] || e >= it.hi[j]) continue;
      out[col0 + e] = ag[j][e];
      if constexpr (!RMS) out[g.cols + col0 + e] = ab[j][e];
    }
  }
}

// Launch 2: dx from dy, x (read again), mean / rstd, gamma and the row's
// (S1, S2) summed over its column blocks.
template <int DT, bool RMS, int CPL>
__global__ void __launch_bounds__(32 * kLncWarps, 2) lnc_bwd_dx_kernel(const LnBwdParams p,
                                                                       const LncGeo g) {
  constexpr int E = DType<DT>::E, W = DType<DT>::V;
  LncItem<W, CPL> it;
  it.init(g, p.x, E);
  const int lane = threadIdx.x & 31;
  const float2* recs = reinterpret_cast<const float2*>(p.ws + g.rec_off);
  const char* const src[2] = {p.dy, p.x};
  uint4 nxt[kLncRB][2][CPL];
  lnc_load<2, W, CPL, true>(nxt, it, g, src, 0, E);
  float gm[CPL][W];
#pragma unroll
  for (int j = 0; j < CPL; ++j) {
#pragma unroll
    for (int e = 0; e < W; ++e) gm[j][e] = 0.f;
    if (it.hi[j] > it.lo[j]) lnc_vec_chunk<DT, W>(p.gamma, g.cols, it.k[j] * W - it.phi, gm[j]);
  }
  for (int i = 0; i < it.nr; i += kLncRB) {
    uint4 cur[kLncRB][2][CPL];
    float mean[kLncRB], rstd[kLncRB], a[kLncRB], bq[kLncRB];
#pragma unroll
    for (int u = 0; u < kLncRB; ++u) {
      mean[u] = rstd[u] = a[u] = bq[u] = 0.f;
      if (i + u < it.nr) {
        const int64_t r = it.row(i + u, g);
        if constexpr (!RMS) mean[u] = __ldg(p.mean + r);
        rstd[u] = __ldg(p.rstd + r);
        // the row's sums: lane l adds records l, l + 32, ... in order, then
        // the lanes' sums by an ordered butterfly
        float t1 = 0.f, t2 = 0.f;
        for (int b = lane; b < g.nb; b += 32) {
          const float2 s = __ldg(recs + r * g.nb + b);
          t1 += s.x;
          t2 += s.y;
        }
        a[u] = (RMS ? 0.f : lnc_warp_sum(t1)) * p.inv_cols;
        bq[u] = lnc_warp_sum(t2) * p.inv_cols;
      }
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int j = 0; j < CPL; ++j) cur[u][t][j] = nxt[u][t][j];
    }
    if (i + kLncRB < it.nr) lnc_load<2, W, CPL, true>(nxt, it, g, src, i + kLncRB, E);
#pragma unroll
    for (int u = 0; u < kLncRB; ++u) {
      if (i + u >= it.nr) break;
      const int64_t r = it.row(i + u, g);
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        if (it.hi[j] <= it.lo[j]) continue;
        float o[W];
        if (rstd[u] == 0.f) {
#pragma unroll
          for (int e = 0; e < W; ++e) o[e] = 0.f;
        } else {
          float dv[W], xv[W];
          lnc_unpack<DT, W>(cur[u][0][j], dv);
          lnc_unpack<DT, W>(cur[u][1][j], xv);
#pragma unroll
          for (int e = 0; e < W; e += 2) {
            float h0, h1, t0, t1;
            if constexpr (RMS) {
              mul2(h0, h1, xv[e], xv[e + 1], rstd[u], rstd[u]);
            } else {
              add2(h0, h1, xv[e], xv[e + 1], -mean[u], -mean[u]);
              mul2(h0, h1, h0, h1, rstd[u], rstd[u]);
            }
            const float g0 = __fmul_rn(dv[e], gm[j][e]), g1 = __fmul_rn(dv[e + 1], gm[j][e + 1]);
            add2(t0, t1, g0, g1, -a[u], -a[u]);             // g - S1 / C
            fma2(t0, t1, h0, h1, -bq[u], -bq[u], t0, t1);   // - xhat S2 / C
            mul2(o[e], o[e + 1], t0, t1, rstd[u], rstd[u]);
          }
        }
        lnc_store<DT, W>(const_cast<char*>(it.chunk(p.dx, r, j, E)), it.lo[j], it.hi[j], o);
      }
    }
  }
}

template <int DT>
LncKernels make_lnc_set() {
  LncKernels s{};
  s.stats[0] = (const void*)lnc_stats_kernel<DT, false, kLncCplFwd>;
  s.stats[1] = (const void*)lnc_stats_kernel<DT, true, kLncCplFwd>;
  s.merge[0] = (const void*)lnc_merge_kernel<false>;
  s.merge[1] = (const void*)lnc_merge_kernel<true>;
  s.norm[0] = (const void*)lnc_norm_kernel<DT, false, kLncCplFwd>;
  s.norm[1] = (const void*)lnc_norm_kernel<DT, true, kLncCplFwd>;
  s.part[0] = (const void*)lnc_bwd_part_kernel<DT, false, kLncCplBwd>;
  s.part[1] = (const void*)lnc_bwd_part_kernel<DT, true, kLncCplBwd>;
  s.dx[0] = (const void*)lnc_bwd_dx_kernel<DT, false, kLncCplBwd>;
  s.dx[1] = (const void*)lnc_bwd_dx_kernel<DT, true, kLncCplBwd>;
  return s;
}

}  // namespace rr
