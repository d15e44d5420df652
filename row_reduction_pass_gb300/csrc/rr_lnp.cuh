// rr_lnp.cuh -- LayerNorm / RMSNorm forward and backward for long rows with
// pipelined row merges ("Engineering a CUDA Machine Learning Framework from
// Scratch", sec. 3.2 for the one-pass moments merged pairwise, sec. 2.2 for
// the analytic backward, sec. 2.3 for the 128-bit accesses).
//
// The rows are laid out as in rr_lnx.cuh: each block (or cluster) works on the
// rows of one phase class, so every chunk of every row it touches is an
// aligned 16-byte block at the same place relative to the row, and gamma /
// beta are staged once per block, shifted to that phase, as fp32 planes.  The
// row data path is that of rr_smx.cuh: every thread copies its own chunks of
// the rows it will work on (gt, gt + G, ... of a group of G threads) into a
// ring of NS shared-memory stages with asynchronous copies, several rows
// ahead, and is their only reader, so no barrier guards the data and a thread
// holds no row in registers.
//
// Forward, per row: each thread sums its values (fp32, four accumulators),
// takes its mean m_t = S_t / n_t and the squared deviations about it; the
// (n_t, S_t, M2_t) triples are merged with the Chan-Golub-LeVeque update on
// double-float sums with exact cross products (rr_ops.cuh), which is the
// pairwise form of the one-pass (Welford) moments; mean = S / C as a
// double-float, var = M2 / C, rstd = 1 / sqrt(var + eps).  RMSNorm merges the
// sums of squares.  A row with a non-finite mean or variance is masked (y = 0,
// mean = rstd = 0).  y = ((x - mean_h) - mean_l) * rstd * gamma + beta.
//
// Backward, per row (mean and rstd given): g = dy * gamma (rounded once),
// xhat = (x - mean) * rstd, S1 = sum g, S2 = sum g * xhat, then
// dx = rstd * ((g - S1 / C) - xhat * S2 / C).  Each thread's column partials
// (sum dy * xhat, sum dy) of its at most NQB chunks stay in registers across
// all its rows (a block's columns never change: one phase); at the end the
// block's groups add theirs in group order into the block's (or cluster's)
// row of the workspace, which col_reduce_kernel sums.
//
// One warp per row (forward, rows of up to solo_max chunks a lane): the
// warp's butterfly merge is the row's statistic and the row is finished in
// its own iteration.  Otherwise each warp publishes its partial of row j to
// the slots of every rank and arrives on the row's merge barrier, takes row
// j - 1's statistics (published one row earlier) and finishes row j - 1, so
// no warp waits for another within a row.  Slots are merged by every warp in
// the same order, so all threads of all ranks hold the same bits.
#pragma once

#include <cstring>

#include "rr_lnx.cuh"

namespace rr {

// A row group's rows, its asynchronous ring of NT tensors and its merges.
template <int W, int NT, bool CL>
struct RowPipe {
  LnxGroup gr;
  LnxRows<W> rw;
  int K, rank, NS, lane, wg, nslot, ahead, S;
  bool solo;
  uint4* ring;
  uint64_t* mrg;
  float4* slots;

  __device__ __forceinline__ void init(const LnxGeo& g, unsigned char* smem, const char* base,
                                       int E) {
    K = 1;
    rank = 0;
    if constexpr (CL) {
      K = static_cast<int>(cluster_nrank());
      rank = static_cast<int>(cluster_rank());
    }
    gr.init(g.G);
    const int R = static_cast<int>(blockDim.x) / g.G;
    rw.init(g, gr, R, base, E, K, rank);
    NS = g.NS;
    S = g.S;
    lane = threadIdx.x & 31;
    wg = gr.gt >> 5;
    nslot = K * gr.nw;
    solo = !CL && gr.nw == 1;
    ahead = solo ? NS - 1 : NS - 2;
    ring = reinterpret_cast<uint4*>(smem + g.ring_off) + (size_t)gr.grp * NS * NT * S;
    mrg = reinterpret_cast<uint64_t*>(smem + g.bar_off) + (size_t)gr.grp * 2;
    slots = reinterpret_cast<float4*>(smem + g.red_off + (size_t)gr.grp * 1024 * K);
    if (gr.gt == 0) {
      mbar_init(&mrg[0], nslot);
      mbar_init(&mrg[1], nslot);
      fence_mbar_init();
    }
  }
  __device__ __forceinline__ int64_t row(int64_t j) const { return rw.first + j * rw.step; }
  __device__ __forceinline__ uint4* stage(int64_t j, int t) const {
    return ring + ((size_t)(j % NS) * NT + t) * S;
  }
  // This thread's chunks of row j of every tensor (src(t, r): the aligned
  // start of this rank's slice of row r of tensor t) into the row's stage; one
  // commit group per call, empty past the group's last row.
  template <class Src>
  __device__ __forceinline__ void fetch(int64_t j, int64_t rows, Src src) {
    if (row(j) < rows) {
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const char* s = src(t, row(j));
        uint4* d = stage(j, t);
        for (int q = 0; q < rw.nq; ++q) {
          const int k = gr.gt + q * gr.G;
          cp_async16(d + k, s + (int64_t)k * 16);
        }
      }
    }
    cp_async_commit();
  }
  // Row j's copies landed (all but the `ahead` newer groups done).
  __device__ __forceinline__ void landed() const {
    if (ahead <= 0) cp_async_wait<0>();
    else if (ahead == 1) cp_async_wait<1>();
    else if (ahead == 2) cp_async_wait<2>();
    else cp_async_wait<3>();
  }
  // This warp's partial of row j (merged over its lanes) to the slots of
  // every rank, then an arrival on each rank's merge barrier of the row.
  template <class St, class Mg>
  __device__ __forceinline__ void publish(int64_t j, St v) {
    static_assert(sizeof(St) <= 16, "a partial fills one 16-byte slot");
    v = group_reduce<St, Mg, 32>(v, Mg());
    if (lane == 0) {
      float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
      memcpy(&f, &v, sizeof(St));
      const int par = static_cast<int>(j & 1);
      float4* sl = slots + par * nslot + rank * gr.nw + wg;
      if constexpr (CL) {
        for (int k = 0; k < K; ++k) {
          st_cluster_f32x4(map_to_rank(sl, k), f.x, f.y, f.z, f.w);
          mbar_arrive_cluster(map_to_rank(&mrg[par], k));
        }
      } else {
        *sl = f;
        mbar_arrive(&mrg[par]);
      }
    }
  }
  // Row j's statistic: lane l merges slots l, l + 32, ... in order, then an
  // ordered butterfly; the same in every warp of every rank.
  template <class St, class Mg>
  __device__ __forceinline__ St merged(int64_t j, bool& dead, int* err) {
    const int par = static_cast<int>(j & 1);
    const uint32_t ph = static_cast<uint32_t>((j >> 1) & 1);
    if (!dead) {
      if constexpr (CL) dead = !mbar_wait_bounded_cluster(&mrg[par], ph, err);
      else dead = !mbar_wait_bounded(&mrg[par], ph, err);
    }
    St v = St::identity();
    for (int i = lane; i < nslot; i += 32) {
      const float4 f = slots[par * nslot + i];
      St t;
      memcpy(&t, &f, sizeof(St));
      v = Mg()(v, t);
    }
    return group_reduce<St, Mg, 32>(v, Mg());
  }
  // Valid values among this thread's chunks (the head / tail chunks it holds
  // have lanes of the neighbouring rows).
  __device__ __forceinline__ int valid_count() const {
    int n = rw.nq * W;
    if (rw.hq == 0) n -= rw.phi;
    if (rw.tq >= 0) n -= W - rw.tail_lanes;
    return n;
  }
};

// Zeroes in d[] the lanes of chunk q that are not this row's (head / tail).
template <int W>
__device__ __forceinline__ void lnp_mask_lanes(const LnxRows<W>& rw, int q, float (&d)[W]) {
  if (q == rw.hq || q == rw.tq) {
    const int lo = q == rw.hq ? rw.phi : 0;
    const int hi = q == rw.tq ? rw.tail_lanes : W;
#pragma unroll
    for (int e = 0; e < W; ++e)
      if (e < lo || e >= hi) d[e] = 0.f;
  }
}

// ------------------------------------------------------------ forward ------
template <int DT, bool RMS, bool CL>
__global__ void __launch_bounds__(kSmxMaxT, 1) lnp_fwd_kernel(const LnFwdParams p, const LnxGeo g) {
  constexpr int E = DType<DT>::E, W = DType<DT>::V;
  using St = std::conditional_t<RMS, Sum1, Moments>;
  using Mg = std::conditional_t<RMS, MergeSum1, MergeMoments>;
  extern __shared__ __align__(128) unsigned char smem[];
  RowPipe<W, 1, CL> rp;
  rp.init(g, smem, p.x, E);
  const LnxRows<W>& rw = rp.rw;
  const int gt = rp.gr.gt, G = rp.gr.G;
  auto src = [&](int, int64_t r) { return rw.slice(p.x, r, E); };
  for (int i = 0; i < rp.ahead; ++i) rp.fetch(i, g.rows, src);
  float* gam = reinterpret_cast<float*>(smem + g.g_off);
  float* bet = gam + (size_t)g.S * W;
  const int col0 = rw.k0 * W - rw.phi;
  lnx_stage_vec<DT, W>(gam, p.gamma, g.S, g.cols, col0);
  if constexpr (!RMS) lnx_stage_vec<DT, W>(bet, p.beta, g.S, g.cols, col0);
  if constexpr (CL) cluster_sync();  // barriers set up before any peer arrives
  else __syncthreads();
  bool dead = false;
  const float ncols = static_cast<float>(g.cols);

  // step 1 for row j: this thread's partial
  auto partial = [&](int64_t j) -> St {
    uint4* st = rp.stage(j, 0);
    lnx_mask_stage<W>(st, rw, gt, G, E);  // other rows' lanes read as 0
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    if constexpr (RMS) {
#pragma unroll 2
      for (int q = 0; q < rw.nq; ++q) {
        float v[W];
        lnx_unpack<DT, W>(st[gt + q * G], v);
#pragma unroll
        for (int e = 0; e < W; e += 4) {
          fma2(a0, a1, v[e], v[e + 1], v[e], v[e + 1], a0, a1);
          fma2(a2, a3, v[e + 2], v[e + 3], v[e + 2], v[e + 3], a2, a3);
        }
      }
      return Sum1{(a0 + a1) + (a2 + a3)};
    } else {
#pragma unroll 2
      for (int q = 0; q < rw.nq; ++q) {
        float v[W];
        lnx_unpack<DT, W>(st[gt + q * G], v);
#pragma unroll
        for (int e = 0; e < W; e += 4) {
          add2(a0, a1, a0, a1, v[e], v[e + 1]);
          add2(a2, a3, a2, a3, v[e + 2], v[e + 3]);
        }
      }
      const int n = rp.valid_count();
      const float s = (a0 + a1) + (a2 + a3);
      if (n == 0) return Moments{0.f, 0.f, 0.f, 0.f};
      const float m = s / static_cast<float>(n);
      float b0 = 0.f, b1 = 0.f, b2 = 0.f, b3 = 0.f;
#pragma unroll 2
      for (int q = 0; q < rw.nq; ++q) {
        float v[W];
        lnx_unpack<DT, W>(st[gt + q * G], v);
#pragma unroll
        for (int e = 0; e < W; e += 2) add2(v[e], v[e + 1], v[e], v[e + 1], -m, -m);
        lnp_mask_lanes<W>(rw, q, v);
#pragma unroll
        for (int e = 0; e < W; e += 4) {
          fma2(b0, b1, v[e], v[e + 1], v[e], v[e + 1], b0, b1);
          fma2(b2, b3, v[e + 2], v[e + 3], v[e + 2], v[e + 3], b2, b3);
        }
      }
      return Moments{static_cast<float>(n), s, 0.f, (b0 + b1) + (b2 + b3)};
    }
  };

  // step 2 for row j (merged statistic t): outputs and the row statistics
  auto finish = [&](int64_t j, const St& t) {
    const int64_t r = rp.row(j);
    const uint4* st = rp.stage(j, 0);
    float mh = 0.f, ml = 0.f, rstd;
    bool masked;
    if constexpr (RMS) {
      const float ms = t.s * p.inv_cols;
      masked = !isfinite(ms);
      rstd = masked ? 0.f : rsqrtf(ms + p.eps);
      if (gt == 0 && rp.rank == 0) p.rstd[r] = rstd;
    } else {
      float sh, sl;
      two_sum(t.sh, t.sl, sh, sl);
      df_mean(sh, sl, ncols, p.inv_cols, mh, ml);
      const float var = t.m2 * p.inv_cols;
      masked = !(isfinite(mh) && isfinite(ml) && isfinite(var));
      rstd = masked ? 0.f : rsqrtf(var + p.eps);
      if (gt == 0 && rp.rank == 0) {
        p.mean[r] = masked ? 0.f : mh + ml;
        p.rstd[r] = rstd;
      }
    }
    char* ys = const_cast<char*>(rw.slice(p.y, r, E));
#pragma unroll 2
    for (int q = 0; q < rw.nq; ++q) {
      const int k = gt + q * G;
      float y[W];
      if (masked) {
#pragma unroll
        for (int e = 0; e < W; ++e) y[e] = 0.f;
      } else {
        float v[W], gm[W];
        lnx_unpack<DT, W>(st[k], v);
        lnx_vec<W>(gam, g.S, k, gm);
        if constexpr (RMS) {
#pragma unroll
          for (int e = 0; e < W; e += 2) {
            float t0, t1;
            mul2(t0, t1, v[e], v[e + 1], rstd, rstd);
            mul2(y[e], y[e + 1], t0, t1, gm[e], gm[e + 1]);
          }
        } else {
          float bt[W];
          lnx_vec<W>(bet, g.S, k, bt);
#pragma unroll
          for (int e = 0; e < W; e += 2) {
            float t0, t1;
            add2(t0, t1, v[e], v[e + 1], -mh, -mh);
            add2(t0, t1, t0, t1, -ml, -ml);
            mul2(t0, t1, t0, t1, rstd, rstd);
            fma2(y[e], y[e + 1], t0, t1, gm[e], gm[e + 1], bt[e], bt[e + 1]);
          }
        }
      }
      lnx_store<DT, W>(ys, k, q, rw, y);
    }
  };

  int64_t j = 0;
  for (;; ++j) {
    if (rp.row(j) >= g.rows) break;
    rp.fetch(j + rp.ahead, g.rows, src);
    rp.landed();
    const St t = partial(j);
    if (rp.solo) {
      finish(j, group_reduce<St, Mg, 32>(t, Mg()));
    } else {
      St prev{};
      if (j >= 1) prev = rp.template merged<St, Mg>(j - 1, dead, p.err);
      rp.template publish<St, Mg>(j, t);
      if (j >= 1) finish(j - 1, prev);
    }
  }
  if (!rp.solo && j >= 1) finish(j - 1, rp.template merged<St, Mg>(j - 1, dead, p.err));
  cp_async_wait<0>();
  if constexpr (CL) cluster_sync();  // no peer still writes this block's slots
}

// ----------------------------------------------------------- backward ------
// MINB = 2: blocks of at most 320 threads, two per SM (96 registers a thread).
template <int DT, int NQB, bool RMS, bool CL, int MINB = 1>
__global__ void __launch_bounds__(MINB == 2 ? 320 : kSmxMaxT, MINB)
    lnp_bwd_kernel(const LnBwdParams p, const LnxGeo g) {
  constexpr int E = DType<DT>::E, W = DType<DT>::V;
  constexpr int kPlanes = RMS ? 1 : 2;
  extern __shared__ __align__(128) unsigned char smem[];
  RowPipe<W, 2, CL> rp;
  rp.init(g, smem, p.x, E);
  const LnxRows<W>& rw = rp.rw;
  const int gt = rp.gr.gt, G = rp.gr.G;
  auto src = [&](int t, int64_t r) { return rw.slice(t == 0 ? p.dy : p.x, r, E); };
  for (int i = 0; i < rp.ahead; ++i) rp.fetch(i, g.rows, src);
  float* gam = reinterpret_cast<float*>(smem + g.g_off);
  const int col0 = rw.k0 * W - rw.phi;
  lnx_stage_vec<DT, W>(gam, p.gamma, g.S, g.cols, col0);
  if constexpr (CL) cluster_sync();
  else __syncthreads();
  bool dead = false;

  // column partials of this thread's chunks: sum dy * xhat (, sum dy)
  float ag[NQB][W], ab[NQB][W];
#pragma unroll
  for (int q = 0; q < NQB; ++q)
#pragma unroll
    for (int e = 0; e < W; ++e) ag[q][e] = ab[q][e] = 0.f;

  // g and xhat of chunk q of row j (stages), given the row's mean / rstd
  auto load_gx = [&](int64_t j, int q, float mean, float rstd, float (&dv)[W], float (&gv)[W],
                     float (&hv)[W]) {
    const int k = gt + q * G;
    float xv[W], gm[W];
    lnx_unpack<DT, W>(rp.stage(j, 0)[k], dv);
    lnx_unpack<DT, W>(rp.stage(j, 1)[k], xv);
    lnx_vec<W>(gam, g.S, k, gm);
#pragma unroll
    for (int e = 0; e < W; e += 2) {
      if constexpr (RMS) {
        mul2(hv[e], hv[e + 1], xv[e], xv[e + 1], rstd, rstd);
      } else {
        add2(hv[e], hv[e + 1], xv[e], xv[e + 1], -mean, -mean);
        mul2(hv[e], hv[e + 1], hv[e], hv[e + 1], rstd, rstd);
      }
      // g rounded once (a product that must not fuse into the sums)
      gv[e] = __fmul_rn(dv[e], gm[e]);
      gv[e + 1] = __fmul_rn(dv[e + 1], gm[e + 1]);
    }
  };

  // step 1 for row j: (S1, S2) of this thread, column partials accumulated
  auto partial = [&](int64_t j, float mean, float rstd) -> Sum2 {
    lnx_mask_stage<W>(rp.stage(j, 0), rw, gt, G, E);
    lnx_mask_stage<W>(rp.stage(j, 1), rw, gt, G, E);
    float s1a = 0.f, s1b = 0.f, s2a = 0.f, s2b = 0.f;
    if (rstd != 0.f) {
#pragma unroll
      for (int q = 0; q < NQB; ++q) {
        if (q < rw.nq) {
          float dv[W], gv[W], hv[W];
          load_gx(j, q, mean, rstd, dv, gv, hv);
#pragma unroll
          for (int e = 0; e < W; e += 2) {
            if constexpr (!RMS) add2(s1a, s1b, s1a, s1b, gv[e], gv[e + 1]);
            fma2(s2a, s2b, gv[e], gv[e + 1], hv[e], hv[e + 1], s2a, s2b);
            fma2(ag[q][e], ag[q][e + 1], dv[e], dv[e + 1], hv[e], hv[e + 1], ag[q][e],
                 ag[q][e + 1]);
            if constexpr (!RMS)
              add2(ab[q][e], ab[q][e + 1], ab[q][e], ab[q][e + 1], dv[e], dv[e + 1]);
          }
        }
      }
    }
    return Sum2{s1a + s1b, s2a + s2b};
  };

  // step 2 for row j: dx
  auto finish = [&](int64_t j, const Sum2& t, float mean, float rstd) {
    const float a = t.s1 * p.inv_cols;
    const float b = t.s2 * p.inv_cols;
    char* ds = const_cast<char*>(rw.slice(p.dx, rp.row(j), E));
#pragma unroll
    for (int q = 0; q < NQB; ++q) {
      if (q < rw.nq) {
        float o[W];
        if (rstd == 0.f) {
#pragma unroll
          for (int e = 0; e < W; ++e) o[e] = 0.f;
        } else {
          float dv[W], gv[W], hv[W];
          load_gx(j, q, mean, rstd, dv, gv, hv);
#pragma unroll
          for (int e = 0; e < W; e += 2) {
            float t0, t1;
            add2(t0, t1, gv[e], gv[e + 1], -a, -a);                // g - a
            fma2(t0, t1, hv[e], hv[e + 1], -b, -b, t0, t1);        // (g - a) - xhat b
            mul2(o[e], o[e + 1], t0, t1, rstd, rstd);
          }
        }
        lnx_store<DT, W>(ds, gt + q * G, q, rw, o);
      }
    }
  };

  // row statistics: rows j - 1 (finish) and j (step 1), one row ahead loaded
  float pm = 0.f, pr = 0.f, cm = 0.f, cr = 0.f, nm = 0.f, nr = 0.f;
  if (rw.first < g.rows) {
    if constexpr (!RMS) nm = __ldg(p.mean + rw.first);
    nr = __ldg(p.rstd + rw.first);
  }
  int64_t j = 0;
  for (;; ++j) {
    if (rp.row(j) >= g.rows) break;
    cm = nm;
    cr = nr;
    if (rp.row(j + 1) < g.rows) {
      if constexpr (!RMS) nm = __ldg(p.mean + rp.row(j + 1));
      nr = __ldg(p.rstd + rp.row(j + 1));
    }
    rp.fetch(j + rp.ahead, g.rows, src);
    rp.landed();
    const Sum2 t = partial(j, cm, cr);
    if (rp.solo) {
      finish(j, group_reduce<Sum2, MergeSum2, 32>(t, MergeSum2()), cm, cr);
    } else {
      Sum2 prev{};
      if (j >= 1) prev = rp.template merged<Sum2, MergeSum2>(j - 1, dead, p.err);
      rp.template publish<Sum2, MergeSum2>(j, t);
      if (j >= 1) finish(j - 1, prev, pm, pr);
    }
    pm = cm;
    pr = cr;
  }
  if (!rp.solo && j >= 1) finish(j - 1, rp.template merged<Sum2, MergeSum2>(j - 1, dead, p.err), pm, pr);
  cp_async_wait<0>();
  if constexpr (CL) cluster_sync();  // no peer still reads or writes this block's slots

  // The block's partial row: every group writes its partials into its own
  // ring (free now: local index i = k * W + e is column col0 + i), then the
  // groups' values are added in group order.  A cluster's ranks each write
  // their columns of the cluster's row.
  __syncthreads();
  float* mine = reinterpret_cast<float*>(rp.ring);
  const int SW = g.S * W;
#pragma unroll
  for (int q = 0; q < NQB; ++q) {
    if (q < rw.nq) {
      const int k = gt + q * G;
#pragma unroll
      for (int e = 0; e < W; ++e) {
        mine[k * W + e] = ag[q][e];
        if constexpr (!RMS) mine[SW + k * W + e] = ab[q][e];
      }
    }
  }
  __syncthreads();
  const int R = static_cast<int>(blockDim.x) / G;
  const int64_t owner = blockIdx.x / rp.K;
  float* out = p.ws + owner * kPlanes * g.cols;
  const size_t gstride = (size_t)g.NS * 2 * g.S * 4;  // floats in one group's ring
  const float* all = reinterpret_cast<const float*>(smem + g.ring_off);
  for (int i = threadIdx.x; i < kPlanes * SW; i += blockDim.x) {
    const int half = i >= SW ? 1 : 0;
    const int c = col0 + (i - half * SW);
    if (c < 0 || c >= g.cols) continue;
    float t = 0.f;
    for (int gi = 0; gi < R; ++gi) t += all[gi * gstride + i];
    out[(int64_t)half * g.cols + c] = t;
  }
}

template <int DT>
LnpKernels make_lnp_fwd_set() {
  LnpKernels s{};
  s.fwd[0][0] = (const void*)lnp_fwd_kernel<DT, false, false>;
  s.fwd[0][1] = (const void*)lnp_fwd_kernel<DT, false, true>;
  s.fwd[1][0] = (const void*)lnp_fwd_kernel<DT, true, false>;
  s.fwd[1][1] = (const void*)lnp_fwd_kernel<DT, true, true>;
  return s;
}
template <int DT, int NQB>
LnpKernels make_lnp_bwd_set() {
  LnpKernels s{};
  s.bwd[0][0] = (const void*)lnp_bwd_kernel<DT, NQB, false, false>;
  s.bwd[0][1] = (const void*)lnp_bwd_kernel<DT, NQB, false, true>;
  s.bwd[1][0] = (const void*)lnp_bwd_kernel<DT, NQB, true, false>;
  s.bwd[1][1] = (const void*)lnp_bwd_kernel<DT, NQB, true, true>;
  s.bwd2[0] = (const void*)lnp_bwd_kernel<DT, NQB, false, false, 2>;
  s.bwd2[1] = (const void*)lnp_bwd_kernel<DT, NQB, true, false, 2>;
  s.nq_bwd = NQB;
  return s;
}

}  // namespace rr
