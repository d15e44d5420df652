// rr_smb.cuh -- softmax / log-softmax backward for long rows, on the
// phase-class row layout and the row pipeline of rr_lnp.cuh (vector-Jacobian
// products of the softmax layer of "NexusGrad", Current main layer stack; the
// forward is sec. 3.1 of "Engineering a CUDA Machine Learning Framework from
// Scratch", sec. 2.3 for the 128-bit accesses).
//
// Per row, from the forward output (y, or z for the log-softmax) and the
// upstream gradient dy, both brought into shared memory by each thread's own
// asynchronous copies of its chunks:
//   softmax:      S = sum y * dy,  dx = y * (dy - S)
//   log-softmax:  S = sum dz,      dx = dz - 2^(z log2 e) * S
// S is summed with compensation (TwoSum) and merged as a double-float, so it
// is S rounded once.
// Lanes of the first and last chunk that belong to the neighbouring rows read
// as 0 in both tensors, so they add nothing to S; they are not stored.  The
// per-thread sums are merged over the warp (one warp per row) or, pipelined,
// over the group and the cluster (rr_lnp.cuh, RowPipe).  dx may be either
// input exactly: a row is in shared memory before any of its dx is written.
#pragma once

#include "rr_lnp.cuh"

namespace rr {

template <int DT, bool LOG, bool CL>
__global__ void __launch_bounds__(kSmxMaxT, 1) smb_kernel(const SoftmaxBwdParams p, const LnxGeo g) {
  constexpr int E = DType<DT>::E, W = DType<DT>::V;
  extern __shared__ __align__(128) unsigned char smem[];
  RowPipe<W, 2, CL> rp;
  rp.init(g, smem, p.y, E);
  const LnxRows<W>& rw = rp.rw;
  const int gt = rp.gr.gt, G = rp.gr.G;
  auto src = [&](int t, int64_t r) { return rw.slice(t == 0 ? p.y : p.dy, r, E); };
  for (int i = 0; i < rp.ahead; ++i) rp.fetch(i, g.rows, src);
  if constexpr (CL) cluster_sync();  // barriers set up before any peer arrives
  else __syncthreads();
  bool dead = false;

  // step 1 for row j: this thread's part of S, compensated (two TwoSum
  // accumulators per packed pair); an fp32 sum of thousands of terms can be off
  // by more than the fp32 tolerance where dx = dz - S (z = 0)
  auto partial = [&](int64_t j) -> DFSum {
    uint4* sy = rp.stage(j, 0);
    uint4* sd = rp.stage(j, 1);
    lnx_mask_stage<W>(sy, rw, gt, G, E);
    lnx_mask_stage<W>(sd, rw, gt, G, E);
    float s0 = 0.f, s1 = 0.f, c0 = 0.f, c1 = 0.f;
#pragma unroll 2
    for (int q = 0; q < rw.nq; ++q) {
      const int k = gt + q * G;
      float v[W];
      lnx_unpack<DT, W>(sd[k], v);
      if constexpr (!LOG) {
        float y[W];
        lnx_unpack<DT, W>(sy[k], y);
#pragma unroll
        for (int e = 0; e < W; e += 2) mul2(v[e], v[e + 1], v[e], v[e + 1], y[e], y[e + 1]);
      }
#pragma unroll
      for (int e = 0; e < W; e += 2) {
        float t0, t1, b0, b1, u0, u1, w0, w1;
        add2(t0, t1, s0, s1, v[e], v[e + 1]);  // t = s + v
        add2(b0, b1, t0, t1, -s0, -s1);        // bb = t - s
        add2(u0, u1, t0, t1, -b0, -b1);        // t - bb
        add2(u0, u1, s0, s1, -u0, -u1);        // s - (t - bb)
        add2(w0, w1, v[e], v[e + 1], -b0, -b1);  // v - bb
        add2(u0, u1, u0, u1, w0, w1);          // the exact error of s + v
        add2(c0, c1, c0, c1, u0, u1);
        s0 = t0;
        s1 = t1;
      }
    }
    float sh, e;
    two_sum(s0, s1, sh, e);
    return DFSum{sh, (c0 + c1) + e};
  };

  // step 2 for row j: dx
  auto finish = [&](int64_t j, const DFSum& t) {
    const float S = t.sh + t.sl;
    const uint4* sy = rp.stage(j, 0);
    const uint4* sd = rp.stage(j, 1);
    char* xs = const_cast<char*>(rw.slice(p.dx, rp.row(j), E));
#pragma unroll 2
    for (int q = 0; q < rw.nq; ++q) {
      const int k = gt + q * G;
      float y[W], d[W], f[W];
      lnx_unpack<DT, W>(sy[k], y);
      lnx_unpack<DT, W>(sd[k], d);
#pragma unroll
      for (int e = 0; e < W; e += 2) {
        if constexpr (LOG) {
          float t0, t1;
          mul2(t0, t1, y[e], y[e + 1], kLog2e, kLog2e);
          fma2(f[e], f[e + 1], ex2(t0), ex2(t1), -S, -S, d[e], d[e + 1]);
        } else {
          float t0, t1;
          add2(t0, t1, d[e], d[e + 1], -S, -S);
          mul2(f[e], f[e + 1], y[e], y[e + 1], t0, t1);
        }
      }
      lnx_store<DT, W>(xs, k, q, rw, f);
    }
  };

  int64_t j = 0;
  for (;; ++j) {
    if (rp.row(j) >= g.rows) break;
    rp.fetch(j + rp.ahead, g.rows, src);
    rp.landed();
    const DFSum t = partial(j);
    if (rp.solo) {
      finish(j, group_reduce<DFSum, MergeDF, 32>(t, MergeDF()));
    } else {
      DFSum prev{};
      if (j >= 1) prev = rp.template merged<DFSum, MergeDF>(j - 1, dead, p.err);
      rp.template publish<DFSum, MergeDF>(j, t);
      if (j >= 1) finish(j - 1, prev);
    }
  }
  if (!rp.solo && j >= 1) finish(j - 1, rp.template merged<DFSum, MergeDF>(j - 1, dead, p.err));
  cp_async_wait<0>();
  if constexpr (CL) cluster_sync();  // no peer still writes this block's slots
}

template <int DT>
SmbKernels make_smb_set() {
  SmbKernels s{};
  s.k[0][0] = (const void*)smb_kernel<DT, false, false>;
  s.k[0][1] = (const void*)smb_kernel<DT, false, true>;
  s.k[1][0] = (const void*)smb_kernel<DT, true, false>;
  s.k[1][1] = (const void*)smb_kernel<DT, true, true>;
  return s;
}

}  // namespace rr
