// rr_lnx.cuh -- LayerNorm / RMSNorm forward and backward for long rows, on
// memory-aligned 16-byte chunks ("Engineering a CUDA Machine Learning
// Framework from Scratch", sec. 3.2 for the one-pass moments, sec. 2.2 for the
// analytic backward, sec. 2.3 for the 128-bit accesses).
//
// A row of C elements starts at byte (base + r * C * E) mod 16 of its first
// 16-byte chunk.  That phase repeats every P rows (P = 16 / gcd(16, C * E mod
// 16), at most 8), so the rows fall into P classes whose rows all start at the
// same phase.  Each block (or cluster of blocks) works on the rows of one class
// only, which makes every chunk of every row it touches an aligned 16-byte
// block at the same place relative to the row: lane e of chunk k of a row is
// column k * W + e - phi (W values per chunk, phi the row's start offset in
// elements).  So:
//   - a row (a slice of it, for a cluster) is brought into shared memory by one
//     1-D bulk copy (TMA) of the aligned chunks covering it, several rows
//     ahead through a ring of stages completed on mbarriers;
//   - gamma / beta are staged once per block, shifted by phi, as fp32;
//   - every store of an interior chunk is one aligned 128-bit store, and only
//     the first and last chunk of a row (which the neighbouring rows share)
//     are written lane by lane.
// A block holds R row groups of G threads (G a multiple of 32); each group
// works on its own rows of the class with its own ring and named barrier, and
// the groups share gamma / beta and (backward) the block's column partials.
// Thread gt of a group owns local chunks k = gt + q * G (q < NQ) of its rows,
// held unpacked in fp32 registers for the whole row.  Lanes of the first and
// last chunk that belong to the neighbouring rows are zeroed in the stage
// before they are read.
//
// The copies read whole aligned 16-byte chunks, so the first (last) row of a
// tensor whose base (end) is not 16-byte aligned reads up to 15 bytes before
// (after) the tensor: always in the same 16-byte block as a byte of the
// tensor, so on a mapped page; those bytes are never used or written.
//
// Moments (forward): an exact mean from compensated (TwoSum) sums merged as
// double-floats over the group and the cluster, then the squared deviations
// about it; rstd = 1 / sqrt(M2 / C + eps).  A row with a non-finite mean or
// variance is masked (y = 0, mean = rstd = 0).  RMSNorm: the mean square.
// Backward: S1 = sum g, S2 = sum g * xhat (g = dy * gamma rounded once), then
// dx = rstd * ((g - S1/C) - xhat * S2/C); each thread's column partials
// (sum dy * xhat, sum dy) stay in registers across all its rows (a block's
// columns never change: one phase); at the end the block's groups add theirs
// in a fixed order into the block's (or cluster's) partial row of the
// workspace, which col_reduce_kernel sums.
#pragma once

#include "rr_kernels.h"
#include "rr_ln.cuh"

namespace rr {

// Launch geometry (host-computed).
struct LnxGeo {
  int64_t rows;
  int32_t cols;
  int32_t P;         // phase classes
  int32_t bpc;       // blocks (or clusters of blocks) per class
  int32_t S;         // chunks per cluster rank (>= chunks of a row when K == 1)
  int32_t NS;        // stages of each group's row ring
  int32_t G;         // threads per row group
  int32_t g_off;     // gamma (, beta) fp32 planes: [vectors][W / 4][S][4]
  int32_t red_off;   // reduction slots: [R][2 parities][32 warps][16 bytes]
  int32_t bar_off;   // mbarriers: [R][NS]
  int32_t ring_off;  // rings: [R][NS][tensors][S] 16-byte chunks
  int32_t cl_off;    // cluster exchange slots: 2 parities x 16 bytes
};

// Register budget: 512-thread blocks (at most 128 registers a thread).
constexpr int kLnxMaxT = 512;

// The row group a thread belongs to.
struct LnxGroup {
  int grp, gt, G, nw, nwp;  // group, thread in group, threads, warps, warps rounded to 2^k
  __device__ __forceinline__ void init(int G_) {
    G = G_;
    grp = threadIdx.x / G;
    gt = threadIdx.x - grp * G;
    nw = G >> 5;
    nwp = 1;
    while (nwp < nw) nwp <<= 1;
  }
  __device__ __forceinline__ void sync() const {
    if (nw > 1) named_bar(1 + grp, G);
    else __syncwarp();
  }
};

// Group-wide reduction of one statistic per row: a butterfly within each
// warp, the warps' results through shared memory after the group's barrier,
// and a butterfly over those (lane l reads warp l mod nwp, the missing warps
// read as the identity), so every thread ends with the same bits.  Slots
// alternate by call parity: a slot is rewritten two calls later, after a
// barrier that every reader of it has passed.
template <class S, class M>
__device__ __forceinline__ S lnx_reduce(S s, M merge, unsigned char* slots, int& calls,
                                        const LnxGroup& gr) {
  s = group_reduce<S, M, 32>(s, merge);
  if (gr.nw == 1) return s;
  unsigned char* base = slots + (calls & 1) * 512;
  ++calls;
  const int lane = threadIdx.x & 31;
  if (lane == 0) *reinterpret_cast<S*>(base + 16 * (gr.gt >> 5)) = s;
  gr.sync();
  const int w = lane & (gr.nwp - 1);
  S o = w < gr.nw ? *reinterpret_cast<const S*>(base + 16 * w) : S::identity();
  for (int off = gr.nwp / 2; off >= 1; off >>= 1) {
    const S t = S::shfl_xor(o, off);
    o = (lane & off) ? merge(t, o) : merge(o, t);
  }
  return o;
}

// A group's view of its phase class: its rows, their phase, the chunks of
// this rank's slice, and the partial chunks this thread holds.
template <int W>
struct LnxRows {
  int64_t first, step;  // rows first, first + step, ... (< rows)
  int phi;              // row start offset within its first chunk, in elements
  int nch;              // chunks covering a row
  int k0, n;            // this rank's slice: chunks [k0, k0 + n) of the row
  int nq;               // chunks this thread owns (gt + q * G < n)
  int tail_lanes;       // valid lanes of the row's last chunk (1 .. W)
  int hq, tq;           // q of this thread's head / tail chunk, -1 if none
  int64_t rowb;         // bytes per row

  __device__ __forceinline__ void init(const LnxGeo& g, const LnxGroup& gr, int R,
                                       const char* base, int E, int K, int rank) {
    const int owner = static_cast<int>(blockIdx.x) / K;
    const int cls = owner % g.P, j = owner / g.P;
    first = cls + (int64_t)g.P * ((int64_t)j * R + gr.grp);
    step = (int64_t)g.P * g.bpc * R;
    rowb = (int64_t)g.cols * E;
    phi = static_cast<int>(((reinterpret_cast<uintptr_t>(base) + (uint64_t)cls * rowb) & 15) / E);
    nch = (phi + g.cols + W - 1) / W;
    tail_lanes = phi + g.cols - W * (nch - 1);
    k0 = rank * g.S;
    n = min(g.S, nch - k0);
    nq = gr.gt < n ? (n - gr.gt + gr.G - 1) / gr.G : 0;
    hq = (rank == 0 && gr.gt == 0 && phi > 0) ? 0 : -1;
    const int kt = nch - 1 - k0;  // the row's last chunk, local index
    tq = (tail_lanes < W && kt >= 0 && kt < n && kt % gr.G == gr.gt) ? kt / gr.G : -1;
  }
  // Aligned address of the first chunk of this rank's slice of row r.
  __device__ __forceinline__ const char* slice(const char* base, int64_t r, int E) const {
    return base + r * rowb - (int64_t)phi * E + (int64_t)k0 * 16;
  }
};

// The bytes [lo, hi) of a 16-byte chunk kept, the rest cleared.
__device__ __forceinline__ uint4 lnx_byte_mask(int lo, int hi) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t m = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b)
      if (4 * i + b >= lo && 4 * i + b < hi) m |= 0xffu << (8 * b);
    w[i] = m;
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ void and16(uint4& c, const uint4& m) {
  c.x &= m.x;
  c.y &= m.y;
  c.z &= m.z;
  c.w &= m.w;
}

// Clears, in a landed stage (tensor base st), the lanes of this thread's head /
// tail chunk that belong to the neighbouring rows (zero bits are 0.0 in fp32
// and bf16), before the thread reads them: the chunks stay exact zeros in every
// sum.  Done in shared memory by the chunk's only reader, so the registers
// holding the row are never indexed by a run-time chunk number.
template <int W>
__device__ __forceinline__ void lnx_mask_stage(uint4* st, const LnxRows<W>& rw, int gt, int G,
                                               int E) {
  if (rw.hq == 0) and16(st[gt], lnx_byte_mask(rw.phi * E, 16));
  if (rw.tq >= 0) and16(st[gt + rw.tq * G], lnx_byte_mask(0, rw.tail_lanes * E));
}

template <int DT, int W>
__device__ __forceinline__ void lnx_unpack(const uint4& c, float (&f)[W]) {
#pragma unroll
  for (int e = 0; e < W; ++e) f[e] = chunk_get<DT>(c, e);
}

// Stores the thread's chunk q (local chunk k, W values) of a row slice: one
// aligned 128-bit store for an interior chunk, the row's own lanes one by one
// for the head / tail chunk.
template <int DT, int W>
__device__ __forceinline__ void lnx_store(char* sl, int k, int q, const LnxRows<W>& rw,
                                          const float (&f)[W]) {
  constexpr int E = DType<DT>::E;
  char* a = sl + (int64_t)k * 16;
  if (q != rw.hq && q != rw.tq) {
    st_chunk_stream(a, chunk_pack<DT>(f));
  } else {
    const int lo = q == rw.hq ? rw.phi : 0;
    const int hi = q == rw.tq ? rw.tail_lanes : W;
#pragma unroll
    for (int e = 0; e < W; ++e)
      if (e >= lo && e < hi) st_elem<DT>(a + e * E, f[e]);
  }
}

// gamma (src) shifted to the block's phase, as fp32 planes: plane p holds
// lanes 4p .. 4p + 3 of every local chunk (16 contiguous bytes per chunk), 0
// outside the row.  Local chunk k is the funnel shift of the two aligned
// 16-byte blocks of the vector that hold its columns; a thread loads up to 8
// chunks' blocks before using any; a block wholly outside the vector is not
// read (its lanes are columns outside the row).
template <int DT, int W>
__device__ __forceinline__ void lnx_stage_vec(float* planes, const char* src, int S, int cols,
                                              int col0) {
  constexpr int E = DType<DT>::E;
  constexpr int QB = 8;
  const uintptr_t v0 = reinterpret_cast<uintptr_t>(src);
  const uintptr_t v1 = v0 + (uintptr_t)cols * E;  // one past the vector
  for (int kb = threadIdx.x; kb < S; kb += QB * blockDim.x) {
    uint4 lo[QB], hi[QB];
#pragma unroll
    for (int i = 0; i < QB; ++i) {
      const int k = kb + i * blockDim.x;
      lo[i] = hi[i] = make_uint4(0u, 0u, 0u, 0u);
      if (k < S) {
        const uintptr_t a = v0 + (intptr_t)(col0 + k * W) * E;
        const uintptr_t b = a & ~uintptr_t(15);
        if (b + 16 > v0 && b < v1) lo[i] = ld_chunk_cached(reinterpret_cast<const char*>(b));
        if ((a & 15) != 0 && b + 32 > v0 && b + 16 < v1)
          hi[i] = ld_chunk_cached(reinterpret_cast<const char*>(b + 16));
      }
    }
#pragma unroll
    for (int i = 0; i < QB; ++i) {
      const int k = kb + i * blockDim.x;
      if (k < S) {
        const uintptr_t a = v0 + (intptr_t)(col0 + k * W) * E;
        const uint4 c = funnel16(lo[i], hi[i], static_cast<int>(a & 15));
        float f[W];
#pragma unroll
        for (int e = 0; e < W; ++e) {
          const int col = col0 + k * W + e;
          f[e] = (col >= 0 && col < cols) ? chunk_get<DT>(c, e) : 0.f;
        }
#pragma unroll
        for (int p = 0; p < W / 4; ++p)
          *reinterpret_cast<float4*>(planes + p * S * 4 + k * 4) =
              make_float4(f[4 * p], f[4 * p + 1], f[4 * p + 2], f[4 * p + 3]);
      }
    }
  }
}
template <int W>
__device__ __forceinline__ void lnx_vec(const float* planes, int S, int k, float (&out)[W]) {
#pragma unroll
  for (int p = 0; p < W / 4; ++p) {
    const float4 t = *reinterpret_cast<const float4*>(planes + p * S * 4 + k * 4);
    out[4 * p] = t.x;
    out[4 * p + 1] = t.y;
    out[4 * p + 2] = t.z;
    out[4 * p + 3] = t.w;
  }
}

// A group's ring of row stages: its leader issues the bulk copies of a row
// into stage s (NT tensors), every thread of the group waits for the stage's
// phase.
template <int NT>
struct LnxRing {
  uint4* ring;
  uint64_t* bars;
  int S, NS;
  uint64_t policy;
  __device__ __forceinline__ uint4* stage(int s, int t) const {
    return ring + ((size_t)s * NT + t) * S;
  }
  __device__ __forceinline__ void issue(int s, const char* const (&src)[NT], int n) const {
    const uint32_t bytes = static_cast<uint32_t>(n) * 16;
    fence_proxy_async_smem();  // earlier generic reads of the stage come first
    mbar_arrive_expect_tx(&bars[s], bytes * NT);
#pragma unroll
    for (int t = 0; t < NT; ++t) bulk_load(stage(s, t), src[t], bytes, &bars[s], policy);
  }
};

// After a wait gave up: waits (bounded, 0.1 s each) for the last copy issued
// into each stage, so no bulk copy is still writing this block's shared memory
// when it exits.  Rows 0 .. nit - 1 of the group were issued, row i into
// stage i % NS.
__device__ __forceinline__ void lnx_drain(uint64_t* bars, int NS, int64_t nit, int* err) {
  for (int s = 0; s < NS; ++s) {
    if (nit <= s) continue;
    const int64_t last = s + ((nit - 1 - s) / NS) * NS;
    mbar_wait_bounded(&bars[s], static_cast<uint32_t>((last / NS) & 1), err, 100000000ull);
  }
}

// Set-up shared by the long-row kernels: the group's ring; its leader
// initialises the ring's barriers and starts the copies of the group's first
// nfirst rows (default NS - 1; issue(i) copies the group's row i into stage
// i % NS).  The other threads touch the barriers only after the block's next
// __syncthreads.
template <int NT, int W, class Issue>
__device__ __forceinline__ void lnx_start(const LnxGeo& g, unsigned char* smem, const LnxGroup& gr,
                                          const LnxRows<W>& rw, LnxRing<NT>& ring, Issue issue,
                                          int nfirst = -1) {
  ring.ring = reinterpret_cast<uint4*>(smem + g.ring_off) + (size_t)gr.grp * g.NS * NT * g.S;
  ring.bars = reinterpret_cast<uint64_t*>(smem + g.bar_off) + (size_t)gr.grp * g.NS;
  ring.S = g.S;
  ring.NS = g.NS;
  ring.policy = policy_evict_first();
  if (gr.gt == 0) {
    for (int s = 0; s < g.NS; ++s) mbar_init(&ring.bars[s], 1);
    fence_mbar_init();
    const int n0 = nfirst < 0 ? g.NS - 1 : nfirst;
    for (int s = 0; s < n0; ++s)
      if (rw.first + s * rw.step < g.rows) issue(s);
  }
}

// ------------------------------------------------------------ forward ------
template <int DT, int NQ, bool RMS, bool CL>
__global__ void __launch_bounds__(kLnxMaxT, 1) lnx_fwd_kernel(const LnFwdParams p, const LnxGeo g) {
  constexpr int E = DType<DT>::E, W = DType<DT>::V;
  extern __shared__ __align__(128) unsigned char smem[];
  int K = 1, rank = 0;
  if constexpr (CL) {
    K = static_cast<int>(cluster_nrank());
    rank = static_cast<int>(cluster_rank());
  }
  LnxGroup gr;
  gr.init(g.G);
  const int R = static_cast<int>(blockDim.x) / g.G;
  LnxRows<W> rw;
  rw.init(g, gr, R, p.x, E, K, rank);
  auto row_of = [&](int64_t it) { return rw.first + it * rw.step; };
  LnxRing<1> ring;
  lnx_start<1, W>(g, smem, gr, rw, ring, [&](int64_t it) {
    const char* src[1] = {rw.slice(p.x, row_of(it), E)};
    ring.issue(static_cast<int>(it % g.NS), src, rw.n);
  });
  float* gam = reinterpret_cast<float*>(smem + g.g_off);
  float* bet = gam + (size_t)g.S * W;
  const int col0 = rw.k0 * W - rw.phi;
  lnx_stage_vec<DT, W>(gam, p.gamma, g.S, g.cols, col0);
  if constexpr (!RMS) lnx_stage_vec<DT, W>(bet, p.beta, g.S, g.cols, col0);
  __syncthreads();
  unsigned char* red = smem + g.red_off + gr.grp * 1024;
  int rcalls = 0, ccalls = 0;
  bool dead = false;  // a wait gave up: later waits are skipped (the kernel still ends)
  const float ns = static_cast<float>(g.cols);

  int64_t it = 0;
  for (;; ++it) {
    const int64_t r = row_of(it);
    if (r >= g.rows) break;
    const int s = static_cast<int>(it % g.NS);
    // the stage the previous row used is free (every thread of the group
    // passed a barrier after reading it): refill it with the row NS - 1 ahead
    if (gr.gt == 0 && row_of(it + g.NS - 1) < g.rows) {
      const char* src[1] = {rw.slice(p.x, row_of(it + g.NS - 1), E)};
      ring.issue(static_cast<int>((it + g.NS - 1) % g.NS), src, rw.n);
    }
    if (!dead) dead = !mbar_wait_bounded(&ring.bars[s], static_cast<uint32_t>((it / g.NS) & 1), p.err);
    float f[NQ][W];
    {
      uint4* st = ring.stage(s, 0);
      lnx_mask_stage<W>(st, rw, gr.gt, gr.G, E);
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        const uint4 c = q < rw.nq ? st[gr.gt + q * gr.G] : make_uint4(0u, 0u, 0u, 0u);
        lnx_unpack<DT, W>(c, f[q]);
      }
    }

    float mh = 0.f, ml = 0.f, rstd;
    bool masked;
    if constexpr (RMS) {
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int q = 0; q < NQ; ++q)
        if (q < rw.nq) {
#pragma unroll
          for (int e = 0; e < W; e += 2)
            fma2(a0, a1, f[q][e], f[q][e + 1], f[q][e], f[q][e + 1], a0, a1);
        }
      Sum1 t = lnx_reduce(Sum1{a0 + a1}, MergeSum1(), red, rcalls, gr);
      if constexpr (CL) t = ln_cluster(t, MergeSum1(), smem + g.cl_off, ccalls, K);
      const float ms = t.s * p.inv_cols;
      masked = !isfinite(ms);
      rstd = masked ? 0.f : rsqrtf(ms + p.eps);
      if (gr.gt == 0 && rank == 0) p.rstd[r] = rstd;
    } else {
      // 1. compensated sum (two interleaved TwoSum accumulators per packed pair)
      float s0 = 0.f, s1 = 0.f, c0 = 0.f, c1 = 0.f;
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        if (q < rw.nq) {
#pragma unroll
          for (int e = 0; e < W; e += 2) {
            const float v0 = f[q][e], v1 = f[q][e + 1];
            float t0, t1, b0, b1, u0, u1, w0, w1;
            add2(t0, t1, s0, s1, v0, v1);     // t = s + v
            add2(b0, b1, t0, t1, -s0, -s1);   // bb = t - s
            add2(u0, u1, t0, t1, -b0, -b1);   // t - bb
            add2(u0, u1, s0, s1, -u0, -u1);   // s - (t - bb)
            add2(w0, w1, v0, v1, -b0, -b1);   // v - bb
            add2(u0, u1, u0, u1, w0, w1);     // exact error of s + v
            add2(c0, c1, c0, c1, u0, u1);
            s0 = t0;
            s1 = t1;
          }
        }
      }
      CascSum S;
      {
        float sh, e;
        two_sum(s0, s1, sh, e);
        S = {sh, (c0 + c1) + e};
      }
      S = lnx_reduce(S, MergeCasc(), red, rcalls, gr);
      if constexpr (CL) S = ln_cluster(S, MergeCasc(), smem + g.cl_off, ccalls, K);
      {
        float sh, sl;
        two_sum(S.s, S.e, sh, sl);
        df_mean(sh, sl, ns, p.inv_cols, mh, ml);
      }
      // 2. squared deviations about the exact mean (other rows' lanes excluded)
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        if (q < rw.nq) {
          float d[W];
#pragma unroll
          for (int e = 0; e < W; e += 2) {
            add2(d[e], d[e + 1], f[q][e], f[q][e + 1], -mh, -mh);
            add2(d[e], d[e + 1], d[e], d[e + 1], -ml, -ml);
          }
          if (q == rw.hq || q == rw.tq) {
            const int lo = q == rw.hq ? rw.phi : 0;
            const int hi = q == rw.tq ? rw.tail_lanes : W;
#pragma unroll
            for (int e = 0; e < W; ++e)
              if (e < lo || e >= hi) d[e] = 0.f;
          }
#pragma unroll
          for (int e = 0; e < W; e += 2) fma2(a0, a1, d[e], d[e + 1], d[e], d[e + 1], a0, a1);
        }
      }
      Sum1 t = lnx_reduce(Sum1{a0 + a1}, MergeSum1(), red, rcalls, gr);
      if constexpr (CL) t = ln_cluster(t, MergeSum1(), smem + g.cl_off, ccalls, K);
      const float var = t.s * p.inv_cols;
      masked = !(isfinite(mh) && isfinite(ml) && isfinite(var));
      rstd = masked ? 0.f : rsqrtf(var + p.eps);
      if (gr.gt == 0 && rank == 0) {
        p.mean[r] = masked ? 0.f : mh + ml;
        p.rstd[r] = rstd;
      }
    }

    // 3. y = ((x - mh) - ml) * rstd * gamma + beta   (RMSNorm: x * rstd * gamma)
    char* ys = const_cast<char*>(rw.slice(p.y, r, E));
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      if (q < rw.nq) {
        const int k = gr.gt + q * gr.G;
        float y[W];
        if (masked) {
#pragma unroll
          for (int e = 0; e < W; ++e) y[e] = 0.f;
        } else {
          float gm[W];
          lnx_vec<W>(gam, g.S, k, gm);
          if constexpr (RMS) {
#pragma unroll
            for (int e = 0; e < W; e += 2) {
              float t0, t1;
              mul2(t0, t1, f[q][e], f[q][e + 1], rstd, rstd);
              mul2(y[e], y[e + 1], t0, t1, gm[e], gm[e + 1]);
            }
          } else {
            float bt[W];
            lnx_vec<W>(bet, g.S, k, bt);
#pragma unroll
            for (int e = 0; e < W; e += 2) {
              float t0, t1;
              add2(t0, t1, f[q][e], f[q][e + 1], -mh, -mh);
              add2(t0, t1, t0, t1, -ml, -ml);
              mul2(t0, t1, t0, t1, rstd, rstd);
              fma2(y[e], y[e + 1], t0, t1, gm[e], gm[e + 1], bt[e], bt[e + 1]);
            }
          }
        }
        lnx_store<DT, W>(ys, k, q, rw, y);
      }
    }
    // the refill at the top of the next row overwrites stage (it % NS) only
    // after every thread of the group has read it: RMSNorm (one reduction) and
    // one-warp groups may have passed no barrier since reading it
    if (RMS || gr.nw == 1) gr.sync();
  }
  if (dead) lnx_drain(ring.bars, g.NS, it, p.err);
  if constexpr (CL) cluster_sync();  // peers may still read this block's slots
}

// ----------------------------------------------------------- backward ------
// MINB = 2: blocks of at most 320 threads, two per SM (96 registers a thread).
template <int DT, int NQ, bool RMS, bool CL, int MINB = 1>
__global__ void __launch_bounds__(MINB == 2 ? 320 : kLnxMaxT, MINB)
    lnx_bwd_kernel(const LnBwdParams p, const LnxGeo g) {
  constexpr int E = DType<DT>::E, W = DType<DT>::V;
  constexpr int kPlanes = RMS ? 1 : 2;
  extern __shared__ __align__(128) unsigned char smem[];
  int K = 1, rank = 0;
  if constexpr (CL) {
    K = static_cast<int>(cluster_nrank());
    rank = static_cast<int>(cluster_rank());
  }
  LnxGroup gr;
  gr.init(g.G);
  const int R = static_cast<int>(blockDim.x) / g.G;
  LnxRows<W> rw;
  rw.init(g, gr, R, p.x, E, K, rank);
  auto row_of = [&](int64_t it) { return rw.first + it * rw.step; };
  LnxRing<2> ring;
  auto issue = [&](int64_t it) {
    const int64_t rr = row_of(it);
    const char* src[2] = {rw.slice(p.dy, rr, E), rw.slice(p.x, rr, E)};
    ring.issue(static_cast<int>(it % g.NS), src, rw.n);
  };
  lnx_start<2, W>(g, smem, gr, rw, ring, issue);
  float* gam = reinterpret_cast<float*>(smem + g.g_off);
  const int col0 = rw.k0 * W - rw.phi;
  lnx_stage_vec<DT, W>(gam, p.gamma, g.S, g.cols, col0);
  __syncthreads();
  unsigned char* red = smem + g.red_off + gr.grp * 1024;
  int rcalls = 0, ccalls = 0;
  bool dead = false;

  // column partials of this thread's chunks: sum dy * xhat (, sum dy)
  float ag[NQ][W], ab[NQ][W];
#pragma unroll
  for (int q = 0; q < NQ; ++q)
#pragma unroll
    for (int e = 0; e < W; ++e) ag[q][e] = ab[q][e] = 0.f;

  // row statistics one row ahead
  float nmean = 0.f, nrstd = 0.f;
  if (rw.first < g.rows) {
    if constexpr (!RMS) nmean = __ldg(p.mean + rw.first);
    nrstd = __ldg(p.rstd + rw.first);
  }
  int64_t it = 0;
  for (;; ++it) {
    const int64_t r = row_of(it);
    if (r >= g.rows) break;
    const int s = static_cast<int>(it % g.NS);
    const float mean = nmean, rstd = nrstd;
    {
      const int64_t rn = row_of(it + 1);
      if (rn < g.rows) {
        if constexpr (!RMS) nmean = __ldg(p.mean + rn);
        nrstd = __ldg(p.rstd + rn);
      }
    }
    if (gr.gt == 0 && row_of(it + g.NS - 1) < g.rows) issue(it + g.NS - 1);
    if (!dead) dead = !mbar_wait_bounded(&ring.bars[s], static_cast<uint32_t>((it / g.NS) & 1), p.err);
    const bool use = rstd != 0.f;
    float gv[NQ][W], hv[NQ][W];
    float s1a = 0.f, s1b = 0.f, s2a = 0.f, s2b = 0.f;
    {
      float dv[NQ][W], xv[NQ][W];
      uint4* sd = ring.stage(s, 0);
      uint4* sx = ring.stage(s, 1);
      lnx_mask_stage<W>(sd, rw, gr.gt, gr.G, E);
      lnx_mask_stage<W>(sx, rw, gr.gt, gr.G, E);
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        const bool in = q < rw.nq;
        const int k = gr.gt + q * gr.G;
        lnx_unpack<DT, W>(in ? sd[k] : make_uint4(0u, 0u, 0u, 0u), dv[q]);
        lnx_unpack<DT, W>(in ? sx[k] : make_uint4(0u, 0u, 0u, 0u), xv[q]);
      }
      if (use) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          if (q < rw.nq) {
            float gm[W];
            lnx_vec<W>(gam, g.S, gr.gt + q * gr.G, gm);
#pragma unroll
            for (int e = 0; e < W; e += 2) {
              const float y0 = dv[q][e], y1 = dv[q][e + 1];
              float h0, h1;
              if constexpr (RMS) {
                mul2(h0, h1, xv[q][e], xv[q][e + 1], rstd, rstd);
              } else {
                add2(h0, h1, xv[q][e], xv[q][e + 1], -mean, -mean);
                mul2(h0, h1, h0, h1, rstd, rstd);
              }
              // g rounded once (a product that must not fuse into the sums)
              const float g0 = __fmul_rn(y0, gm[e]), g1 = __fmul_rn(y1, gm[e + 1]);
              if constexpr (!RMS) add2(s1a, s1b, s1a, s1b, g0, g1);
              fma2(s2a, s2b, g0, g1, h0, h1, s2a, s2b);
              fma2(ag[q][e], ag[q][e + 1], y0, y1, h0, h1, ag[q][e], ag[q][e + 1]);
              if constexpr (!RMS) add2(ab[q][e], ab[q][e + 1], ab[q][e], ab[q][e + 1], y0, y1);
              gv[q][e] = g0;
              gv[q][e + 1] = g1;
              hv[q][e] = h0;
              hv[q][e + 1] = h1;
            }
          }
        }
      }
    }
    Sum2 sm = lnx_reduce(Sum2{s1a + s1b, s2a + s2b}, MergeSum2(), red, rcalls, gr);
    if constexpr (CL) sm = ln_cluster(sm, MergeSum2(), smem + g.cl_off, ccalls, K);
    const float a = sm.s1 * p.inv_cols;
    const float b = sm.s2 * p.inv_cols;
    char* ds = const_cast<char*>(rw.slice(p.dx, r, E));
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      if (q < rw.nq) {
        float o[W];
        if (!use) {
#pragma unroll
          for (int e = 0; e < W; ++e) o[e] = 0.f;
        } else {
#pragma unroll
          for (int e = 0; e < W; e += 2) {
            float t0, t1;
            add2(t0, t1, gv[q][e], gv[q][e + 1], -a, -a);             // g - a
            fma2(t0, t1, hv[q][e], hv[q][e + 1], -b, -b, t0, t1);     // (g - a) - xhat b
            mul2(o[e], o[e + 1], t0, t1, rstd, rstd);
          }
        }
        lnx_store<DT, W>(ds, gr.gt + q * gr.G, q, rw, o);
      }
    }
    if (gr.nw == 1) gr.sync();  // one-warp groups: no barrier since the stage was read
  }
  if (dead) lnx_drain(ring.bars, g.NS, it, p.err);
  if constexpr (CL) cluster_sync();  // peers may still read this block's slots

  // The block's partial row: every group writes its partials into its own
  // ring (free now: local index i = k * W + e is column col0 + i), then the
  // groups' values are added in group order.  A cluster's ranks each write
  // their columns of the cluster's row.
  gr.sync();
  float* mine = reinterpret_cast<float*>(ring.ring);
  const int SW = g.S * W;
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    if (q < rw.nq) {
      const int k = gr.gt + q * gr.G;
#pragma unroll
      for (int e = 0; e < W; ++e) {
        mine[k * W + e] = ag[q][e];
        if constexpr (!RMS) mine[SW + k * W + e] = ab[q][e];
      }
    }
  }
  __syncthreads();
  const int64_t owner = blockIdx.x / K;
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

template <int DT, int NQ>
LnxKernels make_lnx_fwd_set() {
  LnxKernels s{};
  s.fwd[0][0] = (const void*)lnx_fwd_kernel<DT, NQ, false, false>;
  s.fwd[0][1] = (const void*)lnx_fwd_kernel<DT, NQ, false, true>;
  s.fwd[1][0] = (const void*)lnx_fwd_kernel<DT, NQ, true, false>;
  s.fwd[1][1] = (const void*)lnx_fwd_kernel<DT, NQ, true, true>;
  s.nq_fwd = NQ;
  return s;
}
template <int DT, int NQ>
LnxKernels make_lnx_bwd_set() {
  LnxKernels s{};
  s.bwd[0][0] = (const void*)lnx_bwd_kernel<DT, NQ, false, false>;
  s.bwd[0][1] = (const void*)lnx_bwd_kernel<DT, NQ, false, true>;
  s.bwd[1][0] = (const void*)lnx_bwd_kernel<DT, NQ, true, false>;
  s.bwd[1][1] = (const void*)lnx_bwd_kernel<DT, NQ, true, true>;
  s.bwd2[0] = nullptr;  // measured slower (spills at 96 registers)
  s.bwd2[1] = (const void*)lnx_bwd_kernel<DT, NQ, true, false, 2>;
  s.nq_bwd = NQ;
  return s;
}

}  // namespace rr
