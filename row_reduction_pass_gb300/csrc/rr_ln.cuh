// rr_ln.cuh -- LayerNorm forward and backward on column-owned row groups
// ("Engineering a CUDA Machine Learning Framework from Scratch", sec. 3.2 for
// the one-pass moments, sec. 2.2 for the analytic backward).
//
// Rows that fit in the registers of one row group of G threads (G = 1 ..
// 1024) take these kernels.  Thread gt of a group owns the column-aligned
// chunks k = gt + q*G (q < NQ) of every row the group processes; a chunk is W
// columns (W = 16 bytes / element size, or one element in element mode).
// Which of its chunks are whole and whether it holds the row's ragged last
// chunk are therefore the same for every row and are worked out once per
// launch; gamma / beta are converted to fp32 once per block into shared
// memory; the backward keeps its per-column partial sums (sum_r dy*xhat and
// sum_r dy) in registers across all the rows a thread processes and writes
// them out once per block.
//
// RMS = true turns both kernels into RMSNorm (y = x * rstd * gamma with
// rstd = 1/sqrt(mean(x^2) + eps); no mean, no beta): the standard reading of the
// RMSNorm that the "NexusGrad" README lists among its transformer components.
//
// Ragged slots of the last chunk are loaded as 0: they add exactly nothing to
// the compensated sum, to sum dy*gamma, to sum dy*gamma*xhat (dy = 0 there) or
// to the column partials, so only the squared deviations and the stores mask
// them.
#pragma once

#include "rr_kernels.h"
#include "rr_ops.cuh"

namespace rr {

// Launch geometry of a row-group LayerNorm launch (host-computed).
struct LnGeo {
  int64_t rows;
  int32_t cols;
  int32_t nfull;    // whole chunks per row (cols / W)
  int32_t rag;      // elements of the ragged last chunk (0: none)
  int32_t nch;      // chunks per row
  int32_t red_off;  // group-reduction scratch (G > 32): 1 KB per group
  int32_t acc_off;  // backward: column partials, ngroups x 2 x (nch * W) floats
  int32_t pf_off;   // cp.async prefetch slots / row buffers
  int32_t slice;    // columns per block of a cluster (= cols without clusters)
  int32_t cl_off;   // cluster exchange slots (2 x 16 bytes)
};

// Register sizes.  Forward: 64 per thread at any block size.  Backward: up to
// 128 (a thread keeps g = dy*gamma, xhat and its two column accumulators), 64
// for the one-chunk variants of short rows.
template <int MAXT, int NQ = 4> constexpr int ln_fwd_min_blocks() {
  // more than 4 chunks per thread (the deep and the wide cluster variants):
  // up to 128 registers (64 for 1024-thread blocks)
  return NQ > 4 ? (MAXT >= 512 ? 1 : 2) : 1024 / MAXT;
}
template <int MAXT, int NQ> constexpr int ln_bwd_min_blocks() { return (NQ == 1 ? 1024 : 512) / MAXT; }

// A sum carried as a leading float s and an accumulated error e (cascaded
// summation in the manner of Ogita, Rump and Oishi's Sum2): a merge adds the
// leading parts with TwoSum and the rest in plain fp32, so the result is as
// accurate as a sum in twice the precision; renormalised once at the end.
struct CascSum {
  float s, e;
  __device__ __forceinline__ static CascSum identity() { return {0.f, 0.f}; }
  __device__ __forceinline__ static CascSum load_remote(uint32_t a) {
    return {ld_cluster_f32(a), ld_cluster_f32(a + 4)};
  }
  __device__ __forceinline__ static CascSum shfl_xor(const CascSum& v, int off) {
    return {__shfl_xor_sync(0xffffffffu, v.s, off), __shfl_xor_sync(0xffffffffu, v.e, off)};
  }
};
struct MergeCasc {
  __device__ __forceinline__ CascSum operator()(const CascSum& a, const CascSum& b) const {
    float s, err;
    two_sum(a.s, b.s, s, err);
    return {s, (a.e + b.e) + err};
  }
};

// Per-row reductions across a row group: G <= 32 lanes by an ordered
// butterfly; wider groups by a butterfly per warp, the warp results through
// shared memory (two slots per warp, alternating by call parity, so one named
// barrier per call suffices) and a butterfly over those G/32 values (lane l
// reads warp l mod G/32, so every aligned block of G/32 lanes holds them all).
// Every thread of the group ends with the same bits.
template <int G>
struct LnRed {
  unsigned char* slot;
  int calls;
  int bar;
  template <class S, class M>
  __device__ __forceinline__ S operator()(S s, M merge) {
    static_assert(sizeof(S) <= 16, "statistic larger than a scratch slot");
    if constexpr (G <= 32) {
      return group_reduce<S, M, G>(s, merge);
    } else {
      s = group_reduce<S, M, 32>(s, merge);
      unsigned char* base = slot + (calls & 1) * 512;
      ++calls;
      const int lane = threadIdx.x & 31;
      if (lane == 0) *reinterpret_cast<S*>(base + 16 * ((threadIdx.x % G) >> 5)) = s;
      named_bar(bar, G);
      const S o = *reinterpret_cast<const S*>(base + 16 * (lane & (G / 32 - 1)));
      return group_reduce<S, M, G / 32>(o, merge);
    }
  }
};

// A row split over the K <= 8 blocks of a cluster: each block's statistic
// (already reduced over its threads) goes to its exchange slot, and after a
// cluster barrier every thread reads the K slots (all loads issued before the
// first merge, so their remote latencies overlap) and merges them in rank
// order, so all blocks hold the same bits.  Slots alternate by call parity: a
// slot is rewritten two calls later, after the next barrier, which every
// reader of it has passed.
template <class S, class M>
__device__ __forceinline__ S ln_cluster(S s, M merge, unsigned char* slots, int& calls, int K) {
  S* slot = reinterpret_cast<S*>(slots + 16 * (calls & 1));
  ++calls;
  if (threadIdx.x == 0) *slot = s;
  cluster_sync();
  S v[8];
#pragma unroll
  for (int k = 0; k < 8; ++k)
    if (k < K) v[k] = S::load_remote(map_to_rank(slot, k));
  S acc = v[0];
#pragma unroll
  for (int k = 1; k < 8; ++k)
    if (k < K) acc = merge(acc, v[k]);
  return acc;
}

// The chunks of one thread: q < nf are whole, q < nown are owned (the ragged
// last chunk of the row, when this thread holds it, is q = nf).
template <int G, int NQ>
struct LnCols {
  int nf, nown;
  __device__ __forceinline__ void init(int gt, int nfull, int rag) {
    nf = nfull > gt ? (nfull - gt + G - 1) / G : 0;
    nf = nf < NQ ? nf : NQ;
    const bool rq = rag > 0 && nfull >= gt && (nfull - gt) % G == 0 && (nfull - gt) / G < NQ;
    nown = nf + (rq ? 1 : 0);
  }
};

template <int DT, int W>
__device__ __forceinline__ float ln_get(const uint4& c, int e) {
  if constexpr (W == 1) return bits_to_f32<DT>(c.x);
  else return chunk_get<DT>(c, e);
}

// Loads the thread's chunks of the row starting at rs (a tensor spanning
// [tb, te)).  AL: every row start is 16-byte aligned.  Otherwise a row whose
// start is not is read as the funnel shift of the two aligned chunks holding
// each of its chunks (neighbouring lanes share those through L1), or element by
// element where that pair would leave the tensor.
template <int DT, int W, int G, int NQ, bool AL>
__device__ __forceinline__ void ln_load(uint4 (&v)[NQ], const char* rs, int gt,
                                        const LnCols<G, NQ>& cs, int rag, const char* tb,
                                        const char* te) {
  constexpr int E = DType<DT>::E;
  if constexpr (W == 1) {
#pragma unroll
    for (int q = 0; q < NQ; ++q)
      v[q] = make_uint4(q < cs.nown ? ld_elem_bits<DT>(rs + (int64_t)(gt + q * G) * E) : 0u, 0u,
                        0u, 0u);
  } else {
    const uintptr_t ra = reinterpret_cast<uintptr_t>(rs);
    const int h = AL ? 0 : static_cast<int>(ra & 15);
    bool split = false;
    if constexpr (!AL) {
      if (h != 0 && cs.nf > 0) {
        const uintptr_t lo = (ra + (uintptr_t)gt * 16) & ~uintptr_t(15);
        const uintptr_t hi = ((ra + (uintptr_t)(gt + (cs.nf - 1) * G) * 16) & ~uintptr_t(15)) + 32;
        split = lo >= reinterpret_cast<uintptr_t>(tb) && hi <= reinterpret_cast<uintptr_t>(te);
      }
    }
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      const char* a = rs + (int64_t)(gt + q * G) * 16;
      uint4 c = make_uint4(0u, 0u, 0u, 0u);
      if (q < cs.nf) {
        if (AL || h == 0) {
          c = ld_chunk_stream(a);
        } else if (split) {
          c = ld16_split(a);
        } else {
#pragma unroll
          for (int e = 0; e < W; ++e) chunk_set_bits<DT>(c, e, ld_elem_bits<DT>(a + e * E));
        }
      } else if (q < cs.nown) {
#pragma unroll
        for (int e = 0; e < W; ++e)
          if (e < rag) chunk_set_bits<DT>(c, e, ld_elem_bits<DT>(a + e * E));
      }
      v[q] = c;
    }
  }
}

// Stores chunk q (W values f) of the row starting at rs: whole chunks as one
// 128-bit store when the row start is aligned, else as aligned pieces; the
// ragged chunk element by element.
template <int DT, int W, int G, int NQ, bool AL>
__device__ __forceinline__ void ln_store(char* rs, int gt, int q, const LnCols<G, NQ>& cs,
                                         int rag, const float (&f)[W]) {
  constexpr int E = DType<DT>::E;
  if constexpr (W == 1) {
    st_elem<DT>(rs + (int64_t)(gt + q * G) * E, f[0]);
  } else {
    char* a = rs + (int64_t)(gt + q * G) * 16;
    if (q < cs.nf) {
      const uint4 c = chunk_pack<DT>(f);
      if (AL || (reinterpret_cast<uintptr_t>(rs) & 15) == 0) st_chunk_stream(a, c);
      else st16_split(a, c);
    } else {
#pragma unroll
      for (int e = 0; e < W; ++e)
        if (e < rag) st_elem<DT>(a + e * E, f[e]);
    }
  }
}

// gamma / beta (or gamma alone) as fp32 in shared memory.  Chunk mode keeps
// the four columns e = 4p .. 4p+3 of chunk k at plane p, offset 4k, so a lane
// reads 16 contiguous bytes per plane (conflict-free for consecutive chunks).
template <int W>
struct LnPlanes {
  float* base;
  int npl;  // floats per plane
  // The W values of chunk k (W >= 4) or the value of column k (W == 1).
  __device__ __forceinline__ void get(int k, float (&out)[W]) const {
    if constexpr (W >= 4) {
#pragma unroll
      for (int p = 0; p < W / 4; ++p) {
        const float4 t = *reinterpret_cast<const float4*>(base + p * npl + k * 4);
        out[4 * p] = t.x;
        out[4 * p + 1] = t.y;
        out[4 * p + 2] = t.z;
        out[4 * p + 3] = t.w;
      }
    } else {
      out[0] = base[k];
    }
  }
};

// Misaligned rows (chunk mode): a row group's two buffers of the aligned
// 16-byte blocks that cover a row.  Every thread of the group copies blocks
// gt, gt + G, ... of the next row with cp.async; once the copies have landed and
// the group has synchronised, chunk k of the row is the funnel shift of blocks k
// and k + 1 by the row's start address mod 16.  A row whose covering blocks
// would leave the tensor (the first or last rows of a tensor with a misaligned
// base) is not copied; the caller reads it directly.
template <int DT, int W, int G, int NQ>
struct LnRowPf {
  uint4* buf;  // [2 stages][nb] blocks
  int nb;
  int h0, h1;     // row start address mod 16, stage 0 / 1
  bool ok0, ok1;  // the stage holds its row
  __device__ __forceinline__ void issue(const char* rs, int64_t rowb, const char* tb,
                                        const char* te, int stage, int gt, bool valid) {
    bool ok = false;
    int h = 0;
    if (valid) {
      const uintptr_t a = reinterpret_cast<uintptr_t>(rs);
      const uintptr_t lo = a & ~uintptr_t(15), hi = (a + rowb + 15) & ~uintptr_t(15);
      h = static_cast<int>(a & 15);
      ok = lo >= reinterpret_cast<uintptr_t>(tb) && hi <= reinterpret_cast<uintptr_t>(te);
      if (ok) {
        const int n = static_cast<int>((hi - lo) >> 4);
        uint4* d = buf + stage * nb;
        for (int j = gt; j < n; j += G)
          cp_async16(d + j, reinterpret_cast<const void*>(lo + (uintptr_t)j * 16));
      }
    }
    if (stage) {
      ok1 = ok;
      h1 = h;
    } else {
      ok0 = ok;
      h0 = h;
    }
  }
  // The thread's chunks of the row in stage s (ragged slots 0); false when the
  // row was not copied.
  __device__ __forceinline__ bool get(uint4 (&v)[NQ], int s, int gt, const LnCols<G, NQ>& cs,
                                      int rag) const {
    if (!(s ? ok1 : ok0)) return false;
    const int h = s ? h1 : h0;
    const uint4* b = buf + s * nb;
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      uint4 c = make_uint4(0u, 0u, 0u, 0u);
      if (q < cs.nown) {
        const int k = gt + q * G;
        c = funnel16(b[k], b[k + 1], h);
        if (q >= cs.nf) {
#pragma unroll
          for (int e = 0; e < W; ++e)
            if (e >= rag) chunk_set_bits<DT>(c, e, 0u);
        }
      }
      v[q] = c;
    }
    return true;
  }
};

// Converts gamma (or beta) into its planes.  Chunk mode: one 16-byte load per
// chunk (the vector is 16-byte aligned there), up to four chunks in flight per
// thread so the L2 round trips overlap; element mode: scalar loads, unrolled.
template <int DT, int W>
__device__ __forceinline__ void ln_stage(const LnPlanes<W>& pl, const char* src, int cols, int nch) {
  constexpr int E = DType<DT>::E;
  if constexpr (W >= 4) {
    const int nfull = cols / W;
    for (int k0 = threadIdx.x; k0 < nch; k0 += 4 * blockDim.x) {
      uint4 c[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int k = k0 + u * blockDim.x;
        c[u] = make_uint4(0u, 0u, 0u, 0u);
        if (k < nfull) {
          c[u] = ld_chunk_cached(src + (int64_t)k * 16);
        } else if (k < nch) {
#pragma unroll
          for (int e = 0; e < W; ++e)
            if (k * W + e < cols) {
              const float f = ld_elem_cached<DT>(src + (int64_t)(k * W + e) * E);
              chunk_set_bits<DT>(c[u], e, DT == kF32 ? __float_as_uint(f) : __float_as_uint(f) >> 16);
            }
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int k = k0 + u * blockDim.x;
        if (k < nch) {
#pragma unroll
          for (int p = 0; p < W / 4; ++p)
            *reinterpret_cast<float4*>(pl.base + p * pl.npl + k * 4) =
                make_float4(chunk_get<DT>(c[u], 4 * p), chunk_get<DT>(c[u], 4 * p + 1),
                            chunk_get<DT>(c[u], 4 * p + 2), chunk_get<DT>(c[u], 4 * p + 3));
        }
      }
    }
  } else {
#pragma unroll 8
    for (int j = threadIdx.x; j < cols; j += blockDim.x)
      pl.base[j] = ld_elem_cached<DT>(src + (int64_t)j * E);
  }
}

// ------------------------------------------------------------ forward ------
//
// Per row: compensated (TwoSum) sum of the thread's values, reduced over the
// group as a double-float -> exact mean mh + ml; squared deviations
// ((x - mh) - ml)^2 -> M2 -> rstd = 1/sqrt(M2/C + eps); y = xhat*gamma + beta.
// A row with a non-finite mean or variance is masked: y = 0, mean = rstd = 0.
//
// CL: the row is split over the K blocks of a thread-block cluster (one group
// per block, G = block size); block k owns columns [k*slice, (k+1)*slice) and
// the per-row statistics are merged across the cluster (ln_cluster).
template <int DT, int W, int G, int NQ, bool AL, int MAXT, bool RMS, bool CL = false>
__global__ void __launch_bounds__(MAXT, ln_fwd_min_blocks<MAXT, NQ>())
    ln_fwd_kernel(const LnFwdParams p, const LnGeo geo) {
  constexpr int E = DType<DT>::E;
  extern __shared__ __align__(128) unsigned char smem[];
  int K = 1, rank = 0;
  if constexpr (CL) {
    K = static_cast<int>(cluster_nrank());
    rank = static_cast<int>(cluster_rank());
  }
  // this block's columns: the whole row, or its slice of a clustered row
  const int c0 = rank * geo.slice;
  const int ncols = CL ? min(geo.slice, geo.cols - c0) : geo.cols;
  const int nfull = CL ? ncols / W : geo.nfull;
  const int rag = CL ? ncols - nfull * W : geo.rag;
  const int nchb = CL ? nfull + (rag > 0 ? 1 : 0) : geo.nch;
  const int64_t coff = (int64_t)c0 * E;
  const int npad = geo.nch * W;
  const int npl = W >= 4 ? geo.nch * 4 : geo.nch;
  const LnPlanes<W> sg{reinterpret_cast<float*>(smem), npl};
  const LnPlanes<W> sb{reinterpret_cast<float*>(smem) + npad, npl};
  ln_stage<DT, W>(sg, p.gamma + coff, ncols, nchb);
  if constexpr (!RMS) ln_stage<DT, W>(sb, p.beta + coff, ncols, nchb);
  __syncthreads();

  constexpr int ngroups = MAXT / G;
  const int grp = threadIdx.x / G, gt = threadIdx.x % G;
  LnCols<G, NQ> cs;
  cs.init(gt, nfull, rag);
  LnRed<G> rd{smem + geo.red_off + grp * 1024, 0, 1 + grp};
  int ccalls = 0;
  const int64_t blk = blockIdx.x / K;  // the block's (cluster's) index among row owners
  const int64_t step = (int64_t)(gridDim.x / K) * ngroups;
  const int64_t r0 = blk * ngroups + grp;
  // first row of the warp's first group: sub-warp groups stay in lock step
  const int64_t w0 = blk * ngroups + (G < 32 ? (threadIdx.x & ~31) / G : grp);
  const int64_t rowb = (int64_t)geo.cols * E;
  const int64_t sbytes = (int64_t)ncols * E;
  const char* xend = p.x + geo.rows * rowb;
  const float ns = static_cast<float>(geo.cols);

  // The next row is copied with cp.async while the current one is worked on
  // (as in the backward below): aligned rows into this thread's own slots
  // [2 stages][NQ][block]; misaligned rows into the group's row buffers.
  constexpr bool PF = AL && W > 1;
  constexpr bool PFR = !AL && W > 1 && G >= 32;  // short rows: the per-row sync costs more
  uint4* pf = reinterpret_cast<uint4*>(smem + geo.pf_off);
  LnRowPf<DT, W, G, NQ> rpx{pf + (size_t)grp * 2 * (geo.nch + 2), geo.nch + 2, 0, 0, false, false};
  auto issue = [&](int64_t rr, int stage) {
    if constexpr (PF) {
      if (rr < geo.rows) {
        const char* x0 = p.x + rr * rowb + coff;
#pragma unroll
        for (int q = 0; q < NQ; ++q)
          if (q < cs.nf)
            cp_async16(pf + (stage * NQ + q) * MAXT + threadIdx.x,
                       x0 + (int64_t)(gt + q * G) * 16);
      }
    } else if constexpr (PFR) {
      const bool valid = rr < geo.rows;
      rpx.issue(valid ? p.x + rr * rowb + coff : p.x, sbytes, p.x, xend, stage, gt, valid);
    }
    cp_async_commit();
  };
  auto group_sync = [&]() {
    if constexpr (G > 32) named_bar(1 + grp, G);
    else __syncwarp();
  };
  if constexpr (PF || PFR) issue(r0, 0);

  for (int64_t it = 0;; ++it) {
    if (w0 + it * step >= geo.rows) break;
    const int64_t r = r0 + it * step;
    const bool active = r < geo.rows;
    uint4 v[NQ];
    if constexpr (PF) {
      issue(r + step, (int)((it + 1) & 1));
      cp_async_wait<1>();
#pragma unroll
      for (int q = 0; q < NQ; ++q)
        v[q] = (active && q < cs.nf) ? pf[((int)(it & 1) * NQ + q) * MAXT + threadIdx.x]
                                     : make_uint4(0u, 0u, 0u, 0u);
    } else if constexpr (PFR) {
      issue(r + step, (int)((it + 1) & 1));
      cp_async_wait<1>();
      group_sync();
      if (!(active && rpx.get(v, (int)(it & 1), gt, cs, rag))) {
        if (active) {
          ln_load<DT, W, G, NQ, AL>(v, p.x + r * rowb + coff, gt, cs, rag, p.x, xend);
        } else {
#pragma unroll
          for (int q = 0; q < NQ; ++q) v[q] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
    } else if (active) {
      ln_load<DT, W, G, NQ, AL>(v, p.x + r * rowb + coff, gt, cs, rag, p.x, xend);
    } else {
#pragma unroll
      for (int q = 0; q < NQ; ++q) v[q] = make_uint4(0u, 0u, 0u, 0u);
    }

    float mh = 0.f, ml = 0.f, rstd;
    bool masked;
    if constexpr (RMS) {
      // mean square (no cancellation: a plain fp32 sum of squares)
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        if (q < cs.nown) {
          if constexpr (W > 1) {
#pragma unroll
            for (int e = 0; e < W; e += 2) {
              const float v0 = ln_get<DT, W>(v[q], e), v1 = ln_get<DT, W>(v[q], e + 1);
              fma2(a0, a1, v0, v1, v0, v1, a0, a1);
            }
          } else {
            const float v0 = ln_get<DT, W>(v[q], 0);
            a0 = fmaf(v0, v0, a0);
          }
        }
      }
      Sum1 t = rd(Sum1{a0 + a1}, MergeSum1());
      if constexpr (CL) t = ln_cluster(t, MergeSum1(), smem + geo.cl_off, ccalls, K);
      const float ms = t.s * p.inv_cols;
      if (!active) continue;
      masked = !isfinite(ms);
      rstd = masked ? 0.f : rsqrtf(ms + p.eps);
      if (gt == 0 && rank == 0) p.rstd[r] = rstd;
    } else {
      // 1. compensated sum (two interleaved TwoSum accumulators per packed pair)
      float s0 = 0.f, s1 = 0.f, c0 = 0.f, c1 = 0.f;
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        if (q < cs.nown) {
          if constexpr (W > 1) {
#pragma unroll
            for (int e = 0; e < W; e += 2) {
              const float v0 = ln_get<DT, W>(v[q], e), v1 = ln_get<DT, W>(v[q], e + 1);
              float t0, t1, b0, b1, u0, u1, w0_, w1_;
              add2(t0, t1, s0, s1, v0, v1);      // t = s + v
              add2(b0, b1, t0, t1, -s0, -s1);    // bb = t - s
              add2(u0, u1, t0, t1, -b0, -b1);    // t - bb
              add2(u0, u1, s0, s1, -u0, -u1);    // s - (t - bb)
              add2(w0_, w1_, v0, v1, -b0, -b1);  // v - bb
              add2(u0, u1, u0, u1, w0_, w1_);    // exact error of s + v
              add2(c0, c1, c0, c1, u0, u1);
              s0 = t0;
              s1 = t1;
            }
          } else {
            float t, err;
            two_sum(s0, ln_get<DT, W>(v[q], 0), t, err);
            c0 += err;
            s0 = t;
          }
        }
      }
      CascSum S;
      {
        float s, e;
        two_sum(s0, s1, s, e);
        S = {s, (c0 + c1) + e};
      }
      S = rd(S, MergeCasc());
      if constexpr (CL) S = ln_cluster(S, MergeCasc(), smem + geo.cl_off, ccalls, K);
      {
        float sh, sl;
        two_sum(S.s, S.e, sh, sl);
        df_mean(sh, sl, ns, p.inv_cols, mh, ml);
      }

      // 2. squared deviations from the exact mean (ragged slots excluded)
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        if (q < cs.nown) {
          if constexpr (W > 1) {
            const bool whole = q < cs.nf;
#pragma unroll
            for (int e = 0; e < W; e += 2) {
              float d0, d1;
              add2(d0, d1, ln_get<DT, W>(v[q], e), ln_get<DT, W>(v[q], e + 1), -mh, -mh);
              add2(d0, d1, d0, d1, -ml, -ml);
              if (!whole) {
                if (e >= rag) d0 = 0.f;
                if (e + 1 >= rag) d1 = 0.f;
              }
              fma2(a0, a1, d0, d1, d0, d1, a0, a1);
            }
          } else {
            const float d = (ln_get<DT, W>(v[q], 0) - mh) - ml;
            a0 = fmaf(d, d, a0);
          }
        }
      }
      Sum1 t = rd(Sum1{a0 + a1}, MergeSum1());
      if constexpr (CL) t = ln_cluster(t, MergeSum1(), smem + geo.cl_off, ccalls, K);
      const float m2 = t.s;
      if (!active) continue;
      const float var = m2 * p.inv_cols;
      masked = !(isfinite(mh) && isfinite(ml) && isfinite(var));
      rstd = masked ? 0.f : rsqrtf(var + p.eps);
      if (gt == 0 && rank == 0) {
        p.mean[r] = masked ? 0.f : mh + ml;
        p.rstd[r] = rstd;
      }
    }

    // 3. y = ((x - mh) - ml) * rstd * gamma + beta  (RMSNorm: x * rstd * gamma)
    char* yr = p.y + r * rowb + coff;
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      if (q < cs.nown) {
        float f[W];
        if (masked) {
#pragma unroll
          for (int e = 0; e < W; ++e) f[e] = 0.f;
        } else {
          const int k = gt + q * G;
          float gm[W], bt[W];
          sg.get(k, gm);
          if constexpr (!RMS) sb.get(k, bt);
          if constexpr (RMS) {
            if constexpr (W > 1) {
#pragma unroll
              for (int e = 0; e < W; e += 2) {
                float t0, t1;
                mul2(t0, t1, ln_get<DT, W>(v[q], e), ln_get<DT, W>(v[q], e + 1), rstd, rstd);
                mul2(f[e], f[e + 1], t0, t1, gm[e], gm[e + 1]);
              }
            } else {
              f[0] = (ln_get<DT, W>(v[q], 0) * rstd) * gm[0];
            }
          } else if constexpr (W > 1) {
#pragma unroll
            for (int e = 0; e < W; e += 2) {
              float t0, t1;
              add2(t0, t1, ln_get<DT, W>(v[q], e), ln_get<DT, W>(v[q], e + 1), -mh, -mh);
              add2(t0, t1, t0, t1, -ml, -ml);
              mul2(t0, t1, t0, t1, rstd, rstd);
              fma2(f[e], f[e + 1], t0, t1, gm[e], gm[e + 1], bt[e], bt[e + 1]);
            }
          } else {
            f[0] = fmaf(((ln_get<DT, W>(v[q], 0) - mh) - ml) * rstd, gm[0], bt[0]);
          }
        }
        ln_store<DT, W, G, NQ, AL>(yr, gt, q, cs, rag, f);
      }
    }
  }
  if constexpr (PF || PFR) cp_async_wait<0>();
  if constexpr (CL) cluster_sync();  // peers may still read this block's slots
}

// ----------------------------------------------------------- backward ------
//
// Per row (mean, rstd as saved by the forward; rstd == 0 marks a masked row):
// xhat = (x - mean) * rstd, g = dy * gamma (rounded once and used everywhere),
// S1 = sum g, S2 = sum g * xhat over the group, then
// dx = rstd * ((g - S1/C) - xhat * S2/C).  The thread's column partials
// sum dy*xhat and sum dy stay in registers; at the end the groups of a block
// add theirs in a fixed order into one partial row of the workspace
// ([gridDim.x][2][cols] floats), which col_reduce_kernel sums.
//
// With aligned rows (AL, chunk mode) each thread copies its chunks of dy and x
// for the row after the current one into its own shared-memory slots with
// cp.async while it works on the current row (no registers held, no barrier:
// a thread reads only the slots it filled), and the row statistics one row
// ahead into registers.
//
// SA (the deep variants, many chunks per thread): the column partials live in
// the group's region of shared memory instead of registers (planes of four
// columns, so a lane reads and writes 16 contiguous bytes; each slot touched
// only by the thread owning its chunk), and g and xhat are recomputed from the
// stored chunks for dx instead of being held: far fewer registers, so fewer
// threads per row and more rows in flight per SM.
template <int DT, int W, int G, int NQ, bool AL, int MAXT, bool RMS, bool SA = false,
          bool CL = false>
__global__ void __launch_bounds__(MAXT, ln_bwd_min_blocks<MAXT, NQ>())
    ln_bwd_kernel(const LnBwdParams p, const LnGeo geo) {
  constexpr bool PF = AL && W > 1;
  constexpr bool PFR = !AL && W > 1 && NQ > 1;  // one-chunk variants: no room
  constexpr int E = DType<DT>::E;
  extern __shared__ __align__(128) unsigned char smem[];
  int K = 1, rank = 0;
  if constexpr (CL) {
    K = static_cast<int>(cluster_nrank());
    rank = static_cast<int>(cluster_rank());
  }
  // this block's columns: the whole row, or its slice of a clustered row
  const int c0 = rank * geo.slice;
  const int ncols = CL ? min(geo.slice, geo.cols - c0) : geo.cols;
  const int nfull = CL ? ncols / W : geo.nfull;
  const int rag = CL ? ncols - nfull * W : geo.rag;
  const int nchb = CL ? nfull + (rag > 0 ? 1 : 0) : geo.nch;
  const int64_t coff = (int64_t)c0 * E;
  const int npad = geo.nch * W;
  const int npl = W >= 4 ? geo.nch * 4 : geo.nch;
  const LnPlanes<W> sg{reinterpret_cast<float*>(smem), npl};
  ln_stage<DT, W>(sg, p.gamma + coff, ncols, nchb);
  __syncthreads();

  constexpr int ngroups = MAXT / G;
  const int grp = threadIdx.x / G, gt = threadIdx.x % G;
  LnCols<G, NQ> cs;
  cs.init(gt, nfull, rag);
  LnRed<G> rd{smem + geo.red_off + grp * 1024, 0, 1 + grp};
  int ccalls = 0;
  const int64_t blk = blockIdx.x / K;  // the block's (cluster's) index among row owners
  const int64_t step = (int64_t)(gridDim.x / K) * ngroups;
  const int64_t r0 = blk * ngroups + grp;
  const int64_t w0 = blk * ngroups + (G < 32 ? (threadIdx.x & ~31) / G : grp);
  const int64_t rowb = (int64_t)geo.cols * E;
  const int64_t sbytes = (int64_t)ncols * E;
  const int64_t nbytes = geo.rows * rowb;

  static_assert(!SA || W >= 4, "shared-memory partials are for chunk mode");
  constexpr int kPlanes = RMS ? 1 : 2;  // dgamma (, dbeta)
  // column partials: sum dy*xhat, sum dy (LayerNorm only)
  float ag[SA ? 1 : NQ][W], ab[SA ? 1 : NQ][W];
  // SA: this group's partials, [kPlanes][W / 4][nch][4] floats
  float* sacc = reinterpret_cast<float*>(smem + geo.acc_off) + (size_t)grp * kPlanes * npad;
  const int spl = geo.nch * 4;  // floats per plane of four columns
  if constexpr (SA) {
#pragma unroll
    for (int q = 0; q < NQ; ++q)
      if (q < cs.nown) {
        const int k = gt + q * G;
#pragma unroll
        for (int pl = 0; pl < kPlanes * (W / 4); ++pl)
          *reinterpret_cast<float4*>(sacc + pl * spl + k * 4) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
  } else {
#pragma unroll
    for (int q = 0; q < NQ; ++q)
#pragma unroll
      for (int e = 0; e < W; ++e) ag[q][e] = ab[q][e] = 0.f;
  }

  uint4* pf = reinterpret_cast<uint4*>(smem + geo.pf_off);
  auto slot = [&](int stage, int t, int q) -> uint4* {
    return pf + ((stage * 2 + t) * NQ + q) * MAXT + threadIdx.x;
  };
  // misaligned rows: the group's row buffers, [dy | x][2 stages][nb]
  LnRowPf<DT, W, G, NQ> rpd{pf + (size_t)grp * 4 * (geo.nch + 2), geo.nch + 2, 0, 0, false, false};
  LnRowPf<DT, W, G, NQ> rpx{pf + (size_t)grp * 4 * (geo.nch + 2) + 2 * (geo.nch + 2), geo.nch + 2,
                            0, 0, false, false};
  // row rr's chunks into stage `stage` (an empty group past the last row)
  auto issue = [&](int64_t rr, int stage) {
    if constexpr (PF) {
      if (rr < geo.rows) {
        const char* d0 = p.dy + rr * rowb + coff;
        const char* x0 = p.x + rr * rowb + coff;
#pragma unroll
        for (int q = 0; q < NQ; ++q)
          if (q < cs.nf) {
            cp_async16(slot(stage, 0, q), d0 + (int64_t)(gt + q * G) * 16);
            cp_async16(slot(stage, 1, q), x0 + (int64_t)(gt + q * G) * 16);
          }
      }
    } else if constexpr (PFR) {
      const bool valid = rr < geo.rows;
      rpd.issue(valid ? p.dy + rr * rowb + coff : p.dy, sbytes, p.dy, p.dy + nbytes, stage, gt,
                valid);
      rpx.issue(valid ? p.x + rr * rowb + coff : p.x, sbytes, p.x, p.x + nbytes, stage, gt, valid);
    }
    cp_async_commit();
  };
  auto group_sync = [&]() {
    if constexpr (G > 32) named_bar(1 + grp, G);
    else __syncwarp();
  };
  auto stats = [&](int64_t rr, float& mu, float& rs) {
    mu = 0.f;
    rs = 0.f;
    if (rr < geo.rows) {
      if constexpr (!RMS) mu = __ldg(p.mean + rr);
      rs = __ldg(p.rstd + rr);
    }
  };
  float nmean = 0.f, nrstd = 0.f;
  if constexpr (PF || PFR) {
    issue(r0, 0);
    stats(r0, nmean, nrstd);
  }

  for (int64_t it = 0;; ++it) {
    if (w0 + it * step >= geo.rows) break;
    const int64_t r = r0 + it * step;
    const bool active = r < geo.rows;
    float mean, rstd;
    if constexpr (PF || PFR) {
      mean = nmean;
      rstd = nrstd;
      issue(r + step, (int)((it + 1) & 1));
      stats(r + step, nmean, nrstd);
      cp_async_wait<1>();
      if constexpr (PFR) group_sync();
    } else {
      stats(r, mean, rstd);
    }
    const bool use = active && rstd != 0.f;
    float gv[SA ? 1 : NQ][W], hv[SA ? 1 : NQ][W];
    float s1a = 0.f, s1b = 0.f, s2a = 0.f, s2b = 0.f;
    uint4 dv[NQ], xv[NQ];
    if (use) {
      if constexpr (PF) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          dv[q] = q < cs.nf ? *slot((int)(it & 1), 0, q) : make_uint4(0u, 0u, 0u, 0u);
          xv[q] = q < cs.nf ? *slot((int)(it & 1), 1, q) : make_uint4(0u, 0u, 0u, 0u);
        }
      } else if constexpr (PFR) {
        if (!rpd.get(dv, (int)(it & 1), gt, cs, rag))
          ln_load<DT, W, G, NQ, AL>(dv, p.dy + r * rowb + coff, gt, cs, rag, p.dy, p.dy + nbytes);
        if (!rpx.get(xv, (int)(it & 1), gt, cs, rag))
          ln_load<DT, W, G, NQ, AL>(xv, p.x + r * rowb + coff, gt, cs, rag, p.x, p.x + nbytes);
      } else {
        ln_load<DT, W, G, NQ, AL>(dv, p.dy + r * rowb + coff, gt, cs, rag, p.dy, p.dy + nbytes);
        ln_load<DT, W, G, NQ, AL>(xv, p.x + r * rowb + coff, gt, cs, rag, p.x, p.x + nbytes);
      }
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        if (q < cs.nown) {
          float gm[W];
          sg.get(gt + q * G, gm);
          if constexpr (W > 1) {
            // SA: this chunk's partials from shared memory, updated, written back
            const int qa = SA ? 0 : q;
            const int k = gt + q * G;
            if constexpr (SA) {
#pragma unroll
              for (int pq = 0; pq < W / 4; ++pq) {
                const float4 tg = *reinterpret_cast<const float4*>(sacc + pq * spl + k * 4);
                ag[0][4 * pq] = tg.x; ag[0][4 * pq + 1] = tg.y;
                ag[0][4 * pq + 2] = tg.z; ag[0][4 * pq + 3] = tg.w;
                if constexpr (!RMS) {
                  const float4 tb = *reinterpret_cast<const float4*>(sacc + (W / 4 + pq) * spl + k * 4);
                  ab[0][4 * pq] = tb.x; ab[0][4 * pq + 1] = tb.y;
                  ab[0][4 * pq + 2] = tb.z; ab[0][4 * pq + 3] = tb.w;
                }
              }
            }
#pragma unroll
            for (int e = 0; e < W; e += 2) {
              const float y0 = ln_get<DT, W>(dv[q], e), y1 = ln_get<DT, W>(dv[q], e + 1);
              float h0, h1;
              if constexpr (RMS) {
                mul2(h0, h1, ln_get<DT, W>(xv[q], e), ln_get<DT, W>(xv[q], e + 1), rstd, rstd);
              } else {
                add2(h0, h1, ln_get<DT, W>(xv[q], e), ln_get<DT, W>(xv[q], e + 1), -mean, -mean);
                mul2(h0, h1, h0, h1, rstd, rstd);
              }
              const float g0 = __fmul_rn(y0, gm[e]), g1 = __fmul_rn(y1, gm[e + 1]);
              if constexpr (!RMS) add2(s1a, s1b, s1a, s1b, g0, g1);
              fma2(s2a, s2b, g0, g1, h0, h1, s2a, s2b);
              fma2(ag[qa][e], ag[qa][e + 1], y0, y1, h0, h1, ag[qa][e], ag[qa][e + 1]);
              if constexpr (!RMS) add2(ab[qa][e], ab[qa][e + 1], ab[qa][e], ab[qa][e + 1], y0, y1);
              if constexpr (!SA) {
                gv[q][e] = g0;
                gv[q][e + 1] = g1;
                hv[q][e] = h0;
                hv[q][e + 1] = h1;
              }
            }
            if constexpr (SA) {
#pragma unroll
              for (int pq = 0; pq < W / 4; ++pq) {
                *reinterpret_cast<float4*>(sacc + pq * spl + k * 4) =
                    make_float4(ag[0][4 * pq], ag[0][4 * pq + 1], ag[0][4 * pq + 2], ag[0][4 * pq + 3]);
                if constexpr (!RMS)
                  *reinterpret_cast<float4*>(sacc + (W / 4 + pq) * spl + k * 4) = make_float4(
                      ab[0][4 * pq], ab[0][4 * pq + 1], ab[0][4 * pq + 2], ab[0][4 * pq + 3]);
              }
            }
          } else {
            const float y0 = ln_get<DT, W>(dv[q], 0);
            const float h0 = RMS ? ln_get<DT, W>(xv[q], 0) * rstd
                                 : (ln_get<DT, W>(xv[q], 0) - mean) * rstd;
            const float g0 = __fmul_rn(y0, gm[0]);
            if constexpr (!RMS) s1a += g0;
            s2a = fmaf(g0, h0, s2a);
            ag[q][0] = fmaf(y0, h0, ag[q][0]);
            if constexpr (!RMS) ab[q][0] += y0;
            gv[q][0] = g0;
            hv[q][0] = h0;
          }
        }
      }
    }
    Sum2 s = rd(Sum2{s1a + s1b, s2a + s2b}, MergeSum2());
    if constexpr (CL) s = ln_cluster(s, MergeSum2(), smem + geo.cl_off, ccalls, K);
    if (!active) continue;
    const float a = s.s1 * p.inv_cols;
    const float b = s.s2 * p.inv_cols;
    char* dxr = p.dx + r * rowb + coff;
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      if (q < cs.nown) {
        float f[W];
        if (!use) {
#pragma unroll
          for (int e = 0; e < W; ++e) f[e] = 0.f;
        } else if constexpr (SA) {
          // g and xhat again from the stored chunks (the same operations, the
          // same bits as in the first pass)
          float gm[W];
          sg.get(gt + q * G, gm);
#pragma unroll
          for (int e = 0; e < W; e += 2) {
            const float y0 = ln_get<DT, W>(dv[q], e), y1 = ln_get<DT, W>(dv[q], e + 1);
            float h0, h1;
            if constexpr (RMS) {
              mul2(h0, h1, ln_get<DT, W>(xv[q], e), ln_get<DT, W>(xv[q], e + 1), rstd, rstd);
            } else {
              add2(h0, h1, ln_get<DT, W>(xv[q], e), ln_get<DT, W>(xv[q], e + 1), -mean, -mean);
              mul2(h0, h1, h0, h1, rstd, rstd);
            }
            const float g0 = __fmul_rn(y0, gm[e]), g1 = __fmul_rn(y1, gm[e + 1]);
            float t0, t1;
            add2(t0, t1, g0, g1, -a, -a);
            fma2(t0, t1, h0, h1, -b, -b, t0, t1);
            mul2(f[e], f[e + 1], t0, t1, rstd, rstd);
          }
        } else if constexpr (W > 1) {
#pragma unroll
          for (int e = 0; e < W; e += 2) {
            float t0, t1;
            add2(t0, t1, gv[q][e], gv[q][e + 1], -a, -a);               // g - a
            fma2(t0, t1, hv[q][e], hv[q][e + 1], -b, -b, t0, t1);      // (g - a) - xhat b
            mul2(f[e], f[e + 1], t0, t1, rstd, rstd);
          }
        } else {
          f[0] = rstd * ((gv[q][0] - a) - hv[q][0] * b);
        }
        ln_store<DT, W, G, NQ, AL>(dxr, gt, q, cs, rag, f);
      }
    }
  }

  if constexpr (PF || PFR) cp_async_wait<0>();
  if constexpr (CL) cluster_sync();  // peers may still read this block's slots

  // Column partials: each group's to shared memory (SA: already there), then
  // a fixed-order sum over the groups into this block's partial row.
  if constexpr (!SA) {
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      if (q < cs.nown) {
        const int j = (gt + q * G) * W;
#pragma unroll
        for (int e = 0; e < W; ++e) {
          sacc[j + e] = ag[q][e];
          if constexpr (!RMS) sacc[npad + j + e] = ab[q][e];
        }
      }
    }
  }
  __syncthreads();
  // (clusters: the block's slice of its cluster's partial row)
  const float* all = reinterpret_cast<const float*>(smem + geo.acc_off);
  float* out = p.ws + blk * kPlanes * geo.cols + c0;
  for (int i = threadIdx.x; i < kPlanes * ncols; i += MAXT) {
    const int half = i >= ncols ? 1 : 0;
    const int j = i - half * ncols;
    // column j of a group's region: SA planes of four columns, else in order
    const int o = SA ? half * npad + ((j % W) >> 2) * spl + (j / W) * 4 + (j & 3) : half * npad + j;
    float t = 0.f;
    for (int gi = 0; gi < ngroups; ++gi) t += all[(size_t)gi * kPlanes * npad + o];
    out[(int64_t)half * geo.cols + j] = t;
  }
}

// Fills the variants G = 1 .. 1024 of one mode (block size max(256, G)
// forward, max(512, G) backward; the backward stops at G = 512, beyond which a
// 1024-thread block could not give a thread its 128 registers).
// Clustered forward variants: one group of G = 256 / 512 / 1024 threads per
// block, and a 256-thread group holding twice the chunks per thread (fewer,
// fuller threads per slice: the per-row reductions are paid over more values).
template <int DT, int W, int NQ, bool AL, bool RMS>
void ln_fill_cluster(const void* (&row)[4]) {
  row[0] = (const void*)ln_fwd_kernel<DT, W, 256, NQ, AL, 256, RMS, true>;
  row[1] = (const void*)ln_fwd_kernel<DT, W, 512, NQ, AL, 512, RMS, true>;
  row[2] = (const void*)ln_fwd_kernel<DT, W, 1024, NQ, AL, 1024, RMS, true>;
  row[3] = (const void*)ln_fwd_kernel<DT, W, 256, 2 * NQ, AL, 256, RMS, true>;
}

// Clustered backward variants (chunk mode only): one group of 256 / 512 threads
// per block with NQ chunks per thread and the column partials in shared memory.
template <int DT, int W, int NQ, bool AL, bool RMS>
void ln_fill_cluster_bwd(const void* (&row)[4]) {
  row[0] = (const void*)ln_bwd_kernel<DT, W, 256, NQ, AL, 256, RMS, true, true>;
  row[1] = (const void*)ln_bwd_kernel<DT, W, 512, NQ, AL, 512, RMS, true, true>;
  row[2] = nullptr;
  row[3] = nullptr;
}

template <int DT, int W, int NQ, bool AL, bool FWD, int G, bool RMS, bool SA = false>
const void* ln_variant() {
  if constexpr (FWD) {
    return (const void*)ln_fwd_kernel<DT, W, G, NQ, AL, (G > 256 ? G : 256), RMS>;
  } else if constexpr (G <= 512 && SA) {
    return (const void*)ln_bwd_kernel<DT, W, G, NQ, AL, (G > 128 ? G : 128), RMS, true>;
  } else if constexpr (G <= 512) {
    return (const void*)ln_bwd_kernel<DT, W, G, NQ, AL, 512, RMS>;
  } else {
    return nullptr;
  }
}
template <int DT, int W, int NQ, bool AL, bool FWD, bool RMS>
void ln_fill_row(const void* (&row)[kNumLnG]) {
  row[0] = ln_variant<DT, W, NQ, AL, FWD, 1, RMS>();
  row[1] = ln_variant<DT, W, NQ, AL, FWD, 2, RMS>();
  row[2] = ln_variant<DT, W, NQ, AL, FWD, 4, RMS>();
  row[3] = ln_variant<DT, W, NQ, AL, FWD, 8, RMS>();
  row[4] = ln_variant<DT, W, NQ, AL, FWD, 16, RMS>();
  row[5] = ln_variant<DT, W, NQ, AL, FWD, 32, RMS>();
  row[6] = ln_variant<DT, W, NQ, AL, FWD, 64, RMS>();
  row[7] = ln_variant<DT, W, NQ, AL, FWD, 128, RMS>();
  row[8] = ln_variant<DT, W, NQ, AL, FWD, 256, RMS>();
  row[9] = ln_variant<DT, W, NQ, AL, FWD, 512, RMS>();
  row[10] = ln_variant<DT, W, NQ, AL, FWD, 1024, RMS>();
}

template <int DT, int W, bool AL, bool RMS>
void ln_fill_row1(const void* (&row)[kNumLnG]) {
  row[0] = ln_variant<DT, W, 1, AL, false, 1, RMS>();
  row[1] = ln_variant<DT, W, 1, AL, false, 2, RMS>();
  row[2] = ln_variant<DT, W, 1, AL, false, 4, RMS>();
  row[3] = ln_variant<DT, W, 1, AL, false, 8, RMS>();
  row[4] = ln_variant<DT, W, 1, AL, false, 16, RMS>();
  row[5] = ln_variant<DT, W, 1, AL, false, 32, RMS>();
}

// The deep variants: G >= 64; the backward ones keep their column partials in
// shared memory (SA), block size max(G, 128).
template <int DT, int W, int NQ, bool AL, bool FWD, bool RMS>
void ln_fill_deep(const void* (&row)[kNumLnG]) {
  row[6] = ln_variant<DT, W, NQ, AL, FWD, 64, RMS, !FWD>();
  row[7] = ln_variant<DT, W, NQ, AL, FWD, 128, RMS, !FWD>();
  row[8] = ln_variant<DT, W, NQ, AL, FWD, 256, RMS, !FWD>();
  row[9] = ln_variant<DT, W, NQ, AL, FWD, 512, RMS, !FWD>();
  row[10] = ln_variant<DT, W, NQ, AL, FWD, 1024, RMS, !FWD>();
}

// NQC / NQE: chunks (elements) per thread of the chunk (element) mode
// variants; NQD > 0: the deep chunk-mode variants with NQD chunks per thread.
template <int DT, bool FWD, int NQC, int NQE, bool RMS = false, int NQD = 0>
LnKernelSet make_ln_set() {
  constexpr int V = DType<DT>::V;
  LnKernelSet s{};
  ln_fill_row<DT, V, NQC, true, FWD, RMS>(s.k[0]);
  ln_fill_row<DT, V, NQC, false, FWD, RMS>(s.k[1]);
  ln_fill_row<DT, 1, NQE, false, FWD, RMS>(s.k[2]);
  if constexpr (NQD > 0) {
    ln_fill_deep<DT, V, NQD, true, FWD, RMS>(s.kd[0]);
    ln_fill_deep<DT, V, NQD, false, FWD, RMS>(s.kd[1]);
    if constexpr (!FWD) {
      ln_fill_cluster_bwd<DT, V, NQD, true, RMS>(s.kc[0]);
      ln_fill_cluster_bwd<DT, V, NQD, false, RMS>(s.kc[1]);
    }
  }
  s.nqd = NQD;
  if constexpr (FWD) {
    ln_fill_cluster<DT, V, NQC, true, RMS>(s.kc[0]);
    ln_fill_cluster<DT, V, NQC, false, RMS>(s.kc[1]);
    ln_fill_cluster<DT, 1, NQE, false, RMS>(s.kc[2]);
  } else {
    ln_fill_row1<DT, V, true, RMS>(s.k1[0]);
    ln_fill_row1<DT, V, false, RMS>(s.k1[1]);
    ln_fill_row1<DT, 1, false, RMS>(s.k1[2]);
  }
  s.nq[0] = s.nq[1] = NQC;
  s.nq[2] = NQE;
  return s;
}

}  // namespace rr
