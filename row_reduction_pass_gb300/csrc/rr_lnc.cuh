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
// chunks [b * CB, b * CB + CB) of the rows of the class in the group, CB at
// most 128 CPL and chosen so the blocks of a row are equal.  Thread t of the
// block takes chunks b * CB + t + 128 j (j < CPL) of each of the item's rows in
// turn: the threads stream different columns of the same rows, and no thread
// ever waits for another block -- the launches order the phases.  Rows of a few hundred thousand bytes then keep every SM busy
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

constexpr int kLncThreads = 32 * kLncWarps;
constexpr int kLncStride = 16 * kLncThreads;  // bytes between a thread's chunks j, j + 1

// A block's work item and its view of the rows: rows r0 + i P (i < nr) of
// the class; this thread's chunks k0 + 128 j (j < CPL, within the block) of
// each.
template <int W, int CPL>
struct LncItem {
  int cls, b, grp;
  int phi;          // row start offset within its first chunk, in elements
  int64_t r0;       // first row of the item
  int nr;           // its rows
  int64_t rstep;    // bytes from one of its rows to the next (P rows)
  int64_t off0;     // bytes from a row's start to this thread's chunk j = 0
  int lo[CPL], hi[CPL];  // valid lanes [lo, hi) of chunk j (empty outside the row)

  __device__ __forceinline__ void init(const LncGeo& g, const char* base, int E) {
    const int64_t it = blockIdx.x;
    cls = static_cast<int>(it % g.P);
    const int64_t rest = it / g.P;
    b = static_cast<int>(rest % g.nb);
    grp = static_cast<int>(rest / g.nb);
    const int64_t rowb = g.cols * E;
    phi = static_cast<int>(((reinterpret_cast<uintptr_t>(base) + (uint64_t)cls * rowb) & 15) / E);
    const int64_t nch = (phi + g.cols + W - 1) / W;  // chunks covering a row of the class
    const int tail = static_cast<int>(phi + g.cols - (int64_t)W * (nch - 1));
    // rows of the class: cls, cls + P, ...; this group's: [grp * rg, grp * rg + rg)
    const int64_t first = (int64_t)grp * g.rg;
    const int64_t in_class = g.rows > cls ? (g.rows - cls + g.P - 1) / g.P : 0;
    r0 = cls + (int64_t)g.P * first;
    nr = static_cast<int>(first < in_class ? (in_class - first < g.rg ? in_class - first : g.rg) : 0);
    rstep = (int64_t)g.P * rowb;
    const int64_t k0 = (int64_t)b * g.cb + threadIdx.x;
    off0 = k0 * 16 - (int64_t)phi * E;
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
      const int64_t k = k0 + kLncThreads * j;
      lo[j] = k == 0 ? phi : 0;
      hi[j] = k == nch - 1 ? tail : W;
      if (k >= nch || (int)threadIdx.x + kLncThreads * j >= g.cb) lo[j] = hi[j] = 0;
    }
  }
  // This thread's chunk 0 in row i of the item (chunk j is kLncStride j bytes
  // on).
  __device__ __forceinline__ const char* at_row(const char* base, int i, const LncGeo& g,
                                                int64_t rowb) const {
    return base + (r0 + (int64_t)i * g.P) * rowb + off0;
  }
  __device__ __forceinline__ bool has(int j) const { return hi[j] > lo[j]; }
  // Column of lane 0 of chunk j (negative for the lanes before the row).
  __device__ __forceinline__ int64_t col0(int j, int E) const {
    return (off0 + (int64_t)kLncStride * j) / E;
  }
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

// Whether any lane of this warp holds a chunk with lanes outside the row (a
// row's first or last chunk, or a chunk past it): only such warps (the first
// and last of a row's blocks) take the masked code paths.
template <bool B>
struct LncMask {
  static constexpr bool value = B;
};
template <int W, int CPL>
__device__ __forceinline__ bool lnc_warp_ragged(const int (&lo)[CPL], const int (&hi)[CPL]) {
  bool r = false;
#pragma unroll
  for (int j = 0; j < CPL; ++j) r |= lo[j] != 0 || hi[j] != W;
  return __any_sync(0xffffffffu, r);
}

// Stores a chunk: one aligned 128-bit store for an interior chunk, the row's
// own lanes one by one for its first / last chunk.
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

__device__ __forceinline__ uint64_t lnc_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// A block's ring of kLncDepth row stages in dynamic shared memory: stage
// i mod depth holds the block's chunks of row i of the item for T tensors,
// brought by one 1-D bulk copy (TMA) per tensor that thread 0 issues two rows
// (a pair) ahead, completing on the stage's mbarrier; every thread waits for
// the stage's phase (bounded) and reads its own chunks.  Thread 0 refills a
// stage only after a block barrier that follows every thread's last read of
// it.  Bulk copies keep the rows in flight without per-thread request slots
// (per-thread 16-byte copies capped these kernels at ~2.4 TB/s).  Reads: this
// thread's chunk j of the stage is local chunk t + 128 j.  K1 kernels (whose
// data the next launch reads again) mark the lines evict-last in L2, K2
// kernels evict-first.
template <int T, int CPL>
struct LncBulk {
  static constexpr int kCB = kLncThreads * CPL;  // chunks of a stage (a block has at most these)
  uint4* ring;
  uint64_t* bars;
  uint64_t policy;
  uint32_t bytes;      // bytes of one tensor's copy (0: the block has no chunk)
  const char* nxt[T];  // the block's first chunk of the next row to copy
  int issued;
  int local;           // this thread's local chunk j = 0

  template <int W>
  __device__ __forceinline__ void init(unsigned char* smem, const LncItem<W, CPL>& it,
                                       const LncGeo& g, const char* const (&base)[T], int E,
                                       bool keep) {
    ring = reinterpret_cast<uint4*>(smem);
    bars = reinterpret_cast<uint64_t*>(smem + kLncDepth * T * kCB * 16);
    policy = keep ? lnc_policy_evict_last() : policy_evict_first();
    const int64_t rowb = g.cols * E;
    const int64_t phi_b = (int64_t)it.phi * E;
    const int64_t nch = (phi_b + rowb + 15) / 16;
    const int64_t kb = (int64_t)it.b * g.cb;
    const int64_t n = nch - kb < g.cb ? nch - kb : g.cb;
    bytes = n > 0 ? static_cast<uint32_t>(n) * 16 : 0u;
#pragma unroll
    for (int t = 0; t < T; ++t) nxt[t] = base[t] + it.r0 * rowb - phi_b + kb * 16;
    issued = 0;
    local = threadIdx.x;
  }
  __device__ __forceinline__ uint4* stage(int i, int t) const {
    return ring + ((i & (kLncDepth - 1)) * T + t) * kCB;
  }
  __device__ __forceinline__ const uint4& at(int i, int t, int j) const {
    return stage(i, t)[local + kLncThreads * j];
  }
  // Thread 0: the next row's copies (none past the item's rows).
  __device__ __forceinline__ void issue(int nr, int64_t rstep) {
    if (issued < nr && bytes > 0) {
      uint64_t* bar = &bars[issued & (kLncDepth - 1)];
      fence_proxy_async_smem();  // earlier generic reads of the stage come first
      mbar_arrive_expect_tx(bar, bytes * T);
#pragma unroll
      for (int t = 0; t < T; ++t)
        bulk_load(stage(issued, t), nxt[t], bytes, bar, policy);
    }
#pragma unroll
    for (int t = 0; t < T; ++t) nxt[t] += rstep;
    ++issued;
  }
  // Every thread: row i has landed (false if the wait gave up: error recorded).
  __device__ __forceinline__ bool wait(int i, int* err) {
    if (bytes == 0) return true;
    return mbar_wait_bounded(&bars[i & (kLncDepth - 1)],
                             static_cast<uint32_t>((i / kLncDepth) & 1), err);
  }
  // After a wait gave up: thread 0 waits (bounded) for the last copy issued
  // into each stage, so none is still writing the block's shared memory.
  __device__ __forceinline__ void drain(int nr, int* err) const {
    if (bytes == 0) return;
    const int n = issued < nr ? issued : nr;  // rows actually copied
    for (int s = 0; s < kLncDepth; ++s) {
      if (n <= s) continue;
      const int last = s + ((n - 1 - s) / kLncDepth) * kLncDepth;
      mbar_wait_bounded(&bars[s], static_cast<uint32_t>((last / kLncDepth) & 1), err, 100000000ull);
    }
  }
};

// Rows are taken two at a time (one ring refill and one block barrier per
// pair).  The ring's set-up: thread 0 initialises the barriers and
// issues the first depth - 2 rows; the block barrier publishes the barriers.
template <int T, int W, int CPL>
__device__ __forceinline__ void lnc_start(LncBulk<T, CPL>& ring, const LncItem<W, CPL>& it) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < kLncDepth; ++s) mbar_init(&ring.bars[s], 1);
    fence_mbar_init();
    for (int s = 0; s < kLncDepth - 2; ++s) ring.issue(it.nr, it.rstep);
  }
  __syncthreads();
}

// Top of rows i, i + 1: every thread is done with rows i - 2, i - 1 (block
// barrier), thread 0 refills those stages with rows i + depth - 2 and
// i + depth - 1, then all wait for rows i and i + 1.
template <int T, int CPL>
__device__ __forceinline__ void lnc_next2(LncBulk<T, CPL>& ring, int i, int nr, int64_t rstep,
                                          bool& dead, int* err) {
  if (i > 0) __syncthreads();
  if (threadIdx.x == 0) {
    ring.issue(nr, rstep);
    ring.issue(nr, rstep);
  }
  if (!dead) dead = !ring.wait(i, err);
  if (i + 1 < nr && !dead) dead = !ring.wait(i + 1, err);
}

// ------------------------------------------------------------- forward ----

// Launch 1: per (row, column block) records -- Moments (LayerNorm) or the sum
// of squares (RMSNorm) -- into the scratch at p.y rounded up to 16 bytes.
template <int DT, bool RMS, int CPL>
__global__ void __launch_bounds__(kLncThreads, 5) lnc_stats_kernel(const LnFwdParams p,
                                                                const LncGeo g) {
  constexpr int E = DType<DT>::E, W = DType<DT>::V;
  constexpr int RS = 32;  // rows whose warp records are merged together (even)
  extern __shared__ __align__(128) unsigned char lnc_smem[];
  __shared__ Moments part[RS][kLncWarps];
  LncItem<W, CPL> it;
  it.init(g, p.x, E);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  char* recs = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(p.y) + 15) & ~uintptr_t(15));
  LncBulk<1, CPL> ring;
  {
    const char* const base[1] = {p.x};
    ring.init(lnc_smem, it, g, base, E, true);
  }
  lnc_start(ring, it);
  bool dead = false;
  // valid values of this warp's slice of a row (the same for every row)
  int cnt = 0;
#pragma unroll
  for (int j = 0; j < CPL; ++j) cnt += it.hi[j] - it.lo[j];
  const float nw = lnc_warp_sum(static_cast<float>(cnt));
  const float inv_nw = nw > 0.f ? 1.f / nw : 0.f;
  const bool ragged = lnc_warp_ragged<W, CPL>(it.lo, it.hi);

  // the moments of this warp's slice of row i (masked lanes only in ragged
  // warps)
  auto row_moments = [&](int i, auto tag) {
    constexpr bool M = decltype(tag)::value;
    float v[CPL][W];
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
      if (!M || it.has(j)) lnc_unpack<DT, W>(ring.at(i, 0, j), v[j]);
      if constexpr (M) lnc_clip<W>(v[j], it.lo[j], it.hi[j]);  // also a chunk past the row
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
        if constexpr (M) lnc_clip<W>(d, it.lo[j], it.hi[j]);
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
    return m;
  };

  for (int i = 0; i < it.nr; i += 2) {
    lnc_next2(ring, i, it.nr, it.rstep, dead, p.err);
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (u == 1 && i + 1 >= it.nr) break;
      const Moments m = ragged ? row_moments(i + u, LncMask<true>())
                               : row_moments(i + u, LncMask<false>());
      if (lane == 0) part[(i + u) % RS][warp] = m;
    }
    // every RS rows (and at the end): the block's record of each row, its
    // warps' records merged in warp order
    const int done = min(i + 2, it.nr);
    if (done % RS == 0 || done == it.nr) {
      __syncthreads();
      const int base = (done - 1) / RS * RS, ns = done - base;
      if (threadIdx.x < ns) {
        const int ri = threadIdx.x;
        Moments mm = part[ri][0];
        for (int w = 1; w < kLncWarps; ++w) {
          if constexpr (RMS) mm.sh += part[ri][w].sh;
          else mm = MergeMoments()(mm, part[ri][w]);
        }
        const int64_t r = it.r0 + (int64_t)(base + ri) * g.P;
        if constexpr (RMS)
          reinterpret_cast<float*>(recs)[r * g.nb + it.b] = mm.sh;
        else
          reinterpret_cast<float4*>(recs)[r * g.nb + it.b] = make_float4(mm.n, mm.sh, mm.sl, mm.m2);
      }
      __syncthreads();
    }
  }
  if (dead && threadIdx.x == 0) ring.drain(it.nr, p.err);
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
__global__ void __launch_bounds__(kLncThreads, 5) lnc_norm_kernel(const LnFwdParams p,
                                                               const LncGeo g) {
  constexpr int E = DType<DT>::E, W = DType<DT>::V;
  extern __shared__ __align__(128) unsigned char lnc_smem[];
  LncItem<W, CPL> it;
  it.init(g, p.x, E);
  const int64_t rowb = g.cols * E;
  LncBulk<1, CPL> ring;
  {
    const char* const base[1] = {p.x};
    ring.init(lnc_smem, it, g, base, E, false);
  }
  lnc_start(ring, it);
  bool dead = false;
  float gm[CPL][W], bt[CPL][W];
#pragma unroll
  for (int j = 0; j < CPL; ++j) {
#pragma unroll
    for (int e = 0; e < W; ++e) gm[j][e] = bt[j][e] = 0.f;
    if (it.has(j)) {
      lnc_vec_chunk<DT, W>(p.gamma, g.cols, it.col0(j, E), gm[j]);
      if constexpr (!RMS) lnc_vec_chunk<DT, W>(p.beta, g.cols, it.col0(j, E), bt[j]);
    }
  }
  const bool ragged = lnc_warp_ragged<W, CPL>(it.lo, it.hi);
  // y of this warp's slice of row i (lane-wise stores only in ragged warps)
  auto row_out = [&](int i, float mean, float rstd, char* out, auto tag) {
    constexpr bool M = decltype(tag)::value;
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
      if (M && !it.has(j)) continue;
      float v[W], y[W];
      lnc_unpack<DT, W>(ring.at(i, 0, j), v);
      if (rstd == 0.f) {  // masked row
#pragma unroll
        for (int e = 0; e < W; ++e) y[e] = 0.f;
      } else {
#pragma unroll
        for (int e = 0; e < W; e += 2) {
          float t0, t1;
          if constexpr (RMS) {
            mul2(t0, t1, v[e], v[e + 1], rstd, rstd);
            mul2(y[e], y[e + 1], t0, t1, gm[j][e], gm[j][e + 1]);
          } else {
            add2(t0, t1, v[e], v[e + 1], -mean, -mean);
            mul2(t0, t1, t0, t1, rstd, rstd);
            fma2(y[e], y[e + 1], t0, t1, gm[j][e], gm[j][e + 1], bt[j][e], bt[j][e + 1]);
          }
        }
      }
      if constexpr (M) lnc_store<DT, W>(out + kLncStride * j, it.lo[j], it.hi[j], y);
      else st_chunk_stream(out + kLncStride * j, chunk_pack<DT>(y));
    }
  };
  char* out = const_cast<char*>(it.at_row(p.y, 0, g, rowb));
  const float* pm = p.mean + it.r0;
  const float* pr = p.rstd + it.r0;
  const int64_t sP = g.P;
  for (int i = 0; i < it.nr; i += 2, out += 2 * it.rstep, pm += 2 * sP, pr += 2 * sP) {
    const bool two = i + 1 < it.nr;
    const float mean0 = RMS ? 0.f : __ldg(pm), rstd0 = __ldg(pr);
    const float mean1 = RMS || !two ? 0.f : __ldg(pm + sP), rstd1 = two ? __ldg(pr + sP) : 0.f;
    lnc_next2(ring, i, it.nr, it.rstep, dead, p.err);
    if (ragged) {
      row_out(i, mean0, rstd0, out, LncMask<true>());
      if (two) row_out(i + 1, mean1, rstd1, out + it.rstep, LncMask<true>());
    } else {
      row_out(i, mean0, rstd0, out, LncMask<false>());
      if (two) row_out(i + 1, mean1, rstd1, out + it.rstep, LncMask<false>());
    }
  }
  if (dead && threadIdx.x == 0) ring.drain(it.nr, p.err);
}

// ------------------------------------------------------------ backward ----

// Launch 1: per (row, column block) records (S1, S2) at p.ws + g.rec_off
// floats, and the item's column partials (sum dy xhat, sum dy) in its partial
// row (class, row group) of p.ws: [partial][planes][cols].
template <int DT, bool RMS, int CPL>
__global__ void __launch_bounds__(kLncThreads, 5) lnc_bwd_part_kernel(const LnBwdParams p,
                                                                   const LncGeo g) {
  constexpr int E = DType<DT>::E, W = DType<DT>::V;
  constexpr int kPlanes = RMS ? 1 : 2;
  constexpr int RS = 32;  // even
  extern __shared__ __align__(128) unsigned char lnc_smem[];
  __shared__ float2 part[RS][kLncWarps];
  LncItem<W, CPL> it;
  it.init(g, p.x, E);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float2* recs = reinterpret_cast<float2*>(p.ws + g.rec_off);
  LncBulk<2, CPL> ring;
  {
    const char* const base[2] = {p.dy, p.x};
    ring.init(lnc_smem, it, g, base, E, true);
  }
  lnc_start(ring, it);
  bool dead = false;
  float gm[CPL][W], ag[CPL][W], ab[CPL][W];
#pragma unroll
  for (int j = 0; j < CPL; ++j) {
#pragma unroll
    for (int e = 0; e < W; ++e) gm[j][e] = ag[j][e] = ab[j][e] = 0.f;
    if (it.has(j)) lnc_vec_chunk<DT, W>(p.gamma, g.cols, it.col0(j, E), gm[j]);
  }
  const bool ragged = lnc_warp_ragged<W, CPL>(it.lo, it.hi);
  // this warp's slice of row i: its column partials, and (S1, S2) of the lanes
  auto row_sums = [&](int i, float mean, float rstd, float& s1, float& s2, auto tag) {
    constexpr bool M = decltype(tag)::value;
    float s1a = 0.f, s1b = 0.f, s2a = 0.f, s2b = 0.f;
    if (rstd != 0.f) {  // a masked row adds nothing
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        if (M && !it.has(j)) continue;
        float dv[W], xv[W];
        lnc_unpack<DT, W>(ring.at(i, 0, j), dv);
        lnc_unpack<DT, W>(ring.at(i, 1, j), xv);
        if constexpr (M) {
          lnc_clip<W>(dv, it.lo[j], it.hi[j]);
          lnc_clip<W>(xv, it.lo[j], it.hi[j]);
        }
#pragma unroll
        for (int e = 0; e < W; e += 2) {
          float h0, h1;
          if constexpr (RMS) {
            mul2(h0, h1, xv[e], xv[e + 1], rstd, rstd);
          } else {
            add2(h0, h1, xv[e], xv[e + 1], -mean, -mean);
            mul2(h0, h1, h0, h1, rstd, rstd);
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
    s1 = s1a + s1b;
    s2 = s2a + s2b;
  };
  const float* pm = p.mean + it.r0;
  const float* pr = p.rstd + it.r0;
  const int64_t sP = g.P;
  for (int i = 0; i < it.nr; i += 2, pm += 2 * sP, pr += 2 * sP) {
    const bool two = i + 1 < it.nr;
    const float mean0 = RMS ? 0.f : __ldg(pm), rstd0 = __ldg(pr);
    const float mean1 = RMS || !two ? 0.f : __ldg(pm + sP), rstd1 = two ? __ldg(pr + sP) : 0.f;
    lnc_next2(ring, i, it.nr, it.rstep, dead, p.err);
    float s[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
    if (ragged) {
      row_sums(i, mean0, rstd0, s[0][0], s[0][1], LncMask<true>());
      if (two) row_sums(i + 1, mean1, rstd1, s[1][0], s[1][1], LncMask<true>());
    } else {
      row_sums(i, mean0, rstd0, s[0][0], s[0][1], LncMask<false>());
      if (two) row_sums(i + 1, mean1, rstd1, s[1][0], s[1][1], LncMask<false>());
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if constexpr (!RMS) s[u][0] = lnc_warp_sum(s[u][0]);
      s[u][1] = lnc_warp_sum(s[u][1]);
    }
    if (lane == 0) {
      part[i % RS][warp] = make_float2(s[0][0], s[0][1]);
      if (two) part[(i + 1) % RS][warp] = make_float2(s[1][0], s[1][1]);
    }
    const int done = min(i + 2, it.nr);
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
        recs[(it.r0 + (int64_t)(base + ri) * g.P) * g.nb + it.b] = t;
      }
      __syncthreads();
    }
  }
  if (dead && threadIdx.x == 0) ring.drain(it.nr, p.err);
  // the item's column partials: every column of the block, zeros included
  float* out = p.ws + ((int64_t)it.cls * g.ng + it.grp) * kPlanes * g.cols;
#pragma unroll
  for (int j = 0; j < CPL; ++j) {
    if (!it.has(j)) continue;
    const int64_t c0 = it.col0(j, E);
#pragma unroll
    for (int e = 0; e < W; ++e) {
      if (e < it.lo[j] || e >= it.hi[j]) continue;
      out[c0 + e] = ag[j][e];
      if constexpr (!RMS) out[g.cols + c0 + e] = ab[j][e];
    }
  }
}

// Launch 2: dx from dy, x (read again), mean / rstd, gamma and the row's
// (S1, S2) summed over its column blocks.
template <int DT, bool RMS, int CPL>
__global__ void __launch_bounds__(kLncThreads, 6) lnc_bwd_dx_kernel(const LnBwdParams p,
                                                                 const LncGeo g) {
  constexpr int E = DType<DT>::E, W = DType<DT>::V;
  extern __shared__ __align__(128) unsigned char lnc_smem[];
  LncItem<W, CPL> it;
  it.init(g, p.x, E);
  const int64_t rowb = g.cols * E;
  const int lane = threadIdx.x & 31;
  LncBulk<2, CPL> ring;
  {
    const char* const base[2] = {p.dy, p.x};
    ring.init(lnc_smem, it, g, base, E, false);
  }
  lnc_start(ring, it);
  bool dead = false;
  float gm[CPL][W];
#pragma unroll
  for (int j = 0; j < CPL; ++j) {
#pragma unroll
    for (int e = 0; e < W; ++e) gm[j][e] = 0.f;
    if (it.has(j)) lnc_vec_chunk<DT, W>(p.gamma, g.cols, it.col0(j, E), gm[j]);
  }
  const bool ragged = lnc_warp_ragged<W, CPL>(it.lo, it.hi);
  // dx of this warp's slice of row i (lane-wise stores only in ragged warps)
  auto row_dx = [&](int i, float mean, float rstd, float a, float bq, char* out, auto tag) {
    constexpr bool M = decltype(tag)::value;
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
      if (M && !it.has(j)) continue;
      float o[W];
      if (rstd == 0.f) {
#pragma unroll
        for (int e = 0; e < W; ++e) o[e] = 0.f;
      } else {
        float dv[W], xv[W];
        lnc_unpack<DT, W>(ring.at(i, 0, j), dv);
        lnc_unpack<DT, W>(ring.at(i, 1, j), xv);
#pragma unroll
        for (int e = 0; e < W; e += 2) {
          float h0, h1, t0, t1b;
          if constexpr (RMS) {
            mul2(h0, h1, xv[e], xv[e + 1], rstd, rstd);
          } else {
            add2(h0, h1, xv[e], xv[e + 1], -mean, -mean);
            mul2(h0, h1, h0, h1, rstd, rstd);
          }
          const float g0 = __fmul_rn(dv[e], gm[j][e]), g1 = __fmul_rn(dv[e + 1], gm[j][e + 1]);
          add2(t0, t1b, g0, g1, -a, -a);               // g - S1 / C
          fma2(t0, t1b, h0, h1, -bq, -bq, t0, t1b);    // - xhat S2 / C
          mul2(o[e], o[e + 1], t0, t1b, rstd, rstd);
        }
      }
      if constexpr (M) lnc_store<DT, W>(out + kLncStride * j, it.lo[j], it.hi[j], o);
      else st_chunk_stream(out + kLncStride * j, chunk_pack<DT>(o));
    }
  };
  char* out = const_cast<char*>(it.at_row(p.dx, 0, g, rowb));
  const float* pm = p.mean + it.r0;
  const float* pr = p.rstd + it.r0;
  const float2* rec = reinterpret_cast<const float2*>(p.ws + g.rec_off) + it.r0 * g.nb;
  const int64_t sP = g.P, rec_step = (int64_t)g.P * g.nb;
  for (int i = 0; i < it.nr; i += 2, out += 2 * it.rstep, pm += 2 * sP, pr += 2 * sP,
           rec += 2 * rec_step) {
    const bool two = i + 1 < it.nr;
    float mean[2], rstd[2], a[2], bq[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      mean[u] = RMS || (u && !two) ? 0.f : __ldg(pm + u * sP);
      rstd[u] = u && !two ? 0.f : __ldg(pr + u * sP);
      // the row's sums: lane l adds records l, l + 32, ... in order, then the
      // lanes' sums by an ordered butterfly
      float t1 = 0.f, t2 = 0.f;
      if (u == 0 || two)
        for (int b = lane; b < g.nb; b += 32) {
          const float2 s = __ldg(rec + u * rec_step + b);
          t1 += s.x;
          t2 += s.y;
        }
      a[u] = t1;
      bq[u] = t2;
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      a[u] = (RMS ? 0.f : lnc_warp_sum(a[u])) * p.inv_cols;
      bq[u] = lnc_warp_sum(bq[u]) * p.inv_cols;
    }
    lnc_next2(ring, i, it.nr, it.rstep, dead, p.err);
    if (ragged) {
      row_dx(i, mean[0], rstd[0], a[0], bq[0], out, LncMask<true>());
      if (two) row_dx(i + 1, mean[1], rstd[1], a[1], bq[1], out + it.rstep, LncMask<true>());
    } else {
      row_dx(i, mean[0], rstd[0], a[0], bq[0], out, LncMask<false>());
      if (two) row_dx(i + 1, mean[1], rstd[1], a[1], bq[1], out + it.rstep, LncMask<false>());
    }
  }
  if (dead && threadIdx.x == 0) ring.drain(it.nr, p.err);
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
