// rr_engine.cuh -- the row engine shared by every operation.
//
// A row (or, for very long rows, one of K column slices of a row held by the
// K CTAs of a thread-block cluster) is owned by a group of G threads.  Each
// thread holds its share of the row in registers as 16-byte chunks ("chunk
// mode", W = 16 / element size) or single elements ("element mode", W = 1,
// used when row starts are not 16-byte aligned and per-column vectors are
// involved).  One pass over global memory loads the share, the per-thread
// statistic is merged across the group with an ordered butterfly (warp
// shuffles, then shared memory between warps, then distributed shared memory
// between the CTAs of a cluster), and the outputs are written from registers.
//
// Two ways to bring a row in:
//   * direct: every thread issues its own 128-bit loads (ragged heads and tails
//     element by element) and already holds the next row while it reduces the
//     current one (register double buffer);
//   * staged (one group per CTA): a single thread issues 1-D bulk copies
//     (cp.async.bulk, the TMA engine) of the 16-byte aligned interior of the
//     next rows into shared-memory buffers, completing on an mbarrier; threads
//     read their chunks out of shared memory.
//
// The operation (softmax / cross-entropy, LayerNorm fwd, LayerNorm bwd) is a
// policy class `Op`; see the rr_op_*.cuh headers.
#pragma once

#include <type_traits>

#include "rr_device.cuh"

namespace rr {

// Launch-wide description shared by all operations.
struct Geo {
  int64_t rows;
  int64_t cols;
  int64_t slice;     // columns per cluster rank (== cols when the cluster is 1 CTA)
  int32_t nbuf;      // staged mode: shared-memory row buffers (1 or 2)
  int32_t buf_bytes; // staged mode: bytes of one buffer of one tensor
  int32_t red_off;   // byte offset of the reduction scratch in dynamic smem
  int32_t col_off;   // byte offset of the per-group column scratch (LN bwd)
};

// Registers holding one thread's share of a row for NT tensors.
template <int DT, int W, int NT, int NQ>
struct RowRegs {
  static constexpr int E = DType<DT>::E;
  static constexpr bool kChunk = (W > 1);
  using Slot = typename std::conditional<kChunk, uint4, float>::type;
  Slot v[NT][NQ];

  __device__ __forceinline__ float get(int t, int q, int e) const {
    if constexpr (kChunk) return chunk_get<DT>(v[t][q], e);
    else return v[t][q];
  }
};

// Where one thread's chunks of the current row slice live.  Indices inside a
// row are 32-bit (rows are limited to 2^31 columns); per row the thread's
// chunk count and the range of its full (fully valid) chunks are computed once.
template <int DT, int W>
struct RowGeo {
  static constexpr int E = DType<DT>::E;
  static constexpr bool kChunk = (W > 1);
  int c0, c1;       // valid columns of the slice
  int colbase;      // column of element 0 of chunk 0 (c0 - head in chunk mode)
  int nch;          // chunks (elements in element mode) of the slice
  int first;        // this thread's first chunk index
  int step;         // chunk stride between a thread's chunks (= G)
  int head_bytes;   // (slice start) - (chunk 0 address), 0..15 (chunk mode)
  int nq;           // chunks this thread owns
  int qlo, qhi;     // its chunks q in [qlo, qhi) are full

  __device__ __forceinline__ void init(int64_t c0_, int64_t c1_, uint64_t start_addr,
                                       int first_, int step_) {
    c0 = static_cast<int>(c0_);
    c1 = static_cast<int>(c1_);
    first = first_;
    step = step_;
    int cf_lo, cf_hi;
    if constexpr (kChunk) {
      const int head = static_cast<int>(start_addr & 15u) / E;
      head_bytes = head * E;
      colbase = c0 - head;
      const int span = head + (c1 - c0);
      nch = span > 0 ? (span + W - 1) / W : 0;
      cf_lo = head > 0 ? 1 : 0;
      cf_hi = span > 0 ? span / W : 0;
    } else {
      head_bytes = 0;
      colbase = c0;
      nch = c1 > c0 ? c1 - c0 : 0;
      cf_lo = 0;
      cf_hi = nch;
    }
    nq = nch > first ? (nch - first + step - 1) / step : 0;
    qlo = first < cf_lo ? 1 : 0;
    qhi = cf_hi > first ? (cf_hi - first + step - 1) / step : 0;
  }
  __device__ __forceinline__ int chunk(int q) const { return first + q * step; }
  __device__ __forceinline__ bool has(int q) const { return q < nq; }
  __device__ __forceinline__ int col(int q, int e) const { return colbase + chunk(q) * W + e; }
  __device__ __forceinline__ bool full(int q) const { return q >= qlo && q < qhi; }
  __device__ __forceinline__ bool valid(int q, int e) const {
    const int j = col(q, e);
    return j >= c0 && j < c1;
  }
  // Byte offset of chunk q from the slice's chunk-0 address.
  __device__ __forceinline__ int64_t off(int q) const {
    return kChunk ? (int64_t)chunk(q) * 16 : (int64_t)chunk(q) * E;
  }
  // (q, e) of column j if this thread owns it, else q = -1.
  __device__ __forceinline__ void locate(int j, int& q, int& e) const {
    q = -1;
    e = 0;
    const int lc = j - colbase;
    if (j < c0 || j >= c1 || lc < 0) return;
    const int c = lc / W;
    const int d = c - first;
    if (d < 0 || d % step != 0) return;
    if (d / step >= nq) return;
    q = d / step;
    e = lc - c * W;
  }

  // Calls f(q, e) for every valid element this thread owns.
  template <int NQ, class F>
  __device__ __forceinline__ void for_each(F f) const {
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      if (!has(q)) break;
      if (full(q)) {
#pragma unroll
        for (int e = 0; e < W; ++e) f(q, e);
      } else {
#pragma unroll
        for (int e = 0; e < W; ++e)
          if (valid(q, e)) f(q, e);
      }
    }
  }

  // Stores out(q, e) for every valid element of this thread; g0 is the chunk-0
  // address of the output slice.
  template <int NQ, class F>
  __device__ __forceinline__ void store(char* g0, F out) const {
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      if (!has(q)) break;
      char* p = g0 + off(q);
      if constexpr (kChunk) {
        if (full(q)) {
          float f[W];
#pragma unroll
          for (int e = 0; e < W; ++e) f[e] = out(q, e);
          st_chunk_stream(p, chunk_pack<DT>(f));
        } else {
#pragma unroll
          for (int e = 0; e < W; ++e)
            if (valid(q, e)) st_elem<DT>(p + e * E, out(q, e));
        }
      } else {
        st_elem<DT>(p, out(q, 0));
      }
    }
  }

  // Stores chunk q from the W values f[] (only its valid elements if ragged).
  __device__ __forceinline__ void store_chunk(char* g0, int q, const float* f) const {
    char* p = g0 + off(q);
    if constexpr (kChunk) {
      if (full(q)) {
        st_chunk_stream(p, chunk_pack<DT>(f));
      } else {
#pragma unroll
        for (int e = 0; e < W; ++e)
          if (valid(q, e)) st_elem<DT>(p + e * E, f[e]);
      }
    } else {
      st_elem<DT>(p, f[0]);
    }
  }
};

// Direct load of a thread's share of tensor t (fill = value for ragged slots).
template <int DT, int W, int NT, int NQ>
__device__ __forceinline__ void load_direct(RowRegs<DT, W, NT, NQ>& r, int t,
                                            const RowGeo<DT, W>& g, const char* g0,
                                            float fill) {
  constexpr int E = DType<DT>::E;
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    if (!g.has(q)) break;
    const char* p = g0 + g.off(q);
    if constexpr (W > 1) {
      if (g.full(q)) {
        r.v[t][q] = ld_chunk_stream(p);
      } else {
        uint4 c = chunk_fill<DT>(fill);
#pragma unroll
        for (int e = 0; e < W; ++e)
          if (g.valid(q, e)) chunk_set_bits<DT>(c, e, ld_elem_bits<DT>(p + e * E));
        r.v[t][q] = c;
      }
    } else {
      r.v[t][q] = ld_elem<DT>(p);
    }
  }
}

// Staged load: full chunks (interior elements) come from the shared-memory
// mirror of the slice, whose byte 0 corresponds to address floor16(slice start);
// ragged pieces are read from global memory.
template <int DT, int W, int NT, int NQ>
__device__ __forceinline__ void load_staged(RowRegs<DT, W, NT, NQ>& r, int t,
                                            const RowGeo<DT, W>& g, const char* g0,
                                            const unsigned char* sbuf, float fill) {
  constexpr int E = DType<DT>::E;
  const uint64_t a = reinterpret_cast<uint64_t>(g0);
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    if (!g.has(q)) break;
    const char* p = g0 + g.off(q);
    if constexpr (W > 1) {
      if (g.full(q)) {
        r.v[t][q] = *reinterpret_cast<const uint4*>(sbuf + g.off(q));
      } else {
        uint4 c = chunk_fill<DT>(fill);
#pragma unroll
        for (int e = 0; e < W; ++e)
          if (g.valid(q, e)) chunk_set_bits<DT>(c, e, ld_elem_bits<DT>(p + e * E));
        r.v[t][q] = c;
      }
    } else {
      // element mode: g0 is the slice start itself; the mirror starts at floor16
      const uint64_t ea = a + g.off(q);
      const uint64_t lo = (a + 15) & ~uint64_t(15);
      const uint64_t hi = (a + (uint64_t)(g.c1 - g.c0) * E) & ~uint64_t(15);
      if (ea >= lo && ea < hi)
        r.v[t][q] = ld_smem_elem<DT>(reinterpret_cast<const char*>(sbuf) + (ea - (a & ~uint64_t(15))));
      else
        r.v[t][q] = ld_elem<DT>(p);
    }
  }
}

// Group-wide reduction of a statistic for groups of G threads (G <= 32: warp
// shuffles only; G > 32: shuffles, then the per-warp results through shared
// memory and a named barrier for the group).  `red` points at this group's
// scratch of 2 x 32 statistics (double-buffered by row parity).
template <class S, int G, class M>
__device__ __forceinline__ S reduce_group(S s, M merge, S* red, int parity, int gt,
                                          int bar_id) {
  if constexpr (S::kNary) {
    // n-ary form of the pairwise merge: M = max_i m_i, D = sum_i d_i e^(m_i - M);
    // butterflies of max and of plain sums are bitwise identical on every lane.
    s = S::template nary<(G < 32 ? G : 32)>(s);
    if constexpr (G > 32) {
      const int lane = threadIdx.x & 31;
      S* slot = red + parity * 32;
      if (lane == 0) slot[gt >> 5] = s;
      named_bar(bar_id, G);
      s = S::template nary<32>((lane < G / 32) ? slot[lane] : S::identity());
    }
    return s;
  } else if constexpr (G <= 32) {
    return group_reduce<S, M, G>(s, merge);
  } else {
    s = group_reduce<S, M, 32>(s, merge);
    const int lane = threadIdx.x & 31;
    const int w = gt >> 5;
    S* slot = red + parity * 32;
    if (lane == 0) slot[w] = s;
    named_bar(bar_id, G);
    S o = (lane < G / 32) ? slot[lane] : S::identity();
    return group_reduce<S, M, 32>(o, merge);
  }
}

// Merge of the K per-CTA statistics of a cluster through distributed shared
// memory; slot is this CTA's 2-entry slot array (double-buffered by parity).
template <class S, class M>
__device__ __forceinline__ S reduce_cluster(S s, M merge, S* slot, int parity, int K) {
  if (threadIdx.x == 0) slot[parity] = s;
  cluster_sync();
  const int lane = threadIdx.x & 31;
  S o = S::identity();
  if (lane < K) o = S::load_remote(map_to_rank(&slot[parity], lane));
  return group_reduce<S, M, 32>(o, merge);
}

// The engine.  G threads per row group; T = blockDim.x (multiple of G);
// NQ = chunks per thread; STAGED = rows brought in by bulk copies (G == T).
template <class Op, int G, int NQ, int MAXT, bool STAGED>
__global__ void __launch_bounds__(MAXT) row_kernel(const typename Op::Params p, const Geo geo) {
  constexpr int DT = Op::DT, W = Op::W, NT = Op::NT;
  constexpr int E = DType<DT>::E;
  using S = typename Op::Stats;
  extern __shared__ __align__(128) unsigned char smem[];

  const int T = blockDim.x;
  const int ngroups = T / G;
  const int grp = threadIdx.x / G;
  const int gt = threadIdx.x % G;
  int K = 1, rank = 0;
  if constexpr (STAGED) {
    K = static_cast<int>(cluster_nrank());
    rank = static_cast<int>(cluster_rank());
  }
  const int64_t cid = blockIdx.x / K;
  const int64_t ncl = gridDim.x / K;
  const int64_t c0 = rank * geo.slice;
  const int64_t c1 = c0 + geo.slice < geo.cols ? c0 + geo.slice : geo.cols;
  const int64_t step = ncl * ngroups;
  const int64_t my_first = cid * ngroups + grp;
  // first row of the warp's first group: keeps sub-warp groups in lock step
  const int64_t warp_first = cid * ngroups + ((threadIdx.x & ~31) / G);

  S* red = reinterpret_cast<S*>(smem + geo.red_off) + (G > 32 ? grp * 64 : 0);
  S* cl_slot = reinterpret_cast<S*>(smem + geo.red_off) + 64 * (ngroups > 0 ? ngroups : 1);
  const int bar_id = 1 + grp;

  typename Op::Thread ts;
  Op::thread_init(ts, p, geo, c0, c1, gt, G);

  RowRegs<DT, W, NT, NQ> cur;

  if constexpr (!STAGED) {
    // ------------------------------------------------ direct, register double buffer
    typename Op::Meta m_cur = Op::meta(p, my_first < geo.rows ? my_first : -1);
    RowGeo<DT, W> g_cur;
    if (my_first < geo.rows) {
      g_cur.init(c0, c1, Op::start_addr(p, my_first, c0), gt, G);
      if (!Op::skip(m_cur))
#pragma unroll
        for (int t = 0; t < NT; ++t)
          load_direct(cur, t, g_cur, Op::in_chunk0(p, t, my_first, c0, g_cur), Op::fill());
    }
    for (int64_t i = 0;; ++i) {
      const int64_t wr = warp_first + i * step;
      if (wr >= geo.rows) break;
      const int64_t r = my_first + i * step;
      const bool active = r < geo.rows;
      // prefetch the next row into a second register set
      const int64_t rn = r + step;
      typename Op::Meta m_nxt = Op::meta(p, rn < geo.rows ? rn : -1);
      RowGeo<DT, W> g_nxt;
      RowRegs<DT, W, NT, NQ> nxt;
      if (rn < geo.rows) {
        g_nxt.init(c0, c1, Op::start_addr(p, rn, c0), gt, G);
        if (!Op::skip(m_nxt))
#pragma unroll
          for (int t = 0; t < NT; ++t)
            load_direct(nxt, t, g_nxt, Op::in_chunk0(p, t, rn, c0, g_nxt), Op::fill());
      }
      const bool use = active && !Op::skip(m_cur);
      S s = use ? Op::thread_stats(ts, cur, g_cur, m_cur) : S::identity();
      s = reduce_group<S, G>(s, typename Op::Merge(), red, static_cast<int>(i & 1), gt, bar_id);
      if (active) Op::finish(ts, p, geo, r, m_cur, s, cur, g_cur, gt == 0);
      cur = nxt;
      g_cur = g_nxt;
      m_cur = m_nxt;
    }
    Op::epilogue(ts, p, geo, smem + geo.col_off, c0, c1, cid, grp, ngroups, gt, G);
  } else {
    // ------------------------------------------------ staged through shared memory
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)geo.nbuf * NT * geo.buf_bytes);
    const uint64_t policy = policy_evict_first();
    if (threadIdx.x == 0) {
      for (int b = 0; b < geo.nbuf; ++b) mbar_init(&bars[b], 1);
      fence_mbar_init();
    }
    __syncthreads();
    // Issues the bulk copies of row r into buffer b (thread 0 only).
    auto issue = [&](int64_t r, int b) {
      uint32_t total = 0;
      uint64_t lo[NT], hi[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const uint64_t s0 = reinterpret_cast<uint64_t>(Op::in_slice_start(p, t, r, c0));
        const uint64_t s1 = s0 + (uint64_t)(c1 - c0) * E;
        lo[t] = (s0 + 15) & ~uint64_t(15);
        hi[t] = s1 & ~uint64_t(15);
        if (hi[t] > lo[t]) total += static_cast<uint32_t>(hi[t] - lo[t]);
      }
      if (total == 0) return;
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(&bars[b], total);
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        if (hi[t] > lo[t]) {
          // shared byte 0 of the buffer mirrors floor16(slice start)
          const uint64_t s0 = reinterpret_cast<uint64_t>(Op::in_slice_start(p, t, r, c0));
          unsigned char* d =
              smem + ((size_t)b * NT + t) * geo.buf_bytes + (lo[t] - (s0 & ~uint64_t(15)));
          bulk_load(d, reinterpret_cast<const void*>(lo[t]),
                    static_cast<uint32_t>(hi[t] - lo[t]), &bars[b], policy);
        }
      }
    };
    // Whether row r is brought in by a copy (same answer on every thread).
    auto copied = [&](int64_t r, const typename Op::Meta& m) -> bool {
      if (Op::skip(m)) return false;
      const uint64_t s0 = reinterpret_cast<uint64_t>(Op::in_slice_start(p, 0, r, c0));
      const uint64_t s1 = s0 + (uint64_t)(c1 - c0) * E;
      bool any = ((s1 & ~uint64_t(15)) > ((s0 + 15) & ~uint64_t(15)));
      if constexpr (NT > 1) {
        const uint64_t u0 = reinterpret_cast<uint64_t>(Op::in_slice_start(p, 1, r, c0));
        const uint64_t u1 = u0 + (uint64_t)(c1 - c0) * E;
        any = any || ((u1 & ~uint64_t(15)) > ((u0 + 15) & ~uint64_t(15)));
      }
      return any;
    };
    if (threadIdx.x == 0) {
      for (int b = 0; b < geo.nbuf; ++b) {
        const int64_t r = cid + (int64_t)b * ncl;
        if (r < geo.rows && !Op::skip(Op::meta(p, r))) issue(r, b);
      }
    }
    uint32_t phase = 0;  // bit b: parity of the next completion of buffer b
    // per-row metadata is loaded one row ahead (and, for the copy issuer, the
    // row nbuf ahead) so no global load sits on the per-row critical path
    typename Op::Meta m_next = Op::meta(p, cid < geo.rows ? cid : -1);
    for (int64_t i = 0;; ++i) {
      const int64_t r = cid + i * ncl;
      if (r >= geo.rows) break;
      const int b = static_cast<int>(i % geo.nbuf);
      const typename Op::Meta m = m_next;
      m_next = Op::meta(p, r + ncl < geo.rows ? r + ncl : -1);
      const int64_t rfar = r + (int64_t)geo.nbuf * ncl;
      typename Op::Meta m_far{};
      if (threadIdx.x == 0 && rfar < geo.rows) m_far = Op::meta(p, rfar);
      RowGeo<DT, W> g;
      g.init(c0, c1, Op::start_addr(p, r, c0), gt, G);
      const bool use = !Op::skip(m);
      if (use) {
        if (copied(r, m)) {
          mbar_wait_bounded(&bars[b], (phase >> b) & 1u, p.err);
          phase ^= (1u << b);
        }
#pragma unroll
        for (int t = 0; t < NT; ++t)
          load_staged(cur, t, g, Op::in_chunk0(p, t, r, c0, g),
                      smem + ((size_t)b * NT + t) * geo.buf_bytes, Op::fill());
      }
      S s = use ? Op::thread_stats(ts, cur, g, m) : S::identity();
      s = reduce_group<S, G>(s, typename Op::Merge(), red, static_cast<int>(i & 1), gt, bar_id);
      // every thread is done reading buffer b: refill it with the row nbuf ahead
      if (threadIdx.x == 0 && rfar < geo.rows && !Op::skip(m_far)) issue(rfar, b);
      if (K > 1) s = reduce_cluster<S>(s, typename Op::Merge(), cl_slot, static_cast<int>(i & 1), K);
      Op::finish(ts, p, geo, r, m, s, cur, g, gt == 0 && rank == 0);
    }
    Op::epilogue(ts, p, geo, smem + geo.col_off, c0, c1, cid, 0, 1, gt, G);
    if (K > 1) cluster_sync();  // peers may still read this CTA's slots
  }
}

}  // namespace rr
