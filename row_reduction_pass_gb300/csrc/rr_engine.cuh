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
  // Every chunk this thread owns is full (rows without a ragged head or tail):
  // loads and stores can skip the per-chunk checks.
  __device__ __forceinline__ bool all_full() const { return qlo == 0 && qhi >= nq; }
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

// Direct load of a thread's share of tensor t in memory-aligned chunks (fill =
// value for ragged slots).
template <int DT, int W, int NT, int NQ>
__device__ __forceinline__ void load_direct_mem(RowRegs<DT, W, NT, NQ>& r, int t,
                                            const RowGeo<DT, W>& g, const char* g0,
                                            float fill) {
  constexpr int E = DType<DT>::E;
  // rows without a ragged head or tail: no per-chunk checks (one-tensor
  // operations, or several chunks per thread; in the two-chunk two-tensor
  // ones, which also hold the next row, the second copy of the loop cost
  // registers and spilled)
  if constexpr (W > 1 && (NQ > 2 || NT == 1)) {
    if (g.all_full()) {
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        if (!g.has(q)) break;
        r.v[t][q] = ld_chunk_stream(g0 + g.off(q));
      }
      return;
    }
  }
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
__device__ __forceinline__ void load_staged_mem(RowRegs<DT, W, NT, NQ>& r, int t,
                                            const RowGeo<DT, W>& g, const char* g0,
                                            const unsigned char* sbuf, float fill) {
  constexpr int E = DType<DT>::E;
  const uint64_t a = reinterpret_cast<uint64_t>(g0);
  if constexpr (W > 1) {
    if (g.all_full()) {
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        if (!g.has(q)) break;
        r.v[t][q] = *reinterpret_cast<const uint4*>(sbuf + g.off(q));
      }
      return;
    }
  }
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

// Loads a thread's column-aligned chunks of one row tensor.  Chunk k covers
// columns c0 + kW .. c0 + kW + W - 1 of the slice and sits at s0 + 16k, where s0
// (the slice start) may have any element alignment: an aligned chunk is one
// 128-bit load; a misaligned one is the funnel shift of the two aligned chunks
// holding it (from the shared-memory mirror when staged, else through L1), or
// element loads where those would leave [tbeg, tend).  The last chunk of a row
// may be ragged (columns >= c1 are filled with 0).
template <int DT, int W, int NT, int NQ>
__device__ __forceinline__ void load_cols(RowRegs<DT, W, NT, NQ>& r, int t, const RowGeo<DT, W>& g,
                                          const char* s0, const char* tbeg, const char* tend,
                                          const unsigned char* sbuf) {
  constexpr int E = DType<DT>::E;
  const uintptr_t sa = reinterpret_cast<uintptr_t>(s0);
  const int h = static_cast<int>(sa & 15);
  const uintptr_t mbase = sa & ~uintptr_t(15);
  const uintptr_t mlo = (sa + 15) & ~uintptr_t(15);
  const uintptr_t mhi = (sa + (uintptr_t)(g.c1 - g.c0) * E) & ~uintptr_t(15);
  const uintptr_t tb = reinterpret_cast<uintptr_t>(tbeg), te = reinterpret_cast<uintptr_t>(tend);
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    if (!g.has(q)) break;
    const char* a = s0 + (int64_t)g.chunk(q) * (W * E);
    const uintptr_t aa = reinterpret_cast<uintptr_t>(a);
    if constexpr (W > 1) {
      if (g.full(q)) {
        if (h == 0) {
          r.v[t][q] = sbuf ? *reinterpret_cast<const uint4*>(sbuf + (aa - mbase)) : ld_chunk_stream(a);
          continue;
        }
        const uintptr_t fa = aa & ~uintptr_t(15);
        if (sbuf != nullptr && fa >= mlo && fa + 32 <= mhi) {
          const uint4* m = reinterpret_cast<const uint4*>(sbuf + (fa - mbase));
          r.v[t][q] = funnel16(m[0], m[1], h);
          continue;
        }
        if (sbuf == nullptr && fa >= tb && fa + 32 <= te) {
          r.v[t][q] = ld16_split(a);
          continue;
        }
      }
      uint4 c = make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int e = 0; e < W; ++e)
        if (g.valid(q, e)) chunk_set_bits<DT>(c, e, ld_elem_bits<DT>(a + e * E));
      r.v[t][q] = c;
    } else {
      if (sbuf != nullptr && aa >= mlo && aa < mhi)
        r.v[t][q] = ld_smem_elem<DT>(reinterpret_cast<const char*>(sbuf) + (aa - mbase));
      else
        r.v[t][q] = ld_elem<DT>(a);
    }
  }
}

// Stores column-aligned chunk q, already packed into storage bits (chunk mode).
template <int DT, int W>
__device__ __forceinline__ void store_cols_bits(const RowGeo<DT, W>& g, char* s0, int q,
                                                const uint4& v) {
  constexpr int E = DType<DT>::E;
  char* a = s0 + (int64_t)g.chunk(q) * (W * E);
  if (g.full(q)) {
    if ((reinterpret_cast<uintptr_t>(a) & 15) == 0) st_chunk_stream(a, v);
    else st16_split(a, v);
  } else {
#pragma unroll
    for (int e = 0; e < W; ++e)
      if (g.valid(q, e)) st_elem<DT>(a + e * E, chunk_get<DT>(v, e));
  }
}

// Stores column-aligned chunk q (W values f) of one row tensor whose slice
// starts at s0 (any element alignment): one 128-bit store when aligned, aligned
// 2/4/8-byte pieces when not, element stores for a ragged last chunk.
template <int DT, int W>
__device__ __forceinline__ void store_cols(const RowGeo<DT, W>& g, char* s0, int q, const float* f) {
  constexpr int E = DType<DT>::E;
  char* a = s0 + (int64_t)g.chunk(q) * (W * E);
  if constexpr (W > 1) {
    if (g.full(q)) {
      const uint4 v = chunk_pack<DT>(f);
      if ((reinterpret_cast<uintptr_t>(a) & 15) == 0) st_chunk_stream(a, v);
      else st16_split(a, v);
    } else {
#pragma unroll
      for (int e = 0; e < W; ++e)
        if (g.valid(q, e)) st_elem<DT>(a + e * E, f[e]);
    }
  } else {
    st_elem<DT>(a, f[0]);
  }
}

// Reductions of one thread's row statistics across its row group (and, for a
// row split over a cluster, across the cluster's CTAs).  An operation calls
// reduce() / cluster() as often as it needs per row; every thread of the group
// (and every CTA of the cluster) makes the same calls in the same order.
//   reduce():  G <= 32: warp shuffles only.  G > 32: shuffles, then the per-warp
//              results through shared memory and a named barrier for the group.
//   cluster(): the CTAs' results through distributed shared memory after a
//              cluster barrier (identity when the cluster is one CTA).
// Scratch slots are 16 bytes and double-buffered by call parity: a slot is
// rewritten two calls later, after a barrier every reader has passed.
// Statistic types S provide identity(), shfl_xor(), load_remote() and a
// kNary flag (with nary<L>() for the n-ary forms).
struct NoHook {
  __device__ __forceinline__ void operator()() const {}
};

template <int G, class Hook>
struct Reducer {
  unsigned char* red;  // this group's scratch: 2 parities x 32 warps x 16 B
  unsigned char* cl;   // this CTA's cluster slots: 2 parities x 16 B
  const Hook* hook;    // run once per row by thread 0 after the group's first barrier
  int& gcalls;
  int& ccalls;
  int gt, bar_id, K;
  bool hooked;

  template <class S, class M>
  __device__ __forceinline__ S reduce(S s, M merge) {
    static_assert(sizeof(S) <= 16, "statistic larger than a scratch slot");
    if constexpr (G <= 32) {
      if constexpr (S::kNary) return S::template nary<G>(s);
      else return group_reduce<S, M, G>(s, merge);
    } else {
      const int parity = gcalls & 1;
      ++gcalls;
      if constexpr (S::kNary) s = S::template nary<32>(s);
      else s = group_reduce<S, M, 32>(s, merge);
      const int lane = threadIdx.x & 31;
      unsigned char* base = red + parity * 512;
      if (lane == 0) *reinterpret_cast<S*>(base + 16 * (gt >> 5)) = s;
      named_bar(bar_id, G);
      if (!hooked) {
        hooked = true;
        if (threadIdx.x == 0) (*hook)();
      }
      const S o = (lane < G / 32) ? *reinterpret_cast<const S*>(base + 16 * lane) : S::identity();
      if constexpr (S::kNary) return S::template nary<32>(o);
      else return group_reduce<S, M, 32>(o, merge);
    }
  }

  template <class S, class M>
  __device__ __forceinline__ S cluster(S s, M merge) {
    if (K == 1) return s;
    const int parity = ccalls & 1;
    ++ccalls;
    S* slot = reinterpret_cast<S*>(cl + 16 * parity);
    if (threadIdx.x == 0) *slot = s;
    cluster_sync();
    const int lane = threadIdx.x & 31;
    S o = S::identity();
    if (lane < K) o = S::load_remote(map_to_rank(slot, lane));
    return group_reduce<S, M, 32>(o, merge);
  }
};

// The engine.  G threads per row group; T = blockDim.x (multiple of G);
// NQ = chunks per thread; STAGED = rows brought in by bulk copies (G == T).
// Direct variants are held to 64 registers per thread (full occupancy).
template <class Op, int G, int NQ, int MAXT, bool STAGED>
__global__ void __launch_bounds__(MAXT, STAGED ? 1 : 1024 / MAXT)
    row_kernel(const typename Op::Params p, const Geo geo) {
  constexpr int DT = Op::DT, W = Op::W, NT = Op::NT;
  constexpr int E = DType<DT>::E;
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

  unsigned char* red = smem + geo.red_off + (G > 32 ? grp * 1024 : 0);
  unsigned char* cl = smem + geo.red_off + 1024 * (ngroups > 0 ? ngroups : 1);
  int gcalls = 0, ccalls = 0;

  typename Op::Thread ts;
  Op::thread_init(ts, p, geo, c0, c1, gt, G, smem + geo.col_off, grp, ngroups);
  __syncthreads();  // per-group scratch initialised before any row is processed

  RowRegs<DT, W, NT, NQ> cur;

  if constexpr (!STAGED) {
    // ------------------------------------------------ direct
    constexpr bool kPre = Op::kPrefetch;  // register double buffer of the next row
    const NoHook nohook;
    typename Op::Meta m_cur = Op::meta(p, my_first < geo.rows ? my_first : -1);
    RowGeo<DT, W> g_cur;
    if (my_first < geo.rows) g_cur.init(c0, c1, Op::start_addr(p, my_first, c0), gt, G);
    if constexpr (kPre) {
      if (my_first < geo.rows && !Op::skip(m_cur)) Op::load_direct(cur, g_cur, p, geo, my_first, c0);
    }
    // two rows per trip for one-tensor operations, so the next row's
    // registers become the current ones by renaming, not by copies (the
    // two-tensor backward spilled when unrolled)
    constexpr int kRowUnroll = NT == 1 ? 2 : 1;
#pragma unroll kRowUnroll
    for (int64_t i = 0;; ++i) {
      const int64_t wr = warp_first + i * step;
      if (wr >= geo.rows) break;
      const int64_t r = my_first + i * step;
      const bool active = r < geo.rows;
      const int64_t rn = r + step;
      typename Op::Meta m_nxt = Op::meta(p, rn < geo.rows ? rn : -1);
      RowGeo<DT, W> g_nxt;
      if (rn < geo.rows) g_nxt.init(c0, c1, Op::start_addr(p, rn, c0), gt, G);
      RowRegs<DT, W, NT, NQ> nxt;
      if constexpr (kPre) {
        if (rn < geo.rows && !Op::skip(m_nxt)) Op::load_direct(nxt, g_nxt, p, geo, rn, c0);
      } else {
        if (active && !Op::skip(m_cur)) Op::load_direct(cur, g_cur, p, geo, r, c0);
      }
      Reducer<G, NoHook> rd{red, cl, &nohook, gcalls, ccalls, gt, 1 + grp, 1, true};
      Op::process(ts, p, geo, r, m_cur, cur, g_cur, gt == 0, active, rd);
      if constexpr (kPre) cur = nxt;
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
      bool any = false;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const uint64_t s0 = reinterpret_cast<uint64_t>(Op::in_slice_start(p, t, r, c0));
        const uint64_t s1 = s0 + (uint64_t)(c1 - c0) * E;
        any = any || ((s1 & ~uint64_t(15)) > ((s0 + 15) & ~uint64_t(15)));
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
      if (!Op::skip(m)) {
        if (copied(r, m)) {
          mbar_wait_bounded(&bars[b], (phase >> b) & 1u, p.err);
          phase ^= (1u << b);
        }
        Op::load_staged(cur, g, p, geo, r, c0, smem + (size_t)b * NT * geo.buf_bytes,
                        geo.buf_bytes);
      }
      // every thread is done reading buffer b once the row's first group
      // barrier is passed: refill it with the row nbuf ahead
      auto refill = [&]() {
        if (rfar < geo.rows && !Op::skip(m_far)) issue(rfar, b);
      };
      Reducer<G, decltype(refill)> rd{red, cl, &refill, gcalls, ccalls, gt, 1, K, false};
      Op::process(ts, p, geo, r, m, cur, g, gt == 0 && rank == 0, true, rd);
      if (!rd.hooked) {  // no group barrier this row: make one before the refill
        named_bar(1, G);
        if (threadIdx.x == 0) refill();
      }
    }
    Op::epilogue(ts, p, geo, smem + geo.col_off, c0, c1, cid, 0, 1, gt, G);
    if (K > 1) cluster_sync();  // peers may still read this CTA's slots
  }
}

}  // namespace rr
