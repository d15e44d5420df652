// rr_smx.cuh -- softmax, log-softmax and fused softmax cross-entropy for long
// rows, on the phase-aligned row layout of rr_lnx.cuh ("Engineering a CUDA
// Machine Learning Framework from Scratch", sec. 3.1 for the online
// normaliser, sec. 2.1 for the loss gradient fused into the pass, sec. 2.3 for
// the 128-bit accesses).
//
// Each row group brings its row (a cluster rank: its slice) into shared memory
// through a ring of stages, several rows ahead: every thread copies its own
// 16-byte chunks (gt, gt + G, ...) with asynchronous copies and is their only
// reader, so no barrier guards the data.  Every element is read from global
// memory once.  The row stays in its stage while the group works on it, so a
// thread holds no row in registers (many warps per SM hide the latencies);
// the chunks are read three times from there:
//   1. every thread takes the maximum m of its chunks, then d = sum of
//      2^(x log2 e - fl(m log2 e)) times 2^-r (r the rounding residual of
//      fl(m log2 e)), so d is the sum of exp(x - m); the (m, d) pairs (and,
//      for cross-entropy, the label's logit x_l, read by the thread whose
//      chunk holds it) are merged over the group and the cluster: M = max
//      m_i, D = sum d_i exp(m_i - M) (the merge of Milakov & Gimelshein's
//      online normaliser, taken over all partials at once);
//   2. softmax y = 2^(x log2 e - fl(M log2 e)) * (2^-r / d);  log-softmax
//      z = (x - M) - ln d;  cross-entropy dlogits = y - onehot (the label's
//      element is stored again by its owner, minus one), loss = (M - x_l) +
//      ln d.
// Lanes of the first and last chunk that belong to the neighbouring rows are
// set to -inf in the stage by the chunk's only reader before it reads them, so
// they change no maximum and add nothing to the sum.  A fully masked row
// (M = -inf) gives 0 everywhere (loss 0); an ignored label gives loss 0 and
// dlogits 0 (the row is not looked at); a label outside [0, cols) gives loss
// NaN, the plain softmax and one count in *bad.
//
// A row held by one warp is finished within its iteration: the warp's
// butterfly merge gives the row's statistics.  Otherwise the group's warps
// never wait on one another within a row: each warp
// publishes its partial of row j (to the slots of every rank of the cluster)
// and arrives on the row's merge barrier, then takes row j - 1's statistics
// (published one row earlier, so normally complete) and writes row j - 1's
// outputs.  So the merge latency and the warps' skew hide behind a row of
// work.  A thread refills a stage with the row NS ahead once it has written
// that stage's row's outputs.
#pragma once

#include <type_traits>

#include "rr_lnx.cuh"

namespace rr {

// A row's (or a partial's) maximum m, sum d of exp(x - m), and the label's
// logit x (-inf where it is not held).
struct MaxSumLab {
  float m, d, x;
  __device__ __forceinline__ static MaxSumLab identity() { return {-INFINITY, 0.f, -INFINITY}; }
};

// Largest of a chunk's values.
template <int DT> __device__ __forceinline__ float smx_chunk_max(const uint4& c);
template <> __device__ __forceinline__ float smx_chunk_max<kBF16>(const uint4& c) {
  const uint32_t w = bf16x2_max(bf16x2_max(c.x, c.y), bf16x2_max(c.z, c.w));
  return fmaxf(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
template <> __device__ __forceinline__ float smx_chunk_max<kF32>(const uint4& c) {
  return fmaxf(fmaxf(__uint_as_float(c.x), __uint_as_float(c.y)),
               fmaxf(__uint_as_float(c.z), __uint_as_float(c.w)));
}
template <int DT> __device__ __forceinline__ uint4 smx_neg_inf_chunk() {
  const uint32_t w = DT == kBF16 ? 0xff80ff80u : 0xff800000u;
  return make_uint4(w, w, w, w);
}

// In a landed stage, the lanes of this thread's head / tail chunk that belong
// to the neighbouring rows become -inf.
template <int DT, int W>
__device__ __forceinline__ void smx_mask_stage(uint4* st, const LnxRows<W>& rw, int gt, int G) {
  constexpr int E = DType<DT>::E;
  const uint32_t ninf = DT == kBF16 ? 0xff80ff80u : 0xff800000u;
  auto fill = [&](uint4& c, const uint4& keep) {
    c.x = (c.x & keep.x) | (ninf & ~keep.x);
    c.y = (c.y & keep.y) | (ninf & ~keep.y);
    c.z = (c.z & keep.z) | (ninf & ~keep.z);
    c.w = (c.w & keep.w) | (ninf & ~keep.w);
  };
  if (rw.hq == 0) fill(st[gt], lnx_byte_mask(rw.phi * E, 16));
  if (rw.tq >= 0) fill(st[gt + rw.tq * G], lnx_byte_mask(0, rw.tail_lanes * E));
}

// Step 1 for one thread over its chunks gt + q * G, q < nq: m = its maximum
// (one read of the chunks), then d = sum of 2^(x log2 e - fl(m log2 e)) times
// 2^-r, r the rounding residual of fl(m log2 e), so d is the sum of exp(x - m)
// (a second read); d = 0 when m = -inf.
template <int DT>
__device__ __forceinline__ MaxSum smx_thread_stats(const uint4* st, int gt, int G, int nq) {
  constexpr int W = DType<DT>::V;
  float m;
  if constexpr (DT == kBF16) {
    uint32_t m0 = 0xff80ff80u, m1 = m0, m2 = m0, m3 = m0;
#pragma unroll 4
    for (int q = 0; q < nq; ++q) {
      const uint4 c = st[gt + q * G];
      m0 = bf16x2_max(m0, c.x);
      m1 = bf16x2_max(m1, c.y);
      m2 = bf16x2_max(m2, c.z);
      m3 = bf16x2_max(m3, c.w);
    }
    const uint32_t w = bf16x2_max(bf16x2_max(m0, m1), bf16x2_max(m2, m3));
    m = fmaxf(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  } else {
    float m0 = -INFINITY, m1 = m0, m2 = m0, m3 = m0;
#pragma unroll 4
    for (int q = 0; q < nq; ++q) {
      const uint4 c = st[gt + q * G];
      m0 = fmaxf(m0, __uint_as_float(c.x));
      m1 = fmaxf(m1, __uint_as_float(c.y));
      m2 = fmaxf(m2, __uint_as_float(c.z));
      m3 = fmaxf(m3, __uint_as_float(c.w));
    }
    m = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
  }
  if (m == -INFINITY) return {m, 0.f};
  const float mL = m * kLog2e;
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll 2
  for (int q = 0; q < nq; ++q) {
    float v[W];
    lnx_unpack<DT, W>(st[gt + q * G], v);
#pragma unroll
    for (int e = 0; e < W; e += 4) {
      float t0, t1, t2, t3;
      fma2(t0, t1, v[e], v[e + 1], kLog2e, kLog2e, -mL, -mL);
      fma2(t2, t3, v[e + 2], v[e + 3], kLog2e, kLog2e, -mL, -mL);
      add2(a0, a1, a0, a1, ex2(t0), ex2(t1));
      add2(a2, a3, a2, a3, ex2(t2), ex2(t3));
    }
  }
  return {m, ((a0 + a1) + (a2 + a3)) * ex2(-fmaf(m, kLog2e, -mL))};
}

// Merge over the 32 lanes of a warp of partials (m_i, d_i) (and label logits
// x_i): M = max m_i, D = sum d_i * 2^((m_i - M) log2 e) (a lane with m_i =
// -inf adds nothing), X = max x_i.  Butterfly exchanges of commutative
// operations, so every lane ends with the same bits.
template <bool LAB>
__device__ __forceinline__ MaxSumLab smx_warp_merge(const MaxSumLab& v) {
  float M = v.m;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float d = v.m == -INFINITY ? 0.f : v.d * ex2((v.m - M) * kLog2e);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
  float x = v.x;
  if constexpr (LAB) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
  }
  return {M, d, x};
}

// MODE: 0 softmax, 1 log-softmax, 2 cross-entropy (labels).
template <int DT, int MODE, bool CL>
__global__ void __launch_bounds__(kSmxMaxT, 1) smx_kernel(const SoftmaxParams p, const LnxGeo g) {
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
  auto row_of = [&](int64_t j) { return rw.first + j * rw.step; };
  const int NS = g.NS;
  const int lane = threadIdx.x & 31, wg = gr.gt >> 5;
  // the group's merge barriers, by row parity: every warp of every rank
  // published its partial of the row
  uint64_t* mrg = reinterpret_cast<uint64_t*>(smem + g.bar_off) + (size_t)gr.grp * 2;
  // partial slots [row parity][rank][warp], 16 bytes each
  float4* slots = reinterpret_cast<float4*>(smem + g.red_off + (size_t)gr.grp * 1024 * K);
  const int nslot = K * gr.nw;
  // a one-warp group of a one-block row finishes each row in its own
  // iteration (no merge across warps): a stage is free one row earlier
  const bool solo = !CL && gr.nw == 1;
  const int ahead = solo ? NS - 1 : NS - 2;  // rows in flight beyond the current one
  uint4* ring = reinterpret_cast<uint4*>(smem + g.ring_off) + (size_t)gr.grp * NS * g.S;
  auto stage = [&](int64_t j) { return ring + (size_t)(j % NS) * g.S; };
  // each thread copies its own chunks of row j into the row's stage (it is
  // their only reader), one commit group per call (empty past the last row),
  // so "row j landed" is a wait for all but the `ahead` newer groups
  auto fetch = [&](int64_t j) {
    if (row_of(j) < g.rows) {
      const char* src = rw.slice(p.x, row_of(j), E);
      uint4* dst = stage(j);
      for (int q = 0; q < rw.nq; ++q) {
        const int k = gr.gt + q * gr.G;
        cp_async16(dst + k, src + (int64_t)k * 16);
      }
    }
    cp_async_commit();
  };
  auto landed = [&]() {
    if (ahead <= 0) cp_async_wait<0>();
    else if (ahead == 1) cp_async_wait<1>();
    else if (ahead == 2) cp_async_wait<2>();
    else cp_async_wait<3>();
  };
  bool dead = false;  // a wait gave up: later waits are skipped (the kernel still ends)
  if (gr.gt == 0) {
    mbar_init(&mrg[0], nslot);
    mbar_init(&mrg[1], nslot);
    fence_mbar_init();
  }
  for (int64_t i = 0; i < ahead; ++i) fetch(i);
  if constexpr (CL) cluster_sync();  // peers arrive on this block's barriers
  else __syncthreads();
  const int col0 = rw.k0 * W - rw.phi;  // column of lane 0 of local chunk 0

  // where the label's element is, when this thread holds it
  auto locate = [&](int32_t label, int& lk, int& le) {
    lk = -1;
    le = 0;
    if (label < 0 || (int64_t)label >= g.cols) return;
    const int kk = (label - col0) / W;  // label - col0 >= 0 for the rank that holds it
    if (label >= col0 && kk < rw.n && kk % gr.G == gr.gt) {
      lk = kk;
      le = label - col0 - kk * W;
    }
  };
  // this warp's partial of row j, to the slots of every rank
  auto publish = [&](int64_t j, MaxSumLab v) {
    v = smx_warp_merge<MODE == 2>(v);
    if (lane == 0) {
      const int par = static_cast<int>(j & 1);
      float4* sl = slots + par * nslot + rank * gr.nw + wg;
      if constexpr (CL) {
        for (int k = 0; k < K; ++k) {
          st_cluster_f32x4(map_to_rank(sl, k), v.m, v.d, v.x, 0.f);
          mbar_arrive_cluster(map_to_rank(&mrg[par], k));
        }
      } else {
        *sl = make_float4(v.m, v.d, v.x, 0.f);
        mbar_arrive(&mrg[par]);
      }
    }
  };
  // row j's statistics: every warp merges the slots the same way (lane l
  // takes slots l, l + 32, ...: their maximum, then the sum of their d
  // rescaled to the row maximum), so all threads of all ranks hold the same
  // bits
  auto merged = [&](int64_t j) {
    const int par = static_cast<int>(j & 1);
    const uint32_t ph = static_cast<uint32_t>((j >> 1) & 1);
    if (!dead) {
      if constexpr (CL) dead = !mbar_wait_bounded_cluster(&mrg[par], ph, p.err);
      else dead = !mbar_wait_bounded(&mrg[par], ph, p.err);
    }
    const float4* sl = slots + par * nslot;
    float m = -INFINITY, x = -INFINITY;
    for (int i = lane; i < nslot; i += 32) {
      m = fmaxf(m, sl[i].x);
      x = fmaxf(x, sl[i].z);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float d = 0.f;
    for (int i = lane; i < nslot; i += 32) {
      const float4 t = sl[i];
      if (t.x != -INFINITY) d += t.y * ex2((t.x - m) * kLog2e);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
    if constexpr (MODE == 2) {
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
    }
    return MaxSumLab{m, d, x};
  };

  // step 2 for row j (statistics t): outputs, loss, and the stage released
  auto finish = [&](int64_t j, int32_t label, const MaxSumLab& t) {
    const int64_t r = row_of(j);
    const uint4* st = stage(j);
    char* ys = const_cast<char*>(rw.slice(p.y, r, E));
    const bool ignored = MODE == 2 && label == p.ignore;
    const bool in_range = MODE == 2 && label >= 0 && (int64_t)label < g.cols;
    const bool lead = gr.gt == 0 && rank == 0;
    if (MODE == 2 && !ignored && !in_range && lead && p.bad != nullptr) atomicAdd(p.bad, 1);
    const float M = t.m;
    if (ignored || M == -INFINITY) {
      // ignored label or fully masked row: zeros (loss 0)
      if (MODE == 2 && lead) p.loss[r] = 0.f;
      const float z[W] = {};
      for (int q = 0; q < rw.nq; ++q) lnx_store<DT, W>(ys, gr.gt + q * gr.G, q, rw, z);
    } else if constexpr (MODE == 1) {
      const float lnd = logf(t.d);
#pragma unroll 2
      for (int q = 0; q < rw.nq; ++q) {
        const int k = gr.gt + q * gr.G;
        float v[W];
        lnx_unpack<DT, W>(st[k], v);
#pragma unroll
        for (int e = 0; e < W; e += 2) {
          add2(v[e], v[e + 1], v[e], v[e + 1], -M, -M);
          add2(v[e], v[e + 1], v[e], v[e + 1], -lnd, -lnd);
        }
        lnx_store<DT, W>(ys, k, q, rw, v);
      }
    } else {
      const float mL = M * kLog2e;
      const float inv = ex2(-fmaf(M, kLog2e, -mL)) / t.d;
#pragma unroll 2
      for (int q = 0; q < rw.nq; ++q) {
        const int k = gr.gt + q * gr.G;
        float v[W];
        lnx_unpack<DT, W>(st[k], v);
#pragma unroll
        for (int e = 0; e < W; e += 2) {
          float t0, t1;
          fma2(t0, t1, v[e], v[e + 1], kLog2e, kLog2e, -mL, -mL);
          mul2(v[e], v[e + 1], ex2(t0), ex2(t1), inv, inv);
        }
        lnx_store<DT, W>(ys, k, q, rw, v);
      }
      if constexpr (MODE == 2) {
        if (lead) p.loss[r] = in_range ? (M - t.x) + logf(t.d) : __int_as_float(0x7fc00000);
        // the label's element again, minus one (after its chunk: same thread)
        int lk, le;
        locate(label, lk, le);
        if (lk >= 0) {
          const float xl = ld_smem_elem<DT>(reinterpret_cast<const char*>(st + lk) + le * E);
          st_elem<DT>(ys + (int64_t)lk * 16 + le * E, ex2(fmaf(xl, kLog2e, -mL)) * inv - 1.0f);
        }
      }
    }
  };

  int32_t lab_prev = 0, lab_cur = 0, lab_next = 0;  // labels of rows j - 1, j, j + 1
  if constexpr (MODE == 2) {
    if (rw.first < g.rows) lab_next = __ldg(p.labels + rw.first);
  }
  int64_t j = 0;
  for (;; ++j) {
    const int64_t r = row_of(j);
    if (r >= g.rows) break;
    if constexpr (MODE == 2) {
      lab_cur = lab_next;
      if (row_of(j + 1) < g.rows) lab_next = __ldg(p.labels + row_of(j + 1));
    }
    // row j + ahead into the stage that row j + ahead - NS left (finished by
    // this thread in an earlier iteration), then row j's chunks
    fetch(j + ahead);
    landed();
    // step 1: this thread's online (m, d) (and the label's logit)
    MaxSumLab t = MaxSumLab::identity();
    if (!(MODE == 2 && lab_cur == p.ignore)) {
      uint4* st = stage(j);
      smx_mask_stage<DT, W>(st, rw, gr.gt, gr.G);
      const MaxSum th = smx_thread_stats<DT>(st, gr.gt, gr.G, rw.nq);
      t.m = th.m;
      t.d = th.d;
      if constexpr (MODE == 2) {
        int lk, le;
        locate(lab_cur, lk, le);
        if (lk >= 0) t.x = ld_smem_elem<DT>(reinterpret_cast<const char*>(st + lk) + le * E);
      }
    }
    if (solo) {
      // one warp per row: the warp's merge is the row's statistics
      finish(j, lab_cur, smx_warp_merge<MODE == 2>(t));
    } else {
      // row j - 1's statistics (its partials were published one row ago),
      // then row j's partial, then row j - 1's outputs
      MaxSumLab prev{};
      if (j >= 1) prev = merged(j - 1);
      publish(j, t);
      if (j >= 1) finish(j - 1, lab_prev, prev);
    }
    lab_prev = lab_cur;
  }
  if (!solo && j >= 1) finish(j - 1, lab_prev, merged(j - 1));
  cp_async_wait<0>();
  if constexpr (CL) cluster_sync();  // no peer still writes this block's slots
}

template <int DT, int CPT>
SmxKernels make_smx_set() {
  SmxKernels s{};
  s.k[0][0] = (const void*)smx_kernel<DT, 0, false>;
  s.k[0][1] = (const void*)smx_kernel<DT, 0, true>;
  s.k[1][0] = (const void*)smx_kernel<DT, 1, false>;
  s.k[1][1] = (const void*)smx_kernel<DT, 1, true>;
  s.k[2][0] = (const void*)smx_kernel<DT, 2, false>;
  s.k[2][1] = (const void*)smx_kernel<DT, 2, true>;
  s.nq = CPT;
  return s;
}

}  // namespace rr
