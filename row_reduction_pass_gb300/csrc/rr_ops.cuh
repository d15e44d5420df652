// rr_ops.cuh -- the three operations as policies of the row engine.
//
//   OpSoftmaxXent  softmax forward, and (with labels) fused cross-entropy
//                  loss + dlogits = softmax - onehot in the same pass
//                  ("Engineering a CUDA Machine Learning Framework from Scratch",
//                  sec. 3.1 "Online FlashSoftmax" and sec. 2.1).
//                  With SoftmaxParams::log set it writes the log-softmax
//                  z = (x - m) - ln d instead.
//   OpSoftmaxBwd   softmax backward dx = y * (dy - sum y*dy) and log-softmax
//                  backward dx = dz - exp(z) * sum dz (the vector-Jacobian
//                  products of the Softmax layer of the "NexusGrad" README).
//   OpLnFwd        LayerNorm forward with its moments from one pass over
//                  global memory (same page, sec. 3.2): exact mean from a
//                  compensated sum, then M2 about it, in registers; row slices
//                  held by the CTAs of a cluster merged with the Chan / Welford
//                  pairwise update.
//   OpLnBwd        analytic LayerNorm backward (same page, sec. 2.2): dx per
//                  row, and per-column partial sums of dy*xhat and dy that a
//                  second, fixed-order pass reduces into dgamma / dbeta.
#pragma once

#include <math.h>

#include "rr_engine.cuh"

namespace rr {

// Kernel arguments (plain structs shared with the host launcher).
struct SoftmaxParams {
  const char* x;
  char* y;
  const int32_t* labels;  // null: plain softmax
  float* loss;
  int32_t* bad;
  int* err;
  int64_t cols;
  int32_t ignore;
  int32_t log;  // 1: write the log-softmax (x - m) - ln d instead of the softmax
};
struct SoftmaxBwdParams {
  const char* y;   // the forward output: softmax y, or log-softmax z when log
  const char* dy;  // upstream gradient
  char* dx;
  int* err;
  int64_t cols;
  int32_t log;
};
struct LnFwdParams {
  const char* x;
  const char* gamma;
  const char* beta;
  char* y;
  float* mean;
  float* rstd;
  int* err;
  int64_t cols;
  float eps;
  float inv_cols;  // 1 / cols (rounded)
};
struct LnBwdParams {
  const char* dy;
  const char* x;
  const float* mean;
  const float* rstd;
  const char* gamma;
  char* dx;
  float* ws;  // [partials][2][cols] float32 column partials
  int* err;
  int64_t cols;
  float inv_cols;  // 1 / cols (rounded)
};

// ---------------------------------------------------------- statistics ----

// Online-softmax state: running maximum m and sum d of exp(x - m).
struct MaxSum {
  static constexpr bool kNary = true;
  float m, d;
  // Merge of the states of L consecutive lanes (L a power of two <= 32).
  template <int L>
  __device__ __forceinline__ static MaxSum nary(MaxSum v) {
    float m = v.m;
#pragma unroll
    for (int off = L / 2; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float d = (v.m == -INFINITY) ? 0.f : v.d * ex2((v.m - m) * kLog2e);
#pragma unroll
    for (int off = L / 2; off >= 1; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
    return {m, d};
  }
  __device__ __forceinline__ static MaxSum identity() { return {-INFINITY, 0.f}; }
  __device__ __forceinline__ static MaxSum shfl_xor(const MaxSum& v, int off) {
    return {__shfl_xor_sync(0xffffffffu, v.m, off), __shfl_xor_sync(0xffffffffu, v.d, off)};
  }
  __device__ __forceinline__ static MaxSum load_remote(uint32_t a) {
    return {ld_cluster_f32(a), ld_cluster_f32(a + 4)};
  }
};
// Pairwise merge of two online states (Milakov & Gimelshein, 2018):
// m = max(ma, mb), d = da * 2^((ma - m) log2 e) + db * 2^((mb - m) log2 e);
// a side whose m is -inf carries d = 0 and adds nothing.
struct MergeMaxSum {
  __device__ __forceinline__ MaxSum operator()(const MaxSum& a, const MaxSum& b) const {
    const float m = fmaxf(a.m, b.m);
    if (m == -INFINITY) return {m, 0.f};
    return {m, a.d * ex2((a.m - m) * kLog2e) + b.d * ex2((b.m - m) * kLog2e)};
  }
};

// A double-float sum (sh + sl, unevaluated).
struct DFSum {
  static constexpr bool kNary = false;
  float sh, sl;
  __device__ __forceinline__ static DFSum identity() { return {0.f, 0.f}; }
  __device__ __forceinline__ static DFSum shfl_xor(const DFSum& v, int off) {
    return {__shfl_xor_sync(0xffffffffu, v.sh, off), __shfl_xor_sync(0xffffffffu, v.sl, off)};
  }
  __device__ __forceinline__ static DFSum load_remote(uint32_t a) {
    return {ld_cluster_f32(a), ld_cluster_f32(a + 4)};
  }
};

// One plain sum.
struct Sum1 {
  static constexpr bool kNary = false;
  float s;
  __device__ __forceinline__ static Sum1 identity() { return {0.f}; }
  __device__ __forceinline__ static Sum1 shfl_xor(const Sum1& v, int off) {
    return {__shfl_xor_sync(0xffffffffu, v.s, off)};
  }
  __device__ __forceinline__ static Sum1 load_remote(uint32_t a) { return {ld_cluster_f32(a)}; }
};
struct MergeSum1 {
  __device__ __forceinline__ Sum1 operator()(const Sum1& a, const Sum1& b) const {
    return {a.s + b.s};
  }
};

// Moments of a set of values, with the sum kept as an unevaluated pair of
// floats (sh + sl, "double-float") so the mean stays exact to ~2^-48 relative
// even when large values cancel: (count n, sum S = sh + sl, M2 = sum of squared
// deviations from the mean).
struct Moments {
  static constexpr bool kNary = false;
  float n, sh, sl, m2;
  __device__ __forceinline__ static Moments identity() { return {0.f, 0.f, 0.f, 0.f}; }
  __device__ __forceinline__ static Moments shfl_xor(const Moments& v, int off) {
    return {__shfl_xor_sync(0xffffffffu, v.n, off), __shfl_xor_sync(0xffffffffu, v.sh, off),
            __shfl_xor_sync(0xffffffffu, v.sl, off), __shfl_xor_sync(0xffffffffu, v.m2, off)};
  }
  __device__ __forceinline__ static Moments load_remote(uint32_t a) {
    return {ld_cluster_f32(a), ld_cluster_f32(a + 4), ld_cluster_f32(a + 8),
            ld_cluster_f32(a + 12)};
  }
};

// Error-free sum of two floats (Knuth's TwoSum): a + b = s + e exactly.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}

// Double-float addition (exact error of the leading sum kept; commutative
// bit for bit, so butterflies leave every lane with the same value).
struct MergeDF {
  __device__ __forceinline__ DFSum operator()(const DFSum& a, const DFSum& b) const {
    float s, e;
    two_sum(a.sh, b.sh, s, e);
    e += a.sl + b.sl;
    float h, l;
    two_sum(s, e, h, l);
    return {h, l};
  }
};

// Mean S / n of a double-float sum as a double-float (mh + ml), given inv = 1/n
// rounded: mh = fl(S_h * inv), the remainder S_h - mh*n is exact in one FMA, and
// ml = (remainder + S_l) * inv.
__device__ __forceinline__ void df_mean(float sh, float sl, float n, float inv, float& mh,
                                        float& ml) {
  mh = sh * inv;
  const float r = fmaf(-mh, n, sh);
  ml = (r + sl) * inv;
}
__device__ __forceinline__ void df_div(float sh, float sl, float n, float& mh, float& ml) {
  df_mean(sh, sl, n, __frcp_rn(n), mh, ml);
}

// Chan, Golub & LeVeque pairwise update (the parallel form of Welford's
// one-pass recurrence) written on sums: with delta = Sb/nb - Sa/na,
//   n = na + nb,  S = Sa + Sb,  M2 = M2a + M2b + delta^2 na nb / n
//                                   = M2a + M2b + (Sb na - Sa nb)^2 / (na nb n).
// `a` is always the lower-ranked side, so every thread merges identically.
struct MergeMoments {
  __device__ __forceinline__ Moments operator()(const Moments& a, const Moments& b) const {
    if (a.n == 0.f) return b;
    if (b.n == 0.f) return a;
    const float n = a.n + b.n;
    float s, e;
    two_sum(a.sh, b.sh, s, e);
    e += a.sl + b.sl;
    float sh, sl;
    two_sum(s, e, sh, sl);
    // D = Sb * na - Sa * nb with exact products (rounded multiplies, never fused)
    const float p1 = __fmul_rn(b.sh, a.n), e1 = fmaf(b.sh, a.n, -p1);
    const float p2 = __fmul_rn(a.sh, b.n), e2 = fmaf(a.sh, b.n, -p2);
    float dh, de;
    two_sum(p1, -p2, dh, de);
    const float D = dh + (de + (e1 - e2) + (__fmul_rn(b.sl, a.n) - __fmul_rn(a.sl, b.n)));
    const float m2 = a.m2 + b.m2 + (D * D) / (a.n * b.n * n);
    return {n, sh, sl, m2};
  }
};

// Two plain sums.
struct Sum2 {
  static constexpr bool kNary = false;
  float s1, s2;
  __device__ __forceinline__ static Sum2 identity() { return {0.f, 0.f}; }
  __device__ __forceinline__ static Sum2 shfl_xor(const Sum2& v, int off) {
    return {__shfl_xor_sync(0xffffffffu, v.s1, off), __shfl_xor_sync(0xffffffffu, v.s2, off)};
  }
  __device__ __forceinline__ static Sum2 load_remote(uint32_t a) {
    return {ld_cluster_f32(a), ld_cluster_f32(a + 4)};
  }
};
struct MergeSum2 {
  __device__ __forceinline__ Sum2 operator()(const Sum2& a, const Sum2& b) const {
    return {a.s1 + b.s1, a.s2 + b.s2};
  }
};

// ------------------------------------------------- softmax / cross-entropy --

template <int DT_, int W_, int NQ_>
struct OpSoftmaxXent {
  static constexpr int DT = DT_, W = W_, NT = 1, NQ = NQ_;
  static constexpr int E = DType<DT>::E;
  static constexpr bool kPrefetch = true;
  using Params = SoftmaxParams;
  struct Meta {
    int32_t label;
    bool skip;
  };
  struct Thread {};

  __device__ __forceinline__ static Meta meta(const Params& p, int64_t r) {
    if (r < 0 || p.labels == nullptr) return {-1, false};
    const int32_t l = __ldg(p.labels + r);
    return {l, l == p.ignore};
  }
  __device__ __forceinline__ static bool skip(const Meta& m) { return m.skip; }
  __device__ __forceinline__ static float fill() { return -INFINITY; }
  __device__ __forceinline__ static const char* in_slice_start(const Params& p, int, int64_t r,
                                                               int64_t c0) {
    return p.x + (r * p.cols + c0) * E;
  }
  __device__ __forceinline__ static uint64_t start_addr(const Params& p, int64_t r, int64_t c0) {
    return reinterpret_cast<uint64_t>(in_slice_start(p, 0, r, c0));
  }
  __device__ __forceinline__ static const char* in_chunk0(const Params& p, int t, int64_t r,
                                                          int64_t c0, const RowGeo<DT, W>& g) {
    return in_slice_start(p, t, r, c0) - g.head_bytes;
  }
  __device__ __forceinline__ static void thread_init(Thread&, const Params&, const Geo&, int64_t,
                                                     int64_t, int, int, unsigned char*, int, int) {}
  __device__ __forceinline__ static void load_direct(RowRegs<DT, W, NT, NQ>& x,
                                                     const RowGeo<DT, W>& g, const Params& p,
                                                     const Geo&, int64_t r, int64_t c0) {
    load_direct_mem(x, 0, g, in_chunk0(p, 0, r, c0, g), fill());
  }
  __device__ __forceinline__ static void load_staged(RowRegs<DT, W, NT, NQ>& x,
                                                     const RowGeo<DT, W>& g, const Params& p,
                                                     const Geo&, int64_t r, int64_t c0,
                                                     const unsigned char* sbuf, int) {
    load_staged_mem(x, 0, g, in_chunk0(p, 0, r, c0, g), sbuf, fill());
  }

  // Row maximum of the thread's slots.  Ragged slots hold -inf, so every slot
  // of every owned chunk can take part (bf16: packed max, two values at once).
  __device__ __forceinline__ static float thread_max(const RowRegs<DT, W, NT, NQ>& x,
                                                     const RowGeo<DT, W>& g) {
    if constexpr (W > 1 && DT == kBF16) {
      uint32_t mw = 0xff80ff80u;
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        if (!g.has(q)) break;
        const uint4 c = x.v[0][q];
        mw = bf16x2_max(mw, bf16x2_max(bf16x2_max(c.x, c.y), bf16x2_max(c.z, c.w)));
      }
      return fmaxf(__uint_as_float(mw << 16), __uint_as_float(mw & 0xffff0000u));
    } else {
      float m = -INFINITY;
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        if (!g.has(q)) break;
#pragma unroll
        for (int e = 0; e < W; ++e) m = fmaxf(m, x.get(0, q, e));
      }
      return m;
    }
  }

  // Online-softmax state of the thread: m = its maximum, d = sum of exp(x - m).
  // The exponent is one FMA, x*log2(e) - fl(m*log2(e)); the rounding residual
  // r of fl(m*log2(e)) shifts every term by the same factor 2^r, which is
  // divided out once (so d is the plain sum of exp(x - m)).
  __device__ __forceinline__ static MaxSum thread_stats(const RowRegs<DT, W, NT, NQ>& x,
                                                        const RowGeo<DT, W>& g) {
    const float m = thread_max(x, g);
    if (m == -INFINITY) return {m, 0.f};
    const float mL = m * kLog2e;
    const float r = fmaf(m, kLog2e, -mL);
    float d0 = 0.f, d1 = 0.f;
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      if (!g.has(q)) break;
#pragma unroll
      for (int e = 0; e < W; e += 2) {
        if constexpr (W > 1) {
          float t0, t1;
          fma2(t0, t1, x.get(0, q, e), x.get(0, q, e + 1), kLog2e, kLog2e, -mL, -mL);
          add2(d0, d1, d0, d1, ex2(t0), ex2(t1));
        } else {
          d0 += ex2(fmaf(x.get(0, q, e), kLog2e, -mL));
        }
      }
    }
    return {m, (d0 + d1) * ex2(-r)};
  }

  template <class R>
  __device__ __forceinline__ static void process(Thread&, const Params& p, const Geo& geo,
                                                 int64_t r, const Meta& mt,
                                                 const RowRegs<DT, W, NT, NQ>& x,
                                                 const RowGeo<DT, W>& g, bool leader, bool active,
                                                 R& rd) {
    const bool use = active && !mt.skip;
    MaxSum s = use ? thread_stats(x, g) : MaxSum::identity();
    s = rd.reduce(s, MergeMaxSum());
    s = rd.cluster(s, MergeMaxSum());
    if (!active) return;
    char* y0 = p.y + (r * p.cols + g.c0) * E - g.head_bytes;
    const bool masked = (s.m == -INFINITY);
    int ql = -1, el = 0;  // where this thread holds the label column, if it does
    float xl = 0.f;       // and the logit there
    if (p.labels != nullptr) {
      const int32_t label = mt.label;
      const bool in_range = label >= 0 && (int64_t)label < geo.cols;
      // an out-of-range label is counted whatever the row holds
      if (!mt.skip && !in_range && leader && p.bad != nullptr) atomicAdd(p.bad, 1);
      if (in_range && !mt.skip) g.locate(label, ql, el);
      if (mt.skip || masked) {
        if (leader) p.loss[r] = 0.f;
      } else if (!in_range) {
        if (leader) p.loss[r] = __int_as_float(0x7fc00000);
      } else if (ql >= 0) {
#pragma unroll
        for (int q = 0; q < NQ; ++q)
#pragma unroll
          for (int e = 0; e < W; ++e)
            if (q == ql && e == el) xl = x.get(0, q, e);
        p.loss[r] = (s.m - xl) + logf(s.d);
      }
    }
    if (mt.skip || masked) {
      const float z[W] = {};
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        if (!g.has(q)) break;
        g.store_chunk(y0, q, z);
      }
      return;
    }
    // Rows without a ragged head or tail (every chunk full) take loops with
    // no per-chunk checks; the label's element is then rewritten after its
    // chunk (same thread, same address: the later store wins).
    if (p.log) {
      // z_j = (x_j - m) - ln d: x - m first, so z keeps its relative accuracy
      const float lnd = logf(s.d);
      auto logs = [&](int q, float* f) {
        if constexpr (W > 1) {
#pragma unroll
          for (int e = 0; e < W; e += 2) {
            add2(f[e], f[e + 1], x.get(0, q, e), x.get(0, q, e + 1), -s.m, -s.m);
            add2(f[e], f[e + 1], f[e], f[e + 1], -lnd, -lnd);
          }
        } else {
          f[0] = (x.get(0, q, 0) - s.m) - lnd;
        }
      };
      if constexpr (W > 1) {
        if (g.all_full()) {
#pragma unroll
          for (int q = 0; q < NQ; ++q) {
            if (!g.has(q)) break;
            float f[W];
            logs(q, f);
            st_chunk_stream(y0 + g.off(q), chunk_pack<DT>(f));
          }
          return;
        }
      }
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        if (!g.has(q)) break;
        float f[W];
        logs(q, f);
        g.store_chunk(y0, q, f);
      }
      return;
    }
    // p_j = 2^(x_j log2 e - fl(m log2 e)) * 2^(-r) / d
    const float mL = s.m * kLog2e;
    const float rr = fmaf(s.m, kLog2e, -mL);
    const float inv = ex2(-rr) / s.d;
    auto probs = [&](int q, float* f) {
      if constexpr (W > 1) {
#pragma unroll
        for (int e = 0; e < W; e += 2) {
          float t0, t1;
          fma2(t0, t1, x.get(0, q, e), x.get(0, q, e + 1), kLog2e, kLog2e, -mL, -mL);
          mul2(f[e], f[e + 1], ex2(t0), ex2(t1), inv, inv);
        }
      } else {
        f[0] = ex2(fmaf(x.get(0, q, 0), kLog2e, -mL)) * inv;
      }
    };
    if constexpr (W > 1) {
      if (g.all_full()) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          if (!g.has(q)) break;
          float f[W];
          probs(q, f);
          st_chunk_stream(y0 + g.off(q), chunk_pack<DT>(f));
        }
        if (ql >= 0)
          st_elem<DT>(y0 + g.off(ql) + el * E, ex2(fmaf(xl, kLog2e, -mL)) * inv - 1.0f);
        return;
      }
    }
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      if (!g.has(q)) break;
      float f[W];
      probs(q, f);
      if (q == ql) {
#pragma unroll
        for (int e = 0; e < W; ++e)
          if (e == el) f[e] -= 1.0f;
      }
      g.store_chunk(y0, q, f);
    }
  }
  __device__ __forceinline__ static void epilogue(Thread&, const Params&, const Geo&,
                                                  unsigned char*, int64_t, int64_t, int64_t, int,
                                                  int, int, int) {}
};

// ------------------------------------------- softmax / log-softmax backward --
//
// Two row tensors read in the same memory-aligned chunks (the caller gives y,
// dy and dx the same 16-byte alignment, else element mode): one sum per row,
// S = sum y*dy (softmax) or sum dz (log-softmax), then
//   dx = y * (dy - S)            or   dx = dz - exp(z) * S.
// Ragged slots hold 0 in both tensors and add nothing to S.

template <int DT_, int W_, int NQ_>
struct OpSoftmaxBwd {
  static constexpr int DT = DT_, W = W_, NT = 2, NQ = NQ_;
  static constexpr int E = DType<DT>::E;
  static constexpr bool kPrefetch = true;
  using Params = SoftmaxBwdParams;
  struct Meta {};
  struct Thread {};

  __device__ __forceinline__ static Meta meta(const Params&, int64_t) { return {}; }
  __device__ __forceinline__ static bool skip(const Meta&) { return false; }
  __device__ __forceinline__ static const char* in_slice_start(const Params& p, int t, int64_t r,
                                                               int64_t c0) {
    return (t == 0 ? p.y : p.dy) + (r * p.cols + c0) * E;
  }
  __device__ __forceinline__ static uint64_t start_addr(const Params& p, int64_t r, int64_t c0) {
    return reinterpret_cast<uint64_t>(in_slice_start(p, 0, r, c0));
  }
  __device__ __forceinline__ static const char* in_chunk0(const Params& p, int t, int64_t r,
                                                          int64_t c0, const RowGeo<DT, W>& g) {
    return in_slice_start(p, t, r, c0) - g.head_bytes;
  }
  __device__ __forceinline__ static void thread_init(Thread&, const Params&, const Geo&, int64_t,
                                                     int64_t, int, int, unsigned char*, int, int) {}
  __device__ __forceinline__ static void load_direct(RowRegs<DT, W, NT, NQ>& v,
                                                     const RowGeo<DT, W>& g, const Params& p,
                                                     const Geo&, int64_t r, int64_t c0) {
    load_direct_mem(v, 0, g, in_chunk0(p, 0, r, c0, g), 0.f);
    load_direct_mem(v, 1, g, in_chunk0(p, 1, r, c0, g), 0.f);
  }
  __device__ __forceinline__ static void load_staged(RowRegs<DT, W, NT, NQ>& v,
                                                     const RowGeo<DT, W>& g, const Params& p,
                                                     const Geo&, int64_t r, int64_t c0,
                                                     const unsigned char* sbuf, int buf_bytes) {
    load_staged_mem(v, 0, g, in_chunk0(p, 0, r, c0, g), sbuf, 0.f);
    load_staged_mem(v, 1, g, in_chunk0(p, 1, r, c0, g), sbuf + buf_bytes, 0.f);
  }

  template <class R>
  __device__ __forceinline__ static void process(Thread&, const Params& p, const Geo&, int64_t r,
                                                 const Meta&, const RowRegs<DT, W, NT, NQ>& v,
                                                 const RowGeo<DT, W>& g, bool, bool active,
                                                 R& rd) {
    float s0 = 0.f, s1 = 0.f;
    if (active) {
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        if (!g.has(q)) break;
        if constexpr (W > 1) {
#pragma unroll
          for (int e = 0; e < W; e += 2) {
            if (p.log)
              add2(s0, s1, s0, s1, v.get(1, q, e), v.get(1, q, e + 1));
            else
              fma2(s0, s1, v.get(0, q, e), v.get(0, q, e + 1), v.get(1, q, e), v.get(1, q, e + 1),
                   s0, s1);
          }
        } else {
          s0 = p.log ? s0 + v.get(1, q, 0) : fmaf(v.get(0, q, 0), v.get(1, q, 0), s0);
        }
      }
    }
    Sum1 S{s0 + s1};
    S = rd.reduce(S, MergeSum1());
    S = rd.cluster(S, MergeSum1());
    if (!active) return;
    char* dx0 = p.dx + (r * p.cols + g.c0) * E - g.head_bytes;
    auto grads = [&](int q, float* f) {
      if constexpr (W > 1) {
#pragma unroll
        for (int e = 0; e < W; e += 2) {
          if (p.log) {
            const float p0 = ex2(v.get(0, q, e) * kLog2e), p1 = ex2(v.get(0, q, e + 1) * kLog2e);
            fma2(f[e], f[e + 1], p0, p1, -S.s, -S.s, v.get(1, q, e), v.get(1, q, e + 1));
          } else {
            float t0, t1;
            add2(t0, t1, v.get(1, q, e), v.get(1, q, e + 1), -S.s, -S.s);
            mul2(f[e], f[e + 1], v.get(0, q, e), v.get(0, q, e + 1), t0, t1);
          }
        }
      } else {
        f[0] = p.log ? fmaf(ex2(v.get(0, q, 0) * kLog2e), -S.s, v.get(1, q, 0))
                     : v.get(0, q, 0) * (v.get(1, q, 0) - S.s);
      }
    };
    // rows without a ragged head or tail: no per-chunk checks on the stores
    // (variants of several chunks per thread; in the two-chunk ones the second
    // copy of the loop costs registers)
    if constexpr (W > 1 && NQ > 2) {
      if (g.all_full()) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          if (!g.has(q)) break;
          float f[W];
          grads(q, f);
          st_chunk_stream(dx0 + g.off(q), chunk_pack<DT>(f));
        }
        return;
      }
    }
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      if (!g.has(q)) break;
      float f[W];
      grads(q, f);
      g.store_chunk(dx0, q, f);
    }
  }
  __device__ __forceinline__ static void epilogue(Thread&, const Params&, const Geo&,
                                                  unsigned char*, int64_t, int64_t, int64_t, int,
                                                  int, int, int) {}
};

// ------------------------------------------------------- LayerNorm forward --
//
// Both LayerNorm operations work on column-aligned chunks (chunk k of a thread is
// columns c0 + kW ...), whatever the alignment of the row in memory, so gamma,
// beta and the column partials are plain 16-byte vectors.
//
// Moments: one pass over global memory.  In registers, a compensated sum gives
// the exact mean (double-float), then the squared deviations from it give M2;
// each is reduced over the row group.  A row split over a cluster merges its
// CTAs' (n, S, M2) with the Chan/Welford pairwise update.

template <int DT_, int W_, int NQ_>
struct OpLnFwd {
  static constexpr int DT = DT_, W = W_, NT = 1, NQ = NQ_;
  static constexpr int E = DType<DT>::E;
  static constexpr bool kPrefetch = false;
  using Params = LnFwdParams;
  struct Meta {};
  struct Thread {};

  __device__ __forceinline__ static Meta meta(const Params&, int64_t) { return {}; }
  __device__ __forceinline__ static bool skip(const Meta&) { return false; }
  __device__ __forceinline__ static const char* in_slice_start(const Params& p, int, int64_t r,
                                                               int64_t c0) {
    return p.x + (r * p.cols + c0) * E;
  }
  // column space: the row geometry never has a ragged head
  __device__ __forceinline__ static uint64_t start_addr(const Params&, int64_t, int64_t) {
    return 0;
  }
  __device__ __forceinline__ static void thread_init(Thread&, const Params&, const Geo&, int64_t,
                                                     int64_t, int, int, unsigned char*, int, int) {}
  __device__ __forceinline__ static void load_direct(RowRegs<DT, W, NT, NQ>& x,
                                                     const RowGeo<DT, W>& g, const Params& p,
                                                     const Geo& geo, int64_t r, int64_t c0) {
    load_cols(x, 0, g, in_slice_start(p, 0, r, c0), p.x, p.x + geo.rows * geo.cols * E, nullptr);
  }
  __device__ __forceinline__ static void load_staged(RowRegs<DT, W, NT, NQ>& x,
                                                     const RowGeo<DT, W>& g, const Params& p,
                                                     const Geo& geo, int64_t r, int64_t c0,
                                                     const unsigned char* sbuf, int) {
    load_cols(x, 0, g, in_slice_start(p, 0, r, c0), p.x, p.x + geo.rows * geo.cols * E, sbuf);
  }

  template <class R>
  __device__ __forceinline__ static void process(Thread&, const Params& p, const Geo& geo,
                                                 int64_t r, const Meta&,
                                                 const RowRegs<DT, W, NT, NQ>& x,
                                                 const RowGeo<DT, W>& g, bool leader, bool active,
                                                 R& rd) {
    // 1. compensated sum of the thread's values (two interleaved TwoSum
    //    accumulators per packed pair; ragged slots hold 0) -> group sum -> mean
    float s = 0.f, c = 0.f;
    if (active) {
      if constexpr (W > 1) {
        float s0 = 0.f, s1 = 0.f, c0 = 0.f, c1 = 0.f;
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          if (!g.has(q)) break;
#pragma unroll
          for (int e = 0; e < W; e += 2) {
            const float v0 = x.get(0, q, e), v1 = x.get(0, q, e + 1);
            float t0, t1, b0, b1, u0, u1, w0, w1;
            add2(t0, t1, s0, s1, v0, v1);            // t = s + v
            add2(b0, b1, t0, t1, -s0, -s1);          // bb = t - s
            add2(u0, u1, t0, t1, -b0, -b1);          // t - bb
            add2(u0, u1, s0, s1, -u0, -u1);          // s - (t - bb)
            add2(w0, w1, v0, v1, -b0, -b1);          // v - bb
            add2(u0, u1, u0, u1, w0, w1);            // exact error of s + v
            add2(c0, c1, c0, c1, u0, u1);
            s0 = t0;
            s1 = t1;
          }
        }
        float e;
        two_sum(s0, s1, s, e);
        c = (c0 + c1) + e;
      } else {
        g.template for_each<NQ>([&](int q, int e) {
          const float v = x.get(0, q, e);
          float t, err;
          two_sum(s, v, t, err);
          c += err;
          s = t;
        });
      }
    }
    DFSum S;
    two_sum(s, c, S.sh, S.sl);
    S = rd.reduce(S, MergeDF());
    const float ns = static_cast<float>(g.c1 - g.c0);
    const bool whole = (rd.K == 1);
    const float inv_n = whole ? p.inv_cols : __frcp_rn(ns);
    float mh, ml;
    df_mean(S.sh, S.sl, ns, inv_n, mh, ml);
    // 2. squared deviations from that mean -> group sum (ragged slots excluded)
    float m2 = 0.f;
    if (active) {
      if constexpr (W > 1) {
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          if (!g.has(q)) break;
          const bool fullq = g.full(q);
#pragma unroll
          for (int e = 0; e < W; e += 2) {
            float d0, d1;
            add2(d0, d1, x.get(0, q, e), x.get(0, q, e + 1), -mh, -mh);
            add2(d0, d1, d0, d1, -ml, -ml);
            if (!fullq) {
              if (!g.valid(q, e)) d0 = 0.f;
              if (!g.valid(q, e + 1)) d1 = 0.f;
            }
            fma2(a0, a1, d0, d1, d0, d1, a0, a1);
          }
        }
        m2 = a0 + a1;
      } else {
        g.template for_each<NQ>([&](int q, int e) {
          const float d = (x.get(0, q, e) - mh) - ml;
          m2 = fmaf(d, d, m2);
        });
      }
    }
    m2 = rd.reduce(Sum1{m2}, MergeSum1()).s;
    if (!whole) {
      // 3. slices of a cluster: Chan/Welford pairwise merge of (n, S, M2)
      Moments mo = rd.cluster(Moments{ns, S.sh, S.sl, m2}, MergeMoments());
      df_mean(mo.sh, mo.sl, mo.n, p.inv_cols, mh, ml);
      m2 = mo.m2;
    }
    if (!active) return;
    const float var = m2 * p.inv_cols;
    const bool masked = !(isfinite(mh) && isfinite(ml) && isfinite(var));
    const float rstd = masked ? 0.f : rsqrtf(var + p.eps);
    if (leader) {
      p.mean[r] = masked ? 0.f : mh + ml;
      p.rstd[r] = rstd;
    }
    char* y0 = p.y + (r * p.cols + g.c0) * E;
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      if (!g.has(q)) break;
      float f[W];
      if (masked) {
#pragma unroll
        for (int e = 0; e < W; ++e) f[e] = 0.f;
      } else {
        const int64_t j = g.c0 + (int64_t)g.chunk(q) * W;
        if constexpr (W > 1) {
          uint4 gv, bv;
          if (g.full(q)) {
            gv = ld_chunk_cached(p.gamma + j * E);
            bv = ld_chunk_cached(p.beta + j * E);
          } else {
            gv = make_uint4(0, 0, 0, 0);
            bv = gv;
#pragma unroll
            for (int e = 0; e < W; ++e)
              if (g.valid(q, e)) {
                chunk_set_bits<DT>(gv, e, ld_elem_bits<DT>(p.gamma + (j + e) * E));
                chunk_set_bits<DT>(bv, e, ld_elem_bits<DT>(p.beta + (j + e) * E));
              }
          }
#pragma unroll
          for (int e = 0; e < W; e += 2) {
            float t0, t1;
            add2(t0, t1, x.get(0, q, e), x.get(0, q, e + 1), -mh, -mh);
            add2(t0, t1, t0, t1, -ml, -ml);
            mul2(t0, t1, t0, t1, rstd, rstd);
            fma2(f[e], f[e + 1], t0, t1, chunk_get<DT>(gv, e), chunk_get<DT>(gv, e + 1),
                 chunk_get<DT>(bv, e), chunk_get<DT>(bv, e + 1));
          }
        } else {
          const float xh = ((x.get(0, q, 0) - mh) - ml) * rstd;
          f[0] = fmaf(xh, ld_elem_cached<DT>(p.gamma + j * E), ld_elem_cached<DT>(p.beta + j * E));
        }
      }
      store_cols(g, y0, q, f);
    }
  }
  __device__ __forceinline__ static void epilogue(Thread&, const Params&, const Geo&,
                                                  unsigned char*, int64_t, int64_t, int64_t, int,
                                                  int, int, int) {}
};

// ------------------------------------------------------ LayerNorm backward --

template <int DT_, int W_, int NQ_>
struct OpLnBwd {
  static constexpr int DT = DT_, W = W_, NT = 2, NQ = NQ_;  // tensor 0: dy, 1: x
  static constexpr int E = DType<DT>::E;
  static constexpr bool kPrefetch = false;
  using Params = LnBwdParams;
  struct Meta {
    float mean, rstd;
  };
  // part: this group's column partials in shared memory, part[j] = sum of
  // dy*xhat and part[npad + j] = sum of dy over the rows the group processed
  // (j local to the slice).
  struct Thread {
    float* part;
    const char* gamma;  // gamma at the slice start
    int npad;
  };

  __device__ __forceinline__ static Meta meta(const Params& p, int64_t r) {
    if (r < 0) return {0.f, 0.f};
    return {__ldg(p.mean + r), __ldg(p.rstd + r)};
  }
  // A row the forward masked (rstd == 0) is neither read nor accumulated.
  __device__ __forceinline__ static bool skip(const Meta& m) { return m.rstd == 0.f; }
  __device__ __forceinline__ static const char* in_slice_start(const Params& p, int t, int64_t r,
                                                               int64_t c0) {
    return (t == 0 ? p.dy : p.x) + (r * p.cols + c0) * E;
  }
  __device__ __forceinline__ static uint64_t start_addr(const Params&, int64_t, int64_t) {
    return 0;
  }
  __device__ __forceinline__ static void thread_init(Thread& ts, const Params& p, const Geo&,
                                                     int64_t c0, int64_t c1, int gt, int G,
                                                     unsigned char* colbuf, int grp, int) {
    ts.npad = static_cast<int>(((c1 - c0) + W - 1) / W * W);
    ts.part = reinterpret_cast<float*>(colbuf) + (size_t)grp * 2 * ts.npad;
    ts.gamma = p.gamma + c0 * E;
    for (int i = gt; i < 2 * ts.npad; i += G) ts.part[i] = 0.f;
  }
  __device__ __forceinline__ static void load_direct(RowRegs<DT, W, NT, NQ>& v,
                                                     const RowGeo<DT, W>& g, const Params& p,
                                                     const Geo& geo, int64_t r, int64_t c0) {
    const int64_t n = geo.rows * geo.cols * E;
    load_cols(v, 0, g, in_slice_start(p, 0, r, c0), p.dy, p.dy + n, nullptr);
    load_cols(v, 1, g, in_slice_start(p, 1, r, c0), p.x, p.x + n, nullptr);
  }
  __device__ __forceinline__ static void load_staged(RowRegs<DT, W, NT, NQ>& v,
                                                     const RowGeo<DT, W>& g, const Params& p,
                                                     const Geo& geo, int64_t r, int64_t c0,
                                                     const unsigned char* sbuf, int buf_bytes) {
    const int64_t n = geo.rows * geo.cols * E;
    load_cols(v, 0, g, in_slice_start(p, 0, r, c0), p.dy, p.dy + n, sbuf);
    load_cols(v, 1, g, in_slice_start(p, 1, r, c0), p.x, p.x + n, sbuf + buf_bytes);
  }

  // gamma of chunk q as storage bits (zero past the row end); element mode: the value
  __device__ __forceinline__ static uint4 gamma_raw(const Thread& ts, const RowGeo<DT, W>& g,
                                                    int q) {
    const int64_t j = (int64_t)g.chunk(q) * W;
    if constexpr (W > 1) {
      if (g.full(q)) return ld_chunk_cached(ts.gamma + j * E);
      uint4 c = make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int e = 0; e < W; ++e)
        if (g.valid(q, e)) chunk_set_bits<DT>(c, e, ld_elem_bits<DT>(ts.gamma + (j + e) * E));
      return c;
    } else {
      return make_uint4(__float_as_uint(ld_elem_cached<DT>(ts.gamma + j * E)), 0, 0, 0);
    }
  }
  __device__ __forceinline__ static float gam(const uint4& c, int e) {
    if constexpr (W > 1) return chunk_get<DT>(c, e);
    else return __uint_as_float(c.x);
  }

  template <class R>
  __device__ __forceinline__ static void process(Thread& ts, const Params& p, const Geo& geo,
                                                 int64_t r, const Meta& m,
                                                 const RowRegs<DT, W, NT, NQ>& v,
                                                 const RowGeo<DT, W>& g, bool, bool active,
                                                 R& rd) {
    const bool use = active && !skip(m);
    // S1 = sum g, S2 = sum g * xhat with g = dy * gamma, xhat = (x - mean) * rstd
    // (ragged slots hold dy = 0, x = 0 and gamma = 0, so they add nothing)
    float s1 = 0.f, s2 = 0.f;
    if (use) {
      float sa = 0.f, sb = 0.f, qa = 0.f, qb = 0.f;
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        if (!g.has(q)) break;
        const uint4 gr = gamma_raw(ts, g, q);
        if constexpr (W > 1) {
#pragma unroll
          for (int e = 0; e < W; e += 2) {
            float h0, h1;
            // g is a rounded scalar product: the packed multiply may be fused
            // with the add that follows it, and the output pass must recompute
            // exactly the g whose sum is S1 (so that g - mean(g) = 0 when C = 1)
            const float g0 = __fmul_rn(v.get(0, q, e), gam(gr, e));
            const float g1 = __fmul_rn(v.get(0, q, e + 1), gam(gr, e + 1));
            add2(h0, h1, v.get(1, q, e), v.get(1, q, e + 1), -m.mean, -m.mean);
            mul2(h0, h1, h0, h1, m.rstd, m.rstd);
            add2(sa, sb, sa, sb, g0, g1);
            fma2(qa, qb, g0, g1, h0, h1, qa, qb);
          }
        } else {
          const float gg = __fmul_rn(v.get(0, q, 0), gam(gr, 0));
          const float xh = (v.get(1, q, 0) - m.mean) * m.rstd;
          sa += gg;
          qa = fmaf(gg, xh, qa);
        }
      }
      s1 = sa + sb;
      s2 = qa + qb;
    }
    Sum2 s = rd.reduce(Sum2{s1, s2}, MergeSum2());
    s = rd.cluster(s, MergeSum2());
    if (!active) return;
    char* dx0 = p.dx + (r * p.cols + g.c0) * E;
    if (!use) {
      const float z[W] = {};
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        if (!g.has(q)) break;
        store_cols(g, dx0, q, z);
      }
      return;
    }
    const float a = s.s1 * p.inv_cols;
    const float b = s.s2 * p.inv_cols;
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      if (!g.has(q)) break;
      const uint4 gr = gamma_raw(ts, g, q);
      float* pp = ts.part + g.chunk(q) * W;
      if constexpr (W > 1) {
        uint4 out = make_uint4(0, 0, 0, 0);
        // four columns at a time: dx, and the column partials dy*xhat and dy
        // added into shared memory (ragged slots add dy = 0)
#pragma unroll
        for (int e0 = 0; e0 < W; e0 += 4) {
          float f[4], pg[4];
#pragma unroll
          for (int e = e0; e < e0 + 4; e += 2) {
            const float y0 = v.get(0, q, e), y1 = v.get(0, q, e + 1);
            float h0, h1, t0, t1;
            const float g0 = __fmul_rn(y0, gam(gr, e)), g1 = __fmul_rn(y1, gam(gr, e + 1));
            add2(h0, h1, v.get(1, q, e), v.get(1, q, e + 1), -m.mean, -m.mean);
            mul2(h0, h1, h0, h1, m.rstd, m.rstd);  // xhat
            add2(t0, t1, g0, g1, -a, -a);          // g - a
            fma2(t0, t1, h0, h1, -b, -b, t0, t1);  // (g - a) - xhat b
            mul2(f[e - e0], f[e - e0 + 1], t0, t1, m.rstd, m.rstd);
            mul2(pg[e - e0], pg[e - e0 + 1], y0, y1, h0, h1);
          }
          float4 u = *reinterpret_cast<float4*>(pp + e0);
          float4 w = *reinterpret_cast<float4*>(pp + ts.npad + e0);
          add2(u.x, u.y, u.x, u.y, pg[0], pg[1]);
          add2(u.z, u.w, u.z, u.w, pg[2], pg[3]);
          add2(w.x, w.y, w.x, w.y, v.get(0, q, e0), v.get(0, q, e0 + 1));
          add2(w.z, w.w, w.z, w.w, v.get(0, q, e0 + 2), v.get(0, q, e0 + 3));
          *reinterpret_cast<float4*>(pp + e0) = u;
          *reinterpret_cast<float4*>(pp + ts.npad + e0) = w;
          if constexpr (DT == kBF16) {
            const uint32_t lo = pack_bf16x2(f[0], f[1]), hi = pack_bf16x2(f[2], f[3]);
            set_word(out, e0 / 2, lo);
            set_word(out, e0 / 2 + 1, hi);
          } else {
            out = make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                             __float_as_uint(f[3]));
          }
        }
        store_cols_bits(g, dx0, q, out);
      } else {
        const float dyv = v.get(0, q, 0);
        const float gg = __fmul_rn(dyv, gam(gr, 0));
        const float xh = (v.get(1, q, 0) - m.mean) * m.rstd;
        const float f = m.rstd * ((gg - a) - xh * b);
        pp[0] += dyv * xh;
        pp[ts.npad] += dyv;
        store_cols(g, dx0, q, &f);
      }
    }
  }

  // Writes this CTA's (or cluster rank's) column partials as partial row `part`
  // of the workspace: the row groups of the CTA summed in a fixed order.
  __device__ __forceinline__ static void epilogue(Thread& ts, const Params& p, const Geo& geo,
                                                  unsigned char* colbuf, int64_t c0, int64_t c1,
                                                  int64_t part, int, int ngroups, int, int) {
    __syncthreads();
    const int64_t cols = geo.cols;
    const int n = static_cast<int>(c1 - c0);
    const float* sc = reinterpret_cast<const float*>(colbuf);
    float* out = p.ws + part * 2 * cols;
    for (int k = threadIdx.x; k < 2 * n; k += blockDim.x) {
      const int half = k >= n ? 1 : 0;
      const int j = k - half * n;
      float acc = 0.f;
      for (int gi = 0; gi < ngroups; ++gi) acc += sc[(size_t)gi * 2 * ts.npad + half * ts.npad + j];
      out[half * cols + c0 + j] = acc;
    }
  }
};

// Second stage of the LayerNorm / RMSNorm backward: dgamma_j (and dbeta_j) =
// sum over the P partial rows ([P][planes][cols], planes = 2 for LayerNorm, 1
// for RMSNorm), in a fixed order, so the result is deterministic: the block's
// 32 warps are split into `split` slices over the partials
// (col_reduce_split(P)); warp (slice s, column warp c) sums partials s,
// s + split, ... of its 32 columns, and the slices' sums are added in slice
// order.
template <int DT>
__global__ void __launch_bounds__(1024) col_reduce_kernel(const float* __restrict__ ws, int64_t P,
                                                          int64_t cols, int64_t planes,
                                                          char* dgamma, char* dbeta) {
  constexpr int E = DType<DT>::E;
  __shared__ float part[32][33];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int split = col_reduce_split(P);
  const int ncw = 32 / split;             // column warps per block
  const int cw = w % ncw, sl = w / ncw;   // this warp's columns and slice
  const int64_t k = ((int64_t)blockIdx.x * ncw + cw) * 32 + lane;
  const int64_t n2 = planes * cols;
  float s = 0.f;
  if (k < n2) {
    int64_t pp = sl;
    const int64_t st = split;
    for (; pp + 3 * st < P; pp += 4 * st) {
      const float a0 = __ldcs(ws + pp * n2 + k);
      const float a1 = __ldcs(ws + (pp + st) * n2 + k);
      const float a2 = __ldcs(ws + (pp + 2 * st) * n2 + k);
      const float a3 = __ldcs(ws + (pp + 3 * st) * n2 + k);
      s += a0;
      s += a1;
      s += a2;
      s += a3;
    }
    for (; pp < P; pp += st) s += __ldcs(ws + pp * n2 + k);
  }
  part[w][lane] = s;
  __syncthreads();
  if (sl == 0 && k < n2) {
    float t = part[cw][lane];
    for (int i = 1; i < split; ++i) t += part[i * ncw + cw][lane];
    char* dst = (k < cols) ? dgamma + k * E : dbeta + (k - cols) * E;
    st_elem<DT>(dst, t);
  }
}

}  // namespace rr
