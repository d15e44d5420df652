// rr_ops.cuh -- the three operations as policies of the row engine.
//
//   OpSoftmaxXent  softmax forward, and (with labels) fused cross-entropy
//                  loss + dlogits = softmax - onehot in the same pass
//                  ("Engineering a CUDA Machine Learning Framework from Scratch",
//                  sec. 3.1 "Online FlashSoftmax" and sec. 2.1).
//   OpLnFwd        LayerNorm forward with one-pass moments merged by the
//                  Welford / Chan pairwise rule (same page, sec. 3.2).
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

// Mean S / n of a double-float sum as a double-float (mh + ml).
__device__ __forceinline__ void df_div(float sh, float sl, float n, float& mh, float& ml) {
  mh = sh / n;
  const float r = fmaf(-mh, n, sh);  // exact remainder of the division
  ml = (r + sl) / n;
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

// Per-column vector (gamma, beta) slots a thread keeps for its own columns.
template <int DT, int W, int NQ>
struct ColRegs {
  using Slot = typename std::conditional<(W > 1), uint4, float>::type;
  Slot v[NQ];
  __device__ __forceinline__ float get(int q, int e) const {
    if constexpr (W > 1) return chunk_get<DT>(v[q], e);
    else return v[q];
  }
  // Loads the thread's columns (chunk c = first + q * step covers columns
  // c0 + c*W ... ; chunk mode is only used when every row is 16-byte aligned).
  __device__ __forceinline__ void load(const char* base, int64_t c0, int64_t c1, int64_t first,
                                       int step) {
    constexpr int E = DType<DT>::E;
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      const int64_t c = first + (int64_t)q * step;
      const int64_t j = c0 + c * W;
      if (j < c1) {
        if constexpr (W > 1) v[q] = ld_chunk_cached(base + j * E);
        else v[q] = ld_elem_cached<DT>(base + j * E);
      } else {
        if constexpr (W > 1) v[q] = make_uint4(0, 0, 0, 0);
        else v[q] = 0.f;
      }
    }
  }
};

// ------------------------------------------------- softmax / cross-entropy --

template <int DT_, int W_, int NQ_>
struct OpSoftmaxXent {
  static constexpr int DT = DT_, W = W_, NT = 1, NQ = NQ_;
  static constexpr int E = DType<DT>::E;
  using Stats = MaxSum;
  using Merge = MergeMaxSum;
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
                                                     int64_t, int, int) {}

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
  __device__ __forceinline__ static Stats thread_stats(Thread&, const RowRegs<DT, W, NT, NQ>& x,
                                                       const RowGeo<DT, W>& g, const Meta&) {
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

  __device__ __forceinline__ static void finish(Thread&, const Params& p, const Geo& geo,
                                                int64_t r, const Meta& mt, const Stats& s,
                                                const RowRegs<DT, W, NT, NQ>& x,
                                                const RowGeo<DT, W>& g, bool leader) {
    char* y0 = p.y + (r * p.cols + g.c0) * E - g.head_bytes;
    const bool masked = (s.m == -INFINITY);
    int ql = -1, el = 0;  // where this thread holds the label column, if it does
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
        float xl = 0.f;
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
    // p_j = 2^(x_j log2 e - fl(m log2 e)) * 2^(-r) / d
    const float mL = s.m * kLog2e;
    const float rr = fmaf(s.m, kLog2e, -mL);
    const float inv = ex2(-rr) / s.d;
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      if (!g.has(q)) break;
      float f[W];
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

// ------------------------------------------------------- LayerNorm forward --

template <int DT_, int W_, int NQ_>
struct OpLnFwd {
  static constexpr int DT = DT_, W = W_, NT = 1, NQ = NQ_;
  static constexpr int E = DType<DT>::E;
  using Stats = Moments;
  using Merge = MergeMoments;
  using Params = LnFwdParams;
  struct Meta {};
  struct Thread {
    ColRegs<DT, W, NQ> gamma, beta;
  };

  __device__ __forceinline__ static Meta meta(const Params&, int64_t) { return {}; }
  __device__ __forceinline__ static bool skip(const Meta&) { return false; }
  __device__ __forceinline__ static float fill() { return 0.f; }
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
  __device__ __forceinline__ static void thread_init(Thread& ts, const Params& p, const Geo&,
                                                     int64_t c0, int64_t c1, int gt, int G) {
    ts.gamma.load(p.gamma, c0, c1, gt, G);
    ts.beta.load(p.beta, c0, c1, gt, G);
  }

  // Moments of the thread's own values: a compensated (Neumaier) sum, then the
  // squared deviations from that exact mean (two passes over registers); the
  // threads' moments are then merged with the pairwise update.
  __device__ __forceinline__ static Stats thread_stats(Thread&, const RowRegs<DT, W, NT, NQ>& x,
                                                       const RowGeo<DT, W>& g, const Meta&) {
    float n = 0.f, s = 0.f, c = 0.f;
    g.template for_each<NQ>([&](int q, int e) {
      const float v = x.get(0, q, e);
      const float t = s + v;
      c += (fabsf(s) >= fabsf(v)) ? ((s - t) + v) : ((v - t) + s);
      s = t;
      n += 1.f;
    });
    if (n == 0.f) return Stats::identity();
    float sh, sl;
    two_sum(s, c, sh, sl);
    float mh, ml;
    df_div(sh, sl, n, mh, ml);
    float m2 = 0.f;
    g.template for_each<NQ>([&](int q, int e) {
      const float d = (x.get(0, q, e) - mh) - ml;
      m2 = fmaf(d, d, m2);
    });
    return {n, sh, sl, m2};
  }

  __device__ __forceinline__ static void finish(Thread& ts, const Params& p, const Geo& geo,
                                                int64_t r, const Meta&, const Stats& s,
                                                const RowRegs<DT, W, NT, NQ>& x,
                                                const RowGeo<DT, W>& g, bool leader) {
    char* y0 = p.y + (r * p.cols + g.c0) * E - g.head_bytes;
    const float n = static_cast<float>(geo.cols);
    float mh, ml;
    df_div(s.sh, s.sl, n, mh, ml);
    const float var = s.m2 / n;
    const bool masked = !(isfinite(mh) && isfinite(ml) && isfinite(var));
    if (masked) {
      if (leader) {
        p.mean[r] = 0.f;
        p.rstd[r] = 0.f;
      }
      g.template store<NQ>(y0, [&](int, int) { return 0.f; });
      return;
    }
    const float rstd = 1.0f / sqrtf(var + p.eps);
    if (leader) {
      p.mean[r] = mh + ml;
      p.rstd[r] = rstd;
    }
    g.template store<NQ>(y0, [&](int q, int e) {
      const float xh = ((x.get(0, q, e) - mh) - ml) * rstd;
      return fmaf(xh, ts.gamma.get(q, e), ts.beta.get(q, e));
    });
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
  using Stats = Sum2;
  using Merge = MergeSum2;
  using Params = LnBwdParams;
  struct Meta {
    float mean, rstd;
  };
  struct Thread {
    ColRegs<DT, W, NQ> gamma;
    float dg[NQ][W];
    float db[NQ][W];
  };

  __device__ __forceinline__ static Meta meta(const Params& p, int64_t r) {
    if (r < 0) return {0.f, 0.f};
    return {__ldg(p.mean + r), __ldg(p.rstd + r)};
  }
  // A row the forward masked (rstd == 0) is neither read nor accumulated.
  __device__ __forceinline__ static bool skip(const Meta& m) { return m.rstd == 0.f; }
  __device__ __forceinline__ static float fill() { return 0.f; }
  __device__ __forceinline__ static const char* in_slice_start(const Params& p, int t, int64_t r,
                                                               int64_t c0) {
    return (t == 0 ? p.dy : p.x) + (r * p.cols + c0) * E;
  }
  __device__ __forceinline__ static uint64_t start_addr(const Params& p, int64_t r, int64_t c0) {
    return reinterpret_cast<uint64_t>(in_slice_start(p, 0, r, c0));
  }
  __device__ __forceinline__ static const char* in_chunk0(const Params& p, int t, int64_t r,
                                                          int64_t c0, const RowGeo<DT, W>& g) {
    return in_slice_start(p, t, r, c0) - g.head_bytes;
  }
  __device__ __forceinline__ static void thread_init(Thread& ts, const Params& p, const Geo&,
                                                     int64_t c0, int64_t c1, int gt, int G) {
    ts.gamma.load(p.gamma, c0, c1, gt, G);
#pragma unroll
    for (int q = 0; q < NQ; ++q)
#pragma unroll
      for (int e = 0; e < W; ++e) {
        ts.dg[q][e] = 0.f;
        ts.db[q][e] = 0.f;
      }
  }

  __device__ __forceinline__ static Stats thread_stats(Thread& ts,
                                                       const RowRegs<DT, W, NT, NQ>& v,
                                                       const RowGeo<DT, W>& g, const Meta& m) {
    float s1 = 0.f, s2 = 0.f;
    g.template for_each<NQ>([&](int q, int e) {
      const float xh = (v.get(1, q, e) - m.mean) * m.rstd;
      // rounded product (never fused into an FMA) so finish() sees the same g
      const float gg = __fmul_rn(v.get(0, q, e), ts.gamma.get(q, e));
      s1 += gg;
      s2 = fmaf(gg, xh, s2);
    });
    return {s1, s2};
  }

  __device__ __forceinline__ static void finish(Thread& ts, const Params& p, const Geo& geo,
                                                int64_t r, const Meta& m, const Stats& s,
                                                const RowRegs<DT, W, NT, NQ>& v,
                                                const RowGeo<DT, W>& g, bool) {
    char* dx0 = p.dx + (r * p.cols + g.c0) * E - g.head_bytes;
    if (skip(m)) {
      g.template store<NQ>(dx0, [&](int, int) { return 0.f; });
      return;
    }
    const float invc = 1.0f / static_cast<float>(geo.cols);
    const float a = s.s1 * invc;
    const float b = s.s2 * invc;
    g.template store<NQ>(dx0, [&](int q, int e) {
      const float xh = (v.get(1, q, e) - m.mean) * m.rstd;
      const float gg = __fmul_rn(v.get(0, q, e), ts.gamma.get(q, e));
      return m.rstd * ((gg - a) - xh * b);
    });
    g.template for_each<NQ>([&](int q, int e) {
      const float dyv = v.get(0, q, e);
      const float xh = (v.get(1, q, e) - m.mean) * m.rstd;
      ts.dg[q][e] = fmaf(dyv, xh, ts.dg[q][e]);
      ts.db[q][e] += dyv;
    });
  }

  // Writes this CTA's (or cluster's) column partials: partial row `part` of the
  // workspace.  With several row groups per CTA the groups are summed through
  // shared memory in a fixed order first.
  __device__ __forceinline__ static void epilogue(Thread& ts, const Params& p, const Geo& geo,
                                                  unsigned char* colbuf, int64_t c0, int64_t c1,
                                                  int64_t part, int grp, int ngroups, int gt,
                                                  int G) {
    const int64_t cols = geo.cols;
    float* out = p.ws + part * 2 * cols;
    if (ngroups == 1) {
#pragma unroll
      for (int q = 0; q < NQ; ++q)
#pragma unroll
        for (int e = 0; e < W; ++e) {
          const int64_t j = c0 + ((int64_t)gt + (int64_t)q * G) * W + e;
          if (j < c1) {
            out[j] = ts.dg[q][e];
            out[cols + j] = ts.db[q][e];
          }
        }
      return;
    }
    float* sc = reinterpret_cast<float*>(colbuf);  // [ngroups][2][cols]
#pragma unroll
    for (int q = 0; q < NQ; ++q)
#pragma unroll
      for (int e = 0; e < W; ++e) {
        const int64_t j = c0 + ((int64_t)gt + (int64_t)q * G) * W + e;
        if (j < c1) {
          sc[(int64_t)grp * 2 * cols + j] = ts.dg[q][e];
          sc[(int64_t)grp * 2 * cols + cols + j] = ts.db[q][e];
        }
      }
    __syncthreads();
    for (int64_t k = threadIdx.x; k < 2 * cols; k += blockDim.x) {
      float acc = 0.f;
      for (int gi = 0; gi < ngroups; ++gi) acc += sc[(int64_t)gi * 2 * cols + k];
      out[k] = acc;
    }
  }
};

// Second stage of the LayerNorm backward: dgamma_j / dbeta_j = sum over the P
// partial rows, in a fixed order (warp w takes partials w, w+8, ...; the eight
// warp sums are then added in warp order), so the result is deterministic.
template <int DT>
__global__ void __launch_bounds__(256) col_reduce_kernel(const float* __restrict__ ws, int64_t P,
                                                         int64_t cols, char* dgamma, char* dbeta) {
  constexpr int E = DType<DT>::E;
  __shared__ float part[8][33];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t k = (int64_t)blockIdx.x * 32 + lane;
  const int64_t n2 = 2 * cols;
  float s = 0.f;
  if (k < n2) {
    int64_t pp = w;
    for (; pp + 24 < P; pp += 32) {
      const float a0 = __ldcs(ws + pp * n2 + k);
      const float a1 = __ldcs(ws + (pp + 8) * n2 + k);
      const float a2 = __ldcs(ws + (pp + 16) * n2 + k);
      const float a3 = __ldcs(ws + (pp + 24) * n2 + k);
      s += a0;
      s += a1;
      s += a2;
      s += a3;
    }
    for (; pp < P; pp += 8) s += __ldcs(ws + pp * n2 + k);
  }
  part[w][lane] = s;
  __syncthreads();
  if (w == 0 && k < n2) {
    float t = part[0][lane];
#pragma unroll
    for (int i = 1; i < 8; ++i) t += part[i][lane];
    char* dst = (k < cols) ? dgamma + k * E : dbeta + (k - cols) * E;
    st_elem<DT>(dst, t);
  }
}

}  // namespace rr
