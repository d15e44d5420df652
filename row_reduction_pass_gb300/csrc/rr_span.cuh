// rr_span.cuh -- short rows as contiguous spans of rows per warp: softmax,
// log-softmax and cross-entropy, the softmax / log-softmax backward, and the
// LayerNorm / RMSNorm forward and backward, for rows whose byte length is not
// a multiple of 16 (up to 448 bytes by operation; 64 for the norm backward).
//
// With rows this short a row-group kernel moves only a few bytes per thread
// per row, far too little in flight to cover DRAM latency, and a misaligned row
// costs it funnel shifts or element loads.  Here each warp owns
// a span of S = 32 x RPL consecutive rows (about 3 KB; a multiple of 16 bytes,
// so spans start 16-byte aligned when the tensor does): its lanes copy the span
// into the warp's shared-memory buffer with 16-byte cp.async copies, one span
// ahead (two buffers), then lane l computes rows l, l + 32, ... of the span from
// shared memory, writes each row's outputs back over its inputs, and the warp
// stores the span out as 16-byte blocks.  Only warp-level synchronisation: no
// block barrier.  The arithmetic of a row is the online normaliser of the row
// engine (rr_ops.cuh, OpSoftmaxXent) done by one lane: max, sum of exp, output.
#pragma once

#include "rr_kernels.h"
#include "rr_ops.cuh"

namespace rr {

struct SpanGeo {
  int64_t rows;
  int32_t cols;
  int32_t rpl;      // rows per lane per span
  int32_t span_b;   // bytes per span buffer (rows_per_span * cols * E, a multiple of 16)
  int32_t lab_b;    // cross-entropy with 16-byte aligned labels: label bytes per span, else 0;
                    // norm backward: bytes of one row statistic per span
  int32_t staged;   // norm backward: mean / rstd 16-byte aligned, copied with the span
};

constexpr int kSpanWarps = 8;  // warps per block

template <int DT>
__device__ __forceinline__ float span_ld(const unsigned char* s, int i) {
  if constexpr (DT == kF32) return reinterpret_cast<const float*>(s)[i];
  else return bf16_bits_to_f32(reinterpret_cast<const unsigned short*>(s)[i]);
}
template <int DT>
__device__ __forceinline__ void span_st(unsigned char* s, int i, float f) {
  if constexpr (DT == kF32) reinterpret_cast<float*>(s)[i] = f;
  else reinterpret_cast<unsigned short*>(s)[i] = f32_to_bf16_bits(f);
}

// MODE 0: softmax, 1: log-softmax, 2: cross-entropy (loss, dlogits).
template <int DT, int MODE>
__global__ void __launch_bounds__(32 * kSpanWarps)
    span_softmax_kernel(const SoftmaxParams p, const SpanGeo geo) {
  constexpr int E = DType<DT>::E;
  extern __shared__ __align__(128) unsigned char smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int C = geo.cols;
  const int rps = 32 * geo.rpl;  // rows per span
  const int64_t nspans = (geo.rows + rps - 1) / rps;
  const int64_t gw = (int64_t)blockIdx.x * kSpanWarps + warp;
  const int64_t nw = (int64_t)gridDim.x * kSpanWarps;
  unsigned char* buf = smem + (size_t)warp * 2 * geo.span_b;
  // staged labels (cross-entropy): [warps][2 stages][rows per span] int32
  int32_t* lbuf = reinterpret_cast<int32_t*>(smem + (size_t)kSpanWarps * 2 * geo.span_b +
                                             (size_t)warp * 2 * geo.lab_b);
  const int64_t rowb = (int64_t)C * E;
  const int64_t total = geo.rows * rowb;

  // bytes of span s: [s * span_b, min(.., total)); whole 16-byte blocks by
  // cp.async, the ragged end of the tensor's last span element by element
  auto span_bytes = [&](int64_t s) -> int64_t {
    const int64_t b0 = s * geo.span_b;
    const int64_t b1 = b0 + geo.span_b < total ? b0 + geo.span_b : total;
    return b1 - b0;
  };
  auto issue = [&](int64_t s, int stage) {
    if (s < nspans) {
      const int64_t nb = span_bytes(s);
      const char* src = p.x + s * geo.span_b;
      unsigned char* dst = buf + stage * geo.span_b;
      for (int64_t j = lane; j < nb / 16; j += 32) cp_async16(dst + 16 * j, src + 16 * j);
      if (MODE == 2 && geo.lab_b > 0) {
        // the span's labels: whole 16-byte blocks (4 rows each); a last span's
        // ragged rows are read directly
        const int64_t r0 = s * rps;
        const int64_t nr = geo.rows - r0 < rps ? geo.rows - r0 : rps;
        const int32_t* lsrc = p.labels + r0;
        int32_t* ldst = lbuf + stage * (geo.lab_b / 4);
        for (int64_t j = lane; j < nr / 4; j += 32) cp_async16(ldst + 4 * j, lsrc + 4 * j);
      }
    }
    cp_async_commit();
  };

  issue(gw, 0);
  for (int64_t it = 0;; ++it) {
    const int64_t s = gw + it * nw;
    if (s >= nspans) break;
    const int stage = (int)(it & 1);
    unsigned char* sb = buf + stage * geo.span_b;
    const int64_t r0 = s * rps;
    const int nrows = (int)(geo.rows - r0 < rps ? geo.rows - r0 : rps);
    issue(s + nw, stage ^ 1);
    cp_async_wait<1>();
    const int64_t nb = span_bytes(s);
    if (lane == 0)
      for (int64_t b = nb & ~int64_t(15); b < nb; b += E)
        span_st<DT>(sb, (int)(b / E), ld_elem<DT>(p.x + s * geo.span_b + b));
    __syncwarp();

    for (int k = 0; k < geo.rpl; ++k) {
      const int i = lane + 32 * k;
      if (i >= nrows) break;
      const int base = i * C;
      float m = -INFINITY;
      for (int j = 0; j < C; ++j) m = fmaxf(m, span_ld<DT>(sb, base + j));
      const int64_t r = r0 + i;
      bool skip = false;
      int32_t label = -1;
      if constexpr (MODE == 2) {
        label = (geo.lab_b > 0 && i < (nrows & ~3)) ? lbuf[stage * (geo.lab_b / 4) + i]
                                                      : __ldg(p.labels + r);
        skip = label == p.ignore;
        const bool in_range = label >= 0 && label < C;
        if (!skip && !in_range && p.bad != nullptr) atomicAdd(p.bad, 1);
        if (skip || m == -INFINITY) {
          p.loss[r] = 0.f;
        } else if (!in_range) {
          p.loss[r] = __int_as_float(0x7fc00000);
        }
      }
      if (skip || m == -INFINITY) {
        for (int j = 0; j < C; ++j) span_st<DT>(sb, base + j, 0.f);
        continue;
      }
      // d = sum exp(x - m) as sum 2^(x log2e - fl(m log2e)) * 2^(-r), r the
      // rounding residual of fl(m log2e)
      const float mL = m * kLog2e;
      const float rr = fmaf(m, kLog2e, -mL);
      float d = 0.f;
      for (int j = 0; j < C; ++j) d += ex2(fmaf(span_ld<DT>(sb, base + j), kLog2e, -mL));
      d *= ex2(-rr);
      if constexpr (MODE == 1) {
        const float lnd = logf(d);
        for (int j = 0; j < C; ++j)
          span_st<DT>(sb, base + j, (span_ld<DT>(sb, base + j) - m) - lnd);
      } else {
        if constexpr (MODE == 2) {
          if (label >= 0 && label < C)
            p.loss[r] = (m - span_ld<DT>(sb, base + label)) + logf(d);
        }
        const float inv = ex2(-rr) / d;
        for (int j = 0; j < C; ++j) {
          float f = ex2(fmaf(span_ld<DT>(sb, base + j), kLog2e, -mL)) * inv;
          if (MODE == 2 && j == label) f -= 1.0f;
          span_st<DT>(sb, base + j, f);
        }
      }
    }
    __syncwarp();
    // the span out: whole blocks as 16-byte stores, the ragged end by lane 0
    char* dst = p.y + s * geo.span_b;
    for (int64_t j = lane; j < nb / 16; j += 32)
      st_chunk_stream(dst + 16 * j, *reinterpret_cast<const uint4*>(sb + 16 * j));
    if (lane == 0)
      for (int64_t b = nb & ~int64_t(15); b < nb; b += E)
        st_elem<DT>(dst + b, span_ld<DT>(sb, (int)(b / E)));
    __syncwarp();
  }
  cp_async_wait<0>();
}

// Softmax (LOG = false: y, dy) or log-softmax (LOG = true: z, dz) backward of
// short rows, spans as above with two input buffers per stage; dx is written
// over the dy buffer and stored out.  Per row: S = sum y*dy (or sum dz), then
// dx = y * (dy - S) (or dz - exp(z) * S), as OpSoftmaxBwd in rr_ops.cuh.
template <int DT, bool LOG>
__global__ void __launch_bounds__(32 * kSpanWarps)
    span_softmax_bwd_kernel(const SoftmaxBwdParams p, const SpanGeo geo) {
  constexpr int E = DType<DT>::E;
  extern __shared__ __align__(128) unsigned char smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int C = geo.cols;
  const int rps = 32 * geo.rpl;
  const int64_t nspans = (geo.rows + rps - 1) / rps;
  const int64_t gw = (int64_t)blockIdx.x * kSpanWarps + warp;
  const int64_t nw = (int64_t)gridDim.x * kSpanWarps;
  unsigned char* buf = smem + (size_t)warp * 4 * geo.span_b;  // [stage][y | dy]
  const int64_t total = geo.rows * (int64_t)C * E;
  auto span_bytes = [&](int64_t s) -> int64_t {
    const int64_t b0 = s * geo.span_b;
    const int64_t b1 = b0 + geo.span_b < total ? b0 + geo.span_b : total;
    return b1 - b0;
  };
  auto issue = [&](int64_t s, int stage) {
    if (s < nspans) {
      const int64_t nb = span_bytes(s);
      unsigned char* d0 = buf + (2 * stage) * geo.span_b;
      unsigned char* d1 = d0 + geo.span_b;
      const char* s0 = p.y + s * geo.span_b;
      const char* s1 = p.dy + s * geo.span_b;
      for (int64_t j = lane; j < nb / 16; j += 32) {
        cp_async16(d0 + 16 * j, s0 + 16 * j);
        cp_async16(d1 + 16 * j, s1 + 16 * j);
      }
    }
    cp_async_commit();
  };

  issue(gw, 0);
  for (int64_t it = 0;; ++it) {
    const int64_t s = gw + it * nw;
    if (s >= nspans) break;
    const int stage = (int)(it & 1);
    unsigned char* yb = buf + (2 * stage) * geo.span_b;
    unsigned char* gb = yb + geo.span_b;
    const int64_t r0 = s * rps;
    const int nrows = (int)(geo.rows - r0 < rps ? geo.rows - r0 : rps);
    issue(s + nw, stage ^ 1);
    cp_async_wait<1>();
    const int64_t nb = span_bytes(s);
    if (lane == 0)
      for (int64_t b = nb & ~int64_t(15); b < nb; b += E) {
        span_st<DT>(yb, (int)(b / E), ld_elem<DT>(p.y + s * geo.span_b + b));
        span_st<DT>(gb, (int)(b / E), ld_elem<DT>(p.dy + s * geo.span_b + b));
      }
    __syncwarp();
    for (int k = 0; k < geo.rpl; ++k) {
      const int i = lane + 32 * k;
      if (i >= nrows) break;
      const int base = i * C;
      float S = 0.f;
      for (int j = 0; j < C; ++j)
        S = LOG ? S + span_ld<DT>(gb, base + j)
                : fmaf(span_ld<DT>(yb, base + j), span_ld<DT>(gb, base + j), S);
      for (int j = 0; j < C; ++j) {
        const float yv = span_ld<DT>(yb, base + j), gv = span_ld<DT>(gb, base + j);
        span_st<DT>(gb, base + j, LOG ? fmaf(ex2(yv * kLog2e), -S, gv) : yv * (gv - S));
      }
    }
    __syncwarp();
    char* dst = p.dx + s * geo.span_b;
    for (int64_t j = lane; j < nb / 16; j += 32)
      st_chunk_stream(dst + 16 * j, *reinterpret_cast<const uint4*>(gb + 16 * j));
    if (lane == 0)
      for (int64_t b = nb & ~int64_t(15); b < nb; b += E)
        st_elem<DT>(dst + b, span_ld<DT>(gb, (int)(b / E)));
    __syncwarp();
  }
  cp_async_wait<0>();
}

// LayerNorm (RMS = false) or RMSNorm forward of short rows, spans as above.
// One lane owns a whole row, so no reduction across threads: a compensated
// (TwoSum) sum gives the exact mean (mh + ml), then M2 about it (RMSNorm: the
// plain sum of squares), as ln_fwd_kernel in rr_ln.cuh.  gamma / beta are
// converted to fp32 once per block into shared memory after the span buffers.
template <int DT, bool RMS>
__global__ void __launch_bounds__(32 * kSpanWarps)
    span_ln_fwd_kernel(const LnFwdParams p, const SpanGeo geo) {
  constexpr int E = DType<DT>::E;
  extern __shared__ __align__(128) unsigned char smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int C = geo.cols;
  const int rps = 32 * geo.rpl;
  const int64_t nspans = (geo.rows + rps - 1) / rps;
  const int64_t gw = (int64_t)blockIdx.x * kSpanWarps + warp;
  const int64_t nw = (int64_t)gridDim.x * kSpanWarps;
  unsigned char* buf = smem + (size_t)warp * 2 * geo.span_b;
  float* sg = reinterpret_cast<float*>(smem + (size_t)kSpanWarps * 2 * geo.span_b);
  float* sbeta = sg + C;
  for (int j = threadIdx.x; j < C; j += blockDim.x) {
    sg[j] = ld_elem_cached<DT>(p.gamma + (int64_t)j * E);
    if constexpr (!RMS) sbeta[j] = ld_elem_cached<DT>(p.beta + (int64_t)j * E);
  }
  __syncthreads();
  const int64_t total = geo.rows * (int64_t)C * E;
  const float ns = static_cast<float>(C);
  auto span_bytes = [&](int64_t s) -> int64_t {
    const int64_t b0 = s * geo.span_b;
    const int64_t b1 = b0 + geo.span_b < total ? b0 + geo.span_b : total;
    return b1 - b0;
  };
  auto issue = [&](int64_t s, int stage) {
    if (s < nspans) {
      const int64_t nb = span_bytes(s);
      const char* src = p.x + s * geo.span_b;
      unsigned char* dst = buf + stage * geo.span_b;
      for (int64_t j = lane; j < nb / 16; j += 32) cp_async16(dst + 16 * j, src + 16 * j);
    }
    cp_async_commit();
  };

  issue(gw, 0);
  for (int64_t it = 0;; ++it) {
    const int64_t s = gw + it * nw;
    if (s >= nspans) break;
    const int stage = (int)(it & 1);
    unsigned char* sb = buf + stage * geo.span_b;
    const int64_t r0 = s * rps;
    const int nrows = (int)(geo.rows - r0 < rps ? geo.rows - r0 : rps);
    issue(s + nw, stage ^ 1);
    cp_async_wait<1>();
    const int64_t nb = span_bytes(s);
    if (lane == 0)
      for (int64_t b = nb & ~int64_t(15); b < nb; b += E)
        span_st<DT>(sb, (int)(b / E), ld_elem<DT>(p.x + s * geo.span_b + b));
    __syncwarp();
    for (int k = 0; k < geo.rpl; ++k) {
      const int i = lane + 32 * k;
      if (i >= nrows) break;
      const int base = i * C;
      const int64_t r = r0 + i;
      float mh = 0.f, ml = 0.f, var;
      if constexpr (RMS) {
        float a = 0.f;
        for (int j = 0; j < C; ++j) {
          const float v = span_ld<DT>(sb, base + j);
          a = fmaf(v, v, a);
        }
        var = a * p.inv_cols;
      } else {
        float sum = 0.f, c = 0.f;
        for (int j = 0; j < C; ++j) {
          float t, e;
          two_sum(sum, span_ld<DT>(sb, base + j), t, e);
          sum = t;
          c += e;
        }
        float sh, sl;
        two_sum(sum, c, sh, sl);
        df_mean(sh, sl, ns, p.inv_cols, mh, ml);
        float a = 0.f;
        for (int j = 0; j < C; ++j) {
          const float d = (span_ld<DT>(sb, base + j) - mh) - ml;
          a = fmaf(d, d, a);
        }
        var = a * p.inv_cols;
      }
      const bool masked = RMS ? !isfinite(var) : !(isfinite(mh) && isfinite(ml) && isfinite(var));
      const float rstd = masked ? 0.f : rsqrtf(var + p.eps);
      if constexpr (!RMS) p.mean[r] = masked ? 0.f : mh + ml;
      p.rstd[r] = rstd;
      for (int j = 0; j < C; ++j) {
        float f = 0.f;
        if (!masked) {
          const float v = span_ld<DT>(sb, base + j);
          f = RMS ? (v * rstd) * sg[j] : fmaf(((v - mh) - ml) * rstd, sg[j], sbeta[j]);
        }
        span_st<DT>(sb, base + j, f);
      }
    }
    __syncwarp();
    char* dst = p.y + s * geo.span_b;
    for (int64_t j = lane; j < nb / 16; j += 32)
      st_chunk_stream(dst + 16 * j, *reinterpret_cast<const uint4*>(sb + 16 * j));
    if (lane == 0)
      for (int64_t b = nb & ~int64_t(15); b < nb; b += E)
        st_elem<DT>(dst + b, span_ld<DT>(sb, (int)(b / E)));
    __syncwarp();
  }
  cp_async_wait<0>();
}

// LayerNorm (RMS = false) or RMSNorm backward of short rows (at most 64 bytes,
// bf16 96 bytes, so C <= 48; the column pass holds up to 64 columns; with
// longer rows two tensors' spans leave room for one block per SM and the
// other kernels are faster).  Per stage a warp
// copies spans of dy and x and the span's row statistics (mean, rstd: by
// cp.async when they are 16-byte aligned, else loaded into the same buffer).
// Two passes over the staged span:
//  - columns: the column partials sum dy*xhat (and sum dy) in registers, lane
//    l taking column l % C of rows l / C, l / C + 32 / C, ... (C > 32: columns
//    l and l + 32 of every row): consecutive lanes read consecutive elements;
//  - rows: lane l takes rows l, l + 32, ...: S1 = sum g, S2 = sum g*xhat with
//    g = dy*gamma, and dx = rstd*((g - S1/C) - xhat*S2/C), written over dy in
//    shared memory and stored out as 16-byte blocks.
// rstd == 0 marks a row the forward masked: dx = 0 and no contribution.  At the
// end the block adds its lanes' partials in a fixed order (warp, then row
// phase) into its row of the workspace, [gridDim.x][planes][C] floats, which
// col_reduce_kernel sums.
template <int DT, bool RMS>
__global__ void __launch_bounds__(32 * kSpanWarps, 3)
    span_ln_bwd_kernel(const LnBwdParams p, const SpanGeo geo) {
  constexpr int E = DType<DT>::E;
  constexpr int kPlanes = RMS ? 1 : 2;
  extern __shared__ __align__(128) unsigned char smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int C = geo.cols;
  const int rps = 32 * geo.rpl;
  const int64_t nspans = (geo.rows + rps - 1) / rps;
  const int64_t gw = (int64_t)blockIdx.x * kSpanWarps + warp;
  const int64_t nw = (int64_t)gridDim.x * kSpanWarps;
  // [warps][2 stages][dy | x] spans, then [warps][2 stages][mean | rstd][rps]
  // floats, then gamma as fp32
  unsigned char* buf = smem + (size_t)warp * 4 * geo.span_b;
  const int nst = geo.lab_b / 4;  // rows per span, as floats
  float* stats = reinterpret_cast<float*>(smem + (size_t)kSpanWarps * 4 * geo.span_b) +
                 (size_t)warp * 4 * nst;
  float* sg = reinterpret_cast<float*>(smem + (size_t)kSpanWarps * 4 * (geo.span_b + geo.lab_b));
  for (int j = threadIdx.x; j < C; j += blockDim.x) sg[j] = ld_elem_cached<DT>(p.gamma + (int64_t)j * E);
  __syncthreads();

  // column pass geometry: for C <= 32, nph row phases of C lanes (lane l takes
  // column l % C of rows l / C, l / C + nph, ...); for 32 < C <= 64 one phase,
  // lane l taking columns l and l + 32 of every row
  const bool wide = C > 32;
  const int nph = wide ? 1 : 32 / C;
  const int ph = wide ? 0 : lane / C;
  const int j0 = wide ? lane : lane % C;
  const int j1 = lane + 32;
  const bool on = ph < nph;
  const bool on1 = wide && j1 < C;
  float ag = 0.f, ab = 0.f, ag1 = 0.f, ab1 = 0.f;

  const int64_t total = geo.rows * (int64_t)C * E;
  auto span_bytes = [&](int64_t s) -> int64_t {
    const int64_t b0 = s * geo.span_b;
    const int64_t b1 = b0 + geo.span_b < total ? b0 + geo.span_b : total;
    return b1 - b0;
  };
  auto issue = [&](int64_t s, int stage) {
    if (s < nspans) {
      const int64_t nb = span_bytes(s);
      unsigned char* d0 = buf + (2 * stage) * geo.span_b;
      unsigned char* d1 = d0 + geo.span_b;
      const char* s0 = p.dy + s * geo.span_b;
      const char* s1 = p.x + s * geo.span_b;
      for (int64_t j = lane; j < nb / 16; j += 32) {
        cp_async16(d0 + 16 * j, s0 + 16 * j);
        cp_async16(d1 + 16 * j, s1 + 16 * j);
      }
      if (geo.staged) {
        const int64_t r0 = s * rps;
        const int64_t nr = geo.rows - r0 < rps ? geo.rows - r0 : rps;
        float* sm = stats + (2 * stage) * nst;
        for (int64_t j = lane; j < nr / 4; j += 32) {
          if (!RMS) cp_async16(sm + 4 * j, p.mean + r0 + 4 * j);
          cp_async16(sm + nst + 4 * j, p.rstd + r0 + 4 * j);
        }
      }
    }
    cp_async_commit();
  };

  issue(gw, 0);
  for (int64_t it = 0;; ++it) {
    const int64_t s = gw + it * nw;
    if (s >= nspans) break;
    const int stage = (int)(it & 1);
    unsigned char* gbuf = buf + (2 * stage) * geo.span_b;  // dy, then dx
    unsigned char* xbuf = gbuf + geo.span_b;
    float* smean = stats + (2 * stage) * nst;
    float* srstd = smean + nst;
    const int64_t r0 = s * rps;
    const int nrows = (int)(geo.rows - r0 < rps ? geo.rows - r0 : rps);
    issue(s + nw, stage ^ 1);
    cp_async_wait<1>();
    const int64_t nb = span_bytes(s);
    if (lane == 0)
      for (int64_t b = nb & ~int64_t(15); b < nb; b += E) {
        span_st<DT>(gbuf, (int)(b / E), ld_elem<DT>(p.dy + s * geo.span_b + b));
        span_st<DT>(xbuf, (int)(b / E), ld_elem<DT>(p.x + s * geo.span_b + b));
      }
    for (int i = lane + (geo.staged ? (nrows & ~3) : 0); i < nrows; i += 32) {
      if (!RMS) smean[i] = __ldg(p.mean + r0 + i);
      srstd[i] = __ldg(p.rstd + r0 + i);
    }
    __syncwarp();
    if (on)
      for (int i = ph; i < nrows; i += nph) {
        const float rs = srstd[i];
        if (rs == 0.f) continue;
        const float mu = RMS ? 0.f : smean[i];
        const float dyv = span_ld<DT>(gbuf, i * C + j0);
        const float xv = span_ld<DT>(xbuf, i * C + j0);
        const float xh = RMS ? xv * rs : (xv - mu) * rs;
        ag = fmaf(dyv, xh, ag);
        if (!RMS) ab += dyv;
        if (on1) {
          const float dy1 = span_ld<DT>(gbuf, i * C + j1);
          const float x1 = span_ld<DT>(xbuf, i * C + j1);
          const float xh1 = RMS ? x1 * rs : (x1 - mu) * rs;
          ag1 = fmaf(dy1, xh1, ag1);
          if (!RMS) ab1 += dy1;
        }
      }
    __syncwarp();
    for (int k = 0; k < geo.rpl; ++k) {
      const int i = lane + 32 * k;
      if (i >= nrows) break;
      const int base = i * C;
      const float rstd = srstd[i];
      if (rstd == 0.f) {
        for (int j = 0; j < C; ++j) span_st<DT>(gbuf, base + j, 0.f);
        continue;
      }
      const float mean = RMS ? 0.f : smean[i];
      float s1 = 0.f, s2 = 0.f;
      for (int j = 0; j < C; ++j) {
        const float xv = span_ld<DT>(xbuf, base + j);
        const float xh = RMS ? xv * rstd : (xv - mean) * rstd;
        const float g = __fmul_rn(span_ld<DT>(gbuf, base + j), sg[j]);
        if (!RMS) s1 += g;
        s2 = fmaf(g, xh, s2);
      }
      const float a = RMS ? 0.f : s1 * p.inv_cols;
      const float b = s2 * p.inv_cols;
      for (int j = 0; j < C; ++j) {
        const float xv = span_ld<DT>(xbuf, base + j);
        const float xh = RMS ? xv * rstd : (xv - mean) * rstd;
        const float g = __fmul_rn(span_ld<DT>(gbuf, base + j), sg[j]);
        span_st<DT>(gbuf, base + j, fmaf(xh, -b, g - a) * rstd);
      }
    }
    __syncwarp();
    char* dst = p.dx + s * geo.span_b;
    for (int64_t j = lane; j < nb / 16; j += 32)
      st_chunk_stream(dst + 16 * j, *reinterpret_cast<const uint4*>(gbuf + 16 * j));
    if (lane == 0)
      for (int64_t b = nb & ~int64_t(15); b < nb; b += E)
        st_elem<DT>(dst + b, span_ld<DT>(gbuf, (int)(b / E)));
    __syncwarp();
  }
  cp_async_wait<0>();
  __syncthreads();
  // the lanes' partials, [warps][planes][64] floats over the (now idle) span
  // buffers: slot lane holds column j0 of phase ph, slot 32 + lane (wide
  // rows) column lane + 32
  float* red = reinterpret_cast<float*>(smem);
  red[(warp * kPlanes) * 64 + lane] = ag;
  red[(warp * kPlanes) * 64 + 32 + lane] = ag1;
  if (!RMS) {
    red[(warp * kPlanes + 1) * 64 + lane] = ab;
    red[(warp * kPlanes + 1) * 64 + 32 + lane] = ab1;
  }
  __syncthreads();
  float* out = p.ws + (int64_t)blockIdx.x * kPlanes * C;
  for (int idx = threadIdx.x; idx < kPlanes * C; idx += blockDim.x) {
    const int pl = idx / C, j = idx % C;
    float t = 0.f;
    for (int w = 0; w < kSpanWarps; ++w)
      for (int q = 0; q < nph; ++q) t += red[(w * kPlanes + pl) * 64 + q * C + j];
    out[idx] = t;
  }
}

}  // namespace rr
