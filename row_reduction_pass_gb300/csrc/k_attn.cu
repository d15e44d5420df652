// k_attn.cu -- scaled dot-product attention forward built on the online
// softmax ("Engineering a CUDA Machine Learning Framework from Scratch",
// sec. 6.4: the FlashAttention-style extension of sec. 3.1; attention as
// defined by Vaswani et al. 2017, tiled as in Dao et al. 2022).
//
// One CTA of 4 warps owns 64 query rows of one head (16 per warp) and walks
// the key / value tiles of 64 rows (causal: up to the diagonal tile).  Q and
// the K / V tiles are copied into shared memory with 16-byte cp.async (K / V
// double-buffered, rows padded by 8 elements so ldmatrix reads are
// bank-conflict free).  Scores S = Q K^T and the output O += P V are
// warp-level bf16 tensor-core products (mma.sync m16n8k16, fp32
// accumulation); between them each warp keeps, per query row, the running
// maximum m and sum l of the online softmax in the log2 domain (scores scaled
// by scale * log2 e), rescales O by 2^(m_old - m_new) when the maximum grows,
// and turns the probabilities into the bf16 A operand of P V directly from
// the score accumulators.  At the end O / l is stored in bf16 and
// lse = (m + log2 l) * ln 2 in fp32.
//
// Shapes: bf16 q, k, v, o of [bh][s][d], d = 64 or 128, s a multiple of 64,
// 16-byte aligned tensors (checked by the caller).
#include <cstdint>

#include "rr_device.cuh"
#include "rr_kernels.h"

namespace rr {
namespace {

constexpr int kBr = 64;   // query rows per CTA
constexpr int kBc = 64;   // keys per tile
constexpr int kPad = 8;   // padding elements per shared-memory row

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// D = A (16x16, row) * B (16x8, col) + D, bf16 in, fp32 accumulate
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// two floats as a bf16 pair, lo in the low half (round to nearest even)
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Copies a [64][D] bf16 tile (rows of D elements in global memory) into a
// padded [64][D + kPad] shared-memory tile: 8 * D chunks of 16 bytes over the
// CTA's 128 threads.
template <int D>
__device__ __forceinline__ void load_tile(uint16_t* dst, const char* src) {
  constexpr int kChunksPerRow = D / 8;
#pragma unroll
  for (int c = threadIdx.x; c < kBr * kChunksPerRow; c += 128) {
    const int row = c / kChunksPerRow, col8 = c % kChunksPerRow;
    cp_async16(dst + row * (D + kPad) + col8 * 8, src + ((int64_t)row * D + col8 * 8) * 2);
  }
}

template <int D>
__global__ void __launch_bounds__(128) attn_fwd_kernel(const AttnParams p) {
  static_assert(D == 64 || D == 128, "head dimension 64 or 128");
  constexpr int LD = D + kPad;  // shared-memory row stride in elements
  extern __shared__ __align__(128) unsigned char smem[];
  uint16_t* qs = reinterpret_cast<uint16_t*>(smem);
  uint16_t* ks = qs + kBr * LD;        // [2][kBc][LD]
  uint16_t* vs = ks + 2 * kBc * LD;    // [2][kBc][LD]

  // grid (heads, query tiles): blocks are dispatched x fastest, so every head's
  // heaviest causal tile (the most key tiles) goes out before any lighter one
  const int nq = static_cast<int>(p.seq / kBr);
  const int qt = nq - 1 - static_cast<int>(blockIdx.y);
  const int64_t head = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;  // mma fragment row group / thread in group
  const int64_t hoff = head * p.seq * D * 2;  // bytes to this head
  const char* qg = p.q + hoff + (int64_t)qt * kBr * D * 2;
  const char* kg = p.k + hoff;
  const char* vg = p.v + hoff;
  const int ntiles = p.causal ? qt + 1 : nq;

  load_tile<D>(qs, qg);
  load_tile<D>(ks, kg);
  load_tile<D>(vs, vg);
  cp_async_commit();

  uint32_t qf[D / 16][4];  // this warp's 16 query rows as A fragments
  float o[D / 8][4];       // output accumulators: 16 rows x D
#pragma unroll
  for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY;  // running maxima (log2 domain), rows g and g + 8
  float l0 = 0.f, l1 = 0.f;              // this thread's share of the running sums

  for (int kt = 0; kt < ntiles; ++kt) {
    const int st = kt & 1;
    if (kt + 1 < ntiles) {  // next tile into the other stage (freed at the end of kt - 1)
      load_tile<D>(ks + (st ^ 1) * kBc * LD, kg + (int64_t)(kt + 1) * kBc * D * 2);
      load_tile<D>(vs + (st ^ 1) * kBc * LD, vg + (int64_t)(kt + 1) * kBc * D * 2);
    }
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    if (kt == 0) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        ldsm_x4(smem_addr(qs + (warp * 16 + (lane & 15)) * LD + kk * 16 + (lane >> 4) * 8),
                qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
    }
    const uint16_t* kb = ks + st * kBc * LD;
    const uint16_t* vb = vs + st * kBc * LD;

    // S = Q K^T for this warp's 16 rows and the tile's 64 keys (8 n-tiles)
    float s[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(smem_addr(kb + (np * 16 + (lane & 7) + ((lane >> 4) << 3)) * LD + kk * 16 +
                          ((lane >> 3) & 1) * 8),
                b0, b1, b2, b3);
        mma_bf16(s[2 * np], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b0, b1);
        mma_bf16(s[2 * np + 1], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b2, b3);
      }
    }
    // scale into the log2 domain; mask keys after the query on the diagonal tile
    const int r0 = warp * 16 + g;  // query row (in the tile) of s[.][0..1]; r0 + 8 of s[.][2..3]
    float tm0 = -INFINITY, tm1 = -INFINITY;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float x = s[n][e] * p.scale_log2;
        const int key = n * 8 + 2 * t + (e & 1);
        const int row = r0 + (e >> 1) * 8;
        if (p.causal && kt == qt && key > row) x = -INFINITY;
        s[n][e] = x;
      }
      tm0 = fmaxf(tm0, fmaxf(s[n][0], s[n][1]));
      tm1 = fmaxf(tm1, fmaxf(s[n][2], s[n][3]));
    }
    // the four threads of a group share a row: reduce the tile maxima there
    tm0 = fmaxf(tm0, __shfl_xor_sync(0xffffffffu, tm0, 1));
    tm0 = fmaxf(tm0, __shfl_xor_sync(0xffffffffu, tm0, 2));
    tm1 = fmaxf(tm1, __shfl_xor_sync(0xffffffffu, tm1, 1));
    tm1 = fmaxf(tm1, __shfl_xor_sync(0xffffffffu, tm1, 2));
    const float mn0 = fmaxf(m0, tm0), mn1 = fmaxf(m1, tm1);  // finite: key 0 is always seen
    const float a0 = ex2(m0 - mn0), a1 = ex2(m1 - mn1);     // 0 on the first tile
    m0 = mn0;
    m1 = mn1;
    l0 *= a0;
    l1 *= a1;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      o[n][0] *= a0;
      o[n][1] *= a0;
      o[n][2] *= a1;
      o[n][3] *= a1;
    }
    // probabilities, their row sums, and P as bf16 A fragments (k = 16 keys)
    uint32_t pf[4][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      const float p0 = ex2(s[n][0] - m0), p1 = ex2(s[n][1] - m0);
      const float p2 = ex2(s[n][2] - m1), p3 = ex2(s[n][3] - m1);
      l0 += p0 + p1;
      l1 += p2 + p3;
      const int ks16 = n >> 1, hi = n & 1;
      pf[ks16][hi * 2 + 0] = pack_bf16(p0, p1);  // rows g: a0a1 (n even) / a4a5 (n odd)
      pf[ks16][hi * 2 + 1] = pack_bf16(p2, p3);  // rows g + 8: a2a3 / a6a7
    }
    // O += P V: V tile rows are keys (k), columns d (n); ldmatrix.trans gives B
#pragma unroll
    for (int ks16 = 0; ks16 < 4; ++ks16) {
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(smem_addr(vb + (ks16 * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * LD + dp * 16 +
                            (lane >> 4) * 8),
                  b0, b1, b2, b3);
        mma_bf16(o[2 * dp], pf[ks16][0], pf[ks16][1], pf[ks16][2], pf[ks16][3], b0, b1);
        mma_bf16(o[2 * dp + 1], pf[ks16][0], pf[ks16][1], pf[ks16][2], pf[ks16][3], b2, b3);
      }
    }
    __syncthreads();  // every warp is done with stage st before it is refilled
  }
  cp_async_wait<0>();

  // row sums over the group, then O / l and lse
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const float inv0 = 1.f / l0, inv1 = 1.f / l1;
  const int64_t row0 = (int64_t)qt * kBr + warp * 16 + g;  // query index of rows g, g + 8
  char* og = p.o + hoff;
#pragma unroll
  for (int n = 0; n < D / 8; ++n) {
    const int col = n * 8 + 2 * t;
    *reinterpret_cast<uint32_t*>(og + (row0 * D + col) * 2) = pack_bf16(o[n][0] * inv0, o[n][1] * inv0);
    *reinterpret_cast<uint32_t*>(og + ((row0 + 8) * D + col) * 2) =
        pack_bf16(o[n][2] * inv1, o[n][3] * inv1);
  }
  if (p.lse != nullptr && t == 0) {
    constexpr float kLn2 = 0.6931471805599453f;
    p.lse[head * p.seq + row0] = (m0 + __log2f(l0)) * kLn2;
    p.lse[head * p.seq + row0 + 8] = (m1 + __log2f(l1)) * kLn2;
  }
}

}  // namespace

AttnKernel attn_fwd_kernel_for(int d) {
  constexpr int kSmem64 = (kBr + 4 * kBc) * (64 + kPad) * 2;
  constexpr int kSmem128 = (kBr + 4 * kBc) * (128 + kPad) * 2;
  if (d == 64) return AttnKernel{(const void*)attn_fwd_kernel<64>, kSmem64};
  if (d == 128) return AttnKernel{(const void*)attn_fwd_kernel<128>, kSmem128};
  return AttnKernel{nullptr, 0};
}

}  // namespace rr
