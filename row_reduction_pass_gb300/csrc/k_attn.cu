// k_attn.cu -- scaled dot-product attention forward on the online softmax
// ("Engineering a CUDA Machine Learning Framework from Scratch", sec. 6.4: the
// FlashAttention-style extension of the sec. 3.1 online normaliser; attention
// as defined by Vaswani et al. 2017, tiled as in Dao et al. 2022), with both
// products on the 5th-generation tensor cores.
//
// One CTA of four warps owns 128 query rows of one head; thread t owns query
// row t, which is TMEM lane t of every accumulator.  Per key tile of 128 keys:
//   1. S = Q K^T: tcgen05.mma (bf16 in, fp32 accumulate) of the Q tile and the
//      K tile, both read from shared memory (128-byte swizzled, K-major, loaded
//      by TMA), into 128 TMEM columns; issued by one thread, completion
//      tracked on an mbarrier by tcgen05.commit.
//   2. Each thread reads its row of S from TMEM (tcgen05.ld), scales it into
//      the log2 domain, masks keys after its query (causal) or past the end,
//      and updates its running maximum m and sum l of the online softmax; the
//      probabilities 2^(s - m) go back to TMEM as bf16 (tcgen05.st), and the
//      output accumulator O is rescaled in TMEM by 2^(m_old - m_new).
//   3. O += P V: tcgen05.mma with A = P read from TMEM and B = the V tile from
//      shared memory (MN-major: the head dimension is contiguous).
// K / V tiles are double-buffered: the tile after next is loaded once the
// product that last read its stage has completed.  At the end O / l is stored
// in bf16 and lse = (m + log2 l) ln 2 in fp32.
//
// Loads are 3-D TMA boxes of [64 head-dim columns x 128 rows x 1 head] with
// 128-byte swizzle; rows past seq are filled with zeros, so seq needs only be a
// multiple of 64 (those keys are masked, those queries not stored).  Every
// mbarrier wait is bounded (RR_ERR_DEVICE_TIMEOUT in the device error word);
// the tensor memory is allocated by warp 0 and always released.
//
// Shapes: bf16 q, k, v, o of [bh][s][d], d = 64 or 128, s a multiple of 64,
// 16-byte aligned tensors (checked by the caller).
#include <cstdint>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "rr_device.cuh"
#include "rr_kernels.h"

namespace rr {
namespace {

constexpr int kBM = 128;          // query rows per CTA: MMA M, TMEM lanes
constexpr int kBN = 128;          // keys per tile: N of S = Q K^T, K of O = P V
constexpr int kBoxBytes = kBM * 128;  // one TMA box: 128 rows x 64 bf16 (128 bytes)

template <int D>
struct AttnCfg {
  static constexpr int kBoxes = D / 64;                 // boxes per Q / K / V tile
  static constexpr int kTile = kBoxes * kBoxBytes;      // bytes of a Q, K or V tile
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kTile;                  // [2 stages][K, V]
  static constexpr int kOffBar = kTile + 4 * kTile;     // mbarriers and the TMEM address
  static constexpr int kSmem = kOffBar + 128 + 1024;    // + slack for 1024-byte alignment
  // TMEM columns: S [0, 128), P (bf16 pairs) [128, 192), O [kColO, kColO + D)
  static constexpr uint32_t kCols = D == 64 ? 256 : 512;
  static constexpr uint32_t kColS = 0, kColP = 128, kColO = D == 64 ? 192 : 256;
  // instruction descriptors (kind::f16): D fp32, A and B bf16, M = 128;
  // S: B K-major, N = 128.  O: B MN-major (bit 16), N = D.
  static constexpr uint32_t kIdescS =
      (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
  static constexpr uint32_t kIdescO = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) |
                                      ((uint32_t)(D >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
};

// Shared-memory matrix descriptor, 128-byte swizzle: start address, leading
// and stride byte offsets (16-byte units), the fixed 0b001 at bits 46-48.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3ffff) >> 4) | ((uint64_t)((lbo >> 4) & 0x3fff) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3fff) << 32) | (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem desc] * B[smem desc]
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc]
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                       uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// The mbarrier completes one arrival once every earlier tcgen05 operation of
// this thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}
// 32 consecutive TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
      "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
      "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// 3-D TMA tile load [dst] <- map at {c0, c1, c2}, completing bytes on bar.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
      : "memory");
}
// two floats as a bf16 pair, lo in the low half (round to nearest even)
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

template <int D>
__global__ void __launch_bounds__(128, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const AttnParams p) {
  static_assert(D == 64 || D == 128, "head dimension 64 or 128");
  using C = AttnCfg<D>;
  extern __shared__ unsigned char smem_raw[];
  // 128-byte swizzled tiles want 1024-byte alignment
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* sq = smem + C::kOffQ;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* bar_q = bars + 0;
  uint64_t* bar_full = bars + 1;  // [2]: K / V tile landed in the stage
  uint64_t* bar_s = bars + 3;     // S = Q K^T done
  uint64_t* bar_o = bars + 4;     // O += P V done
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 8);
  auto stage_k = [&](int s) { return smem + C::kOffKV + (2 * s) * C::kTile; };
  auto stage_v = [&](int s) { return smem + C::kOffKV + (2 * s + 1) * C::kTile; };

  const int tid = threadIdx.x, warp = tid >> 5;
  const int seq = static_cast<int>(p.seq);
  const int head = static_cast<int>(blockIdx.x);
  // grid (heads, query tiles): blocks are dispatched x fastest, so every head's
  // heaviest causal tile (the most key tiles) goes out before any lighter one
  const int qt = static_cast<int>(gridDim.y) - 1 - static_cast<int>(blockIdx.y);
  const int q0 = qt * kBM;
  const int last_key = p.causal ? min(seq - 1, q0 + kBM - 1) : seq - 1;
  const int nkv = last_key / kBN + 1;

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tslot)),
                 "r"(C::kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    for (int i = 0; i < 5; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;  // this warp's TMEM lanes
  const uint32_t tS = tmem + lane_base + C::kColS;
  const uint32_t tP = tmem + lane_base + C::kColP;
  const uint32_t tO = tmem + lane_base + C::kColO;

  auto issue_kv = [&](int j) {  // key tile j into stage j & 1 (thread 0)
    const int s = j & 1;
    mbar_arrive_expect_tx(&bar_full[s], 2 * C::kTile);
#pragma unroll
    for (int b = 0; b < C::kBoxes; ++b) {
      tma_load_3d(stage_k(s) + b * kBoxBytes, &tk, 64 * b, j * kBN, head, &bar_full[s]);
      tma_load_3d(stage_v(s) + b * kBoxBytes, &tv, 64 * b, j * kBN, head, &bar_full[s]);
    }
  };
  if (tid == 0) {
    mbar_arrive_expect_tx(bar_q, C::kTile);
#pragma unroll
    for (int b = 0; b < C::kBoxes; ++b) tma_load_3d(sq + b * kBoxBytes, &tq, 64 * b, q0, head, bar_q);
    issue_kv(0);
    if (nkv > 1) issue_kv(1);
  }

  const int row = q0 + tid;   // this thread's query
  float m = -INFINITY, l = 0.f;  // running maximum (log2 domain) and sum
  bool dead = false;             // a wait gave up: no further waits (the kernel still ends)
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    if (!dead) dead = !mbar_wait_bounded(bar, parity, p.err);
  };
  const uint32_t q_addr = smem_addr(sq);

  for (int j = 0; j < nkv; ++j) {
    const int s = j & 1;
    if (tid == 0) {
      wait(&bar_full[s], (uint32_t)((j >> 1) & 1));
      if (j == 0) wait(bar_q, 0);
      tc_fence_after();
      const uint32_t k_addr = smem_addr(stage_k(s));
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        // K-step kk: box kk / 4, 32-byte column block kk % 4 within the 128-byte swizzle row
        const uint32_t off = (uint32_t)((kk >> 2) * kBoxBytes + (kk & 3) * 32);
        mma_ss(tmem + C::kColS, sw128_desc(q_addr + off, 16, 1024),
               sw128_desc(k_addr + off, 16, 1024), C::kIdescS, kk > 0 ? 1u : 0u);
      }
      mma_commit(bar_s);
      // the stage of tile j - 1 is free once O += P V of tile j - 1 is done:
      // tile j + 1 goes there (tiles 0 and 1 were loaded up front)
      if (j >= 1 && j + 1 < nkv) {
        wait(bar_o, (uint32_t)((j - 1) & 1));
        issue_kv(j + 1);
      }
    }
    wait(bar_s, (uint32_t)(j & 1));  // also covers O += P V of tile j - 1 (committed earlier)
    tc_fence_after();

    // keys of this tile to mask: after the query (causal, diagonal tile) or past the end
    const int key0 = j * kBN;
    const bool need_mask = p.causal ? (key0 + kBN - 1 > q0) : (key0 + kBN > seq);
    const int lim = p.causal ? min(row, seq - 1) : seq - 1;  // last visible key
    // 1. the tile's row maximum (log2 domain)
    float mx = -INFINITY;
#pragma unroll
    for (int c = 0; c < kBN / 32; ++c) {
      uint32_t v[32];
      tmem_ld32(tS + 32 * c, v);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        float x = __uint_as_float(v[i]) * p.scale_log2;
        if (need_mask && key0 + 32 * c + i > lim) x = -INFINITY;
        mx = fmaxf(mx, x);
      }
    }
    const float m_new = fmaxf(m, mx);  // finite: key 0 is visible to every row
    const float alpha = ex2(m - m_new);  // 0 on the first tile
    // 2. P = 2^(s - m_new) as bf16 into TMEM, the row sum from the fp32 values
    float ls = 0.f;
#pragma unroll
    for (int c = 0; c < kBN / 32; ++c) {
      uint32_t v[32];
      tmem_ld32(tS + 32 * c, v);
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        float x0 = __uint_as_float(v[i]) * p.scale_log2;
        float x1 = __uint_as_float(v[i + 1]) * p.scale_log2;
        if (need_mask && key0 + 32 * c + i > lim) x0 = -INFINITY;
        if (need_mask && key0 + 32 * c + i + 1 > lim) x1 = -INFINITY;
        const float p0 = ex2(x0 - m_new), p1 = ex2(x1 - m_new);
        ls += p0 + p1;
        pk[i >> 1] = pack_bf16(p0, p1);
      }
      tmem_st16(tP + 16 * c, pk);
    }
    l = l * alpha + ls;
    m = m_new;
    // 3. O *= alpha (O += P V of tile j - 1 is complete: see the wait above)
    if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tO + 32 * c, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
        tmem_st32(tO + 32 * c, v);
      }
    }
    tmem_st_wait();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      const uint32_t v_addr = smem_addr(stage_v(s));
#pragma unroll
      for (int kk = 0; kk < kBN / 16; ++kk) {
        // 16 keys per step: two 8-row groups of the swizzled V tile (1024 bytes
        // each); the head dimension's 64-column blocks are kBoxBytes apart
        mma_ts(tmem + C::kColO, tmem + C::kColP + 8 * kk,
               sw128_desc(v_addr + kk * 2048, kBoxBytes, 1024), C::kIdescO,
               (j > 0 || kk > 0) ? 1u : 0u);
      }
      mma_commit(bar_o);
    }
  }

  // O / l in bf16 and lse, for the rows inside the sequence
  wait(bar_o, (uint32_t)((nkv - 1) & 1));
  tc_fence_after();
  const float inv = 1.f / l;
  char* orow = p.o + ((int64_t)head * seq + row) * D * 2;
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    uint32_t v[32];
    tmem_ld32(tO + 32 * c, v);
    if (row < seq) {
#pragma unroll
      for (int i = 0; i < 32; i += 8) {
        const uint4 w = make_uint4(
            pack_bf16(__uint_as_float(v[i]) * inv, __uint_as_float(v[i + 1]) * inv),
            pack_bf16(__uint_as_float(v[i + 2]) * inv, __uint_as_float(v[i + 3]) * inv),
            pack_bf16(__uint_as_float(v[i + 4]) * inv, __uint_as_float(v[i + 5]) * inv),
            pack_bf16(__uint_as_float(v[i + 6]) * inv, __uint_as_float(v[i + 7]) * inv));
        *reinterpret_cast<uint4*>(orow + (32 * c + i) * 2) = w;
      }
    }
  }
  if (p.lse != nullptr && row < seq)
    p.lse[(int64_t)head * seq + row] = (m + __log2f(l)) * 0.6931471805599453f;

  tc_fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(C::kCols)
                 : "memory");
}

// cuTensorMapEncodeTiled from the driver (resolved once; the library links
// only the runtime).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

}  // namespace

AttnKernel attn_fwd_kernel_for(int d) {
  if (d == 64) return AttnKernel{(const void*)attn_fwd_kernel<64>, AttnCfg<64>::kSmem};
  if (d == 128) return AttnKernel{(const void*)attn_fwd_kernel<128>, AttnCfg<128>::kSmem};
  return AttnKernel{nullptr, 0};
}

const char* attn_fwd_launch(const AttnParams& p, int64_t bh, int d, cudaStream_t stream) {
  const AttnKernel ak = attn_fwd_kernel_for(d);
  if (ak.fn == nullptr) return "head_dim must be 64 or 128";
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return "cuTensorMapEncodeTiled is not available from the driver";
  // [bh][seq][d] bf16 as a 3-D tensor (d innermost); boxes of 64 x 128 x 1
  // with 128-byte swizzle; rows past seq read as zeros
  CUtensorMap maps[3];
  const char* ptrs[3] = {p.q, p.k, p.v};
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)p.seq, (cuuint64_t)bh};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)p.seq * d * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)kBM, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  for (int i = 0; i < 3; ++i) {
    if (encode(&maps[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<char*>(ptrs[i]), dims,
               strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return "tensor map encoding failed";
  }
  AttnParams pc = p;
  void* args[] = {&maps[0], &maps[1], &maps[2], &pc};
  const dim3 grid((unsigned)bh, (unsigned)((p.seq + kBM - 1) / kBM));
  if (cudaLaunchKernel(ak.fn, grid, dim3(128), args, (size_t)ak.smem, stream) != cudaSuccess)
    return "launch failed";
  return nullptr;
}

}  // namespace rr
