// k_attn.cu -- scaled dot-product attention forward on the online softmax
// ("Engineering a CUDA Machine Learning Framework from Scratch", sec. 6.4: the
// FlashAttention-style extension of the sec. 3.1 online normaliser; attention
// as defined by Vaswani et al. 2017, tiled as in Dao et al. 2022), with both
// products on the 5th-generation tensor cores.
//
// A softmax warpgroup of four warps owns 128 query rows of one head at a time;
// thread t owns query row t, which is TMEM lane t of every accumulator.  Per
// key tile (128 keys for d = 64, 64 for d = 128):
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
// in bf16 and lse = (m + log2 l) ln 2 in fp32.  Each CTA (one per SM) runs two
// such pipelines, each with its own two issuer warps (below).
//
// Loads are 3-D TMA boxes of [64 head-dim columns x 128 rows x 1 head] with
// 128-byte swizzle; rows past seq are filled with zeros, so seq needs only be a
// multiple of 64 (those keys are masked, those queries not stored).  O leaves
// through shared memory: each warp's 32 rows x 64 columns go into a staging box
// in the same swizzled layout and out by a TMA store of whole lines.  Every
// mbarrier wait is bounded (RR_ERR_DEVICE_TIMEOUT in the device error word);
// the tensor memory is allocated by warp 0 and always released.
//
// Shapes: bf16 q, k, v, o of [bh][s][d], d = 64 or 128, s a multiple of 64,
// 16-byte aligned tensors (checked by the caller).
#include <algorithm>
#include <cstdint>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "rr_device.cuh"
#include "rr_kernels.h"

namespace rr {
namespace {

constexpr int kBM = 128;              // query rows per tile: MMA M, TMEM lanes
constexpr int kBoxBytes = kBM * 128;  // one Q box: 128 rows x 64 bf16 (128 bytes)

// Instruction descriptors (kind::f16): D fp32 (bits 4-5), A and B bf16 (bits
// 7-9, 10-12), B K-major or MN-major (bit 16), N >> 3 (bits 17-22), M >> 4
// (bits 24-28).  S = Q K^T: B K-major, N = the key tile.  O = P V: B MN-major
// (the head dimension is contiguous in V), N = D.
__host__ __device__ constexpr uint32_t attn_idesc(int m, int n, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn_major ? (1u << 16) : 0u) |
         ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

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
// 3-D TMA tile store map at {c0, c1, c2} <- [src] (this CTA's shared memory),
// committed as one bulk group of this thread; elements outside the tensor are
// not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int c0,
                                             int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(src))
      : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// This thread's bulk stores have read their shared memory (it may be
// overwritten) / have completed.
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// two floats as a bf16 pair, lo in the low half (round to nearest even)
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// 32 TMEM columns of this thread's lane, without waiting (tcgen05.wait::ld
// before the registers are used).
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t (&v)[32]) {
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
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// Bounded wait without asking to be suspended (the issuer reacts at once);
// after a wait gave up (dead) it returns immediately.
__device__ __forceinline__ void wait_spin(uint64_t* bar, uint32_t parity, bool& dead, int* err) {
  if (dead) return;
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if ((it & 255u) == 0 && global_timer_ns() - t0 > 1000000000ull) {
      atomicCAS(err, 0, 6);
      dead = true;
      return;
    }
  }
}

// Persistent CTAs (one per SM), each running two independent pipelines w =
// 0, 1: a softmax warpgroup (warps 4w .. 4w + 3; thread t owns query row t of
// the tile, TMEM lane t) and two issuer warps (lane 0 of each): warp 8 + w
// loads Q and K and issues S = Q K^T, warp 10 + w loads V and issues O += P V,
// so neither product waits behind the other's loads and barrier waits.
// Pipeline w owns TMEM columns [256 w,
// 256 w + 256): S [0, BN), NPB buffers of P (bf16 pairs, BN / 2 columns each)
// from BN, O [256 - D, 256) (head_dim 128: two P buffers in the 256 columns),
// and its own Q tile and two-stage rings of K and of V tiles in shared memory.
// The two pipelines interleave on the SM: one's softmax runs while the tensor
// cores work for the other.
// A pipeline works through query tiles (head, tile) in a zigzag of the list
// sorted heaviest first (causal: most key tiles first), so the pipelines of
// all SMs end together.  Its key tiles are numbered t = 0, 1, ... across its
// query tiles.  Issuers, per key tile t:
//   S(t + 1) = Q K(t + 1)^T as soon as the softmax has read S(t) (so it runs
//     during the softmax of t) -> bar_s; K(t + 2) then loads into the stage
//     S(t) has finished with;
//   once P(t) is written: O += P(t) V(t) -> bar_o[t % NPB]; V(t + 1) loads into
//     the stage O += P V of t - 1 has finished with.
//   The next query tile's Q loads once the current one's last S is done; its
//   first O += P V (which overwrites O) waits for the softmax to read O.
// Softmax, per key tile: [bar_s] read S -> bar_sfree; max, P = 2^(s - m),
// sums; [O += P V of t - NPB done] write P(t) into buffer t % NPB; [O += P V
// of t - 1 done, only when O is rescaled] O *= alpha -> bar_p[t % NPB]; after
// a query tile's last key tile: [its O += P V done] O / l, lse -> bar_ofree.
// With two P buffers the softmax of t does not wait for O += P V of t - 1, so
// it runs as soon as S(t) is there.
template <int D>
struct AttnPL {
  static constexpr int BN = D == 64 ? 128 : 64;        // keys per tile
  static constexpr int NS = 2;                         // K / V stages
  static constexpr int NPB = D == 128 ? 2 : 1;         // P buffers in TMEM
  static constexpr int kBoxes = D / 64;
  static constexpr int kQBytes = kBoxes * kBoxBytes;   // 128 rows
  static constexpr int kKVBox = BN * 128;              // one K or V box of BN rows
  static constexpr int kKVBytes = kBoxes * kKVBox;
  static constexpr int kPipe = kQBytes + NS * 2 * kKVBytes;  // smem of one pipeline
  static constexpr int kStageWarp = 32 * 128;          // O staging: 32 rows x 64 columns
  static constexpr int kOffStage = 2 * kPipe;          // 4 warps' boxes per pipeline
  static constexpr int kOffBar = kOffStage + 2 * 4 * kStageWarp;
  static constexpr int kSmem = kOffBar + 512 + 1024;
  static constexpr uint32_t kColS = 0, kColP = BN, kColO = 256 - D;
  static constexpr uint32_t kIdescS = attn_idesc(kBM, BN, false);
  static constexpr uint32_t kIdescO = attn_idesc(kBM, D, true);
};

// The r-th query tile of pipeline slot `slot` among nslots: a zigzag over the
// list sorted by decreasing work (causal: tile nq - 1 of every head first),
// or -1 past the end.  Writes the head and query tile.
__device__ __forceinline__ bool attn_item(int r, int slot, int nslots, int bh, int nq, int& head,
                                          int& qt) {
  const int i = r * nslots + ((r & 1) ? nslots - 1 - slot : slot);
  if (i >= bh * nq) return false;
  qt = nq - 1 - i / bh;
  head = i % bh;
  return true;
}

template <int D>
__global__ void __launch_bounds__(384, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
                    const AttnParams p) {
  static_assert(D == 64 || D == 128, "head dimension 64 or 128");
  using C = AttnPL<D>;
  constexpr int BN = C::BN;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5;
  const int w = warp < 8 ? warp >> 2 : (warp - 8) & 1;  // this thread's pipeline
  unsigned char* pipe = smem + w * C::kPipe;
  unsigned char* sq = pipe;
  auto stage_k = [&](int s) { return pipe + C::kQBytes + (2 * s) * C::kKVBytes; };
  auto stage_v = [&](int s) { return pipe + C::kQBytes + (2 * s + 1) * C::kKVBytes; };
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar) + w * 16;
  uint64_t* bar_q = bars + 0;
  uint64_t* bar_s = bars + 1;
  uint64_t* bar_sfree = bars + 2;   // 128 arrivals
  uint64_t* bar_ofree = bars + 3;   // 128 arrivals
  uint64_t* bar_p = bars + 4;       // [NPB] P written, 128 arrivals
  uint64_t* bar_o = bars + 6;       // [NPB] O += P V done with the P buffer
  uint64_t* bar_kfull = bars + 8;   // [2] K tile landed
  uint64_t* bar_vfull = bars + 10;  // [2] V tile landed
  uint64_t* bar_kempty = bars + 12; // [2] S done with the K stage
  uint64_t* bar_vempty = bars + 14; // [2] O += P V done with the V stage
  uint32_t* tslot = reinterpret_cast<uint32_t*>(reinterpret_cast<uint64_t*>(smem + C::kOffBar) + 40);

  const int seq = static_cast<int>(p.seq);
  const int bh = static_cast<int>(p.bh);
  const int nq = (seq + kBM - 1) / kBM;
  const int slot = static_cast<int>(blockIdx.x) * 2 + w, nslots = 2 * static_cast<int>(gridDim.x);
  auto tiles_of = [&](int qt) {  // key tiles a query tile needs
    const int last_key = p.causal ? min(seq - 1, qt * kBM + kBM - 1) : seq - 1;
    return last_key / BN + 1;
  };

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tslot)),
                 "r"(512u)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if ((warp == 8 || warp == 9) && (tid & 31) == 0) {
    mbar_init(bar_q, 1);
    mbar_init(bar_s, 1);
    mbar_init(bar_sfree, 128);
    mbar_init(bar_ofree, 128);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_p[i], 128);
      mbar_init(&bar_o[i], 1);
      mbar_init(&bar_kfull[i], 1);
      mbar_init(&bar_vfull[i], 1);
      mbar_init(&bar_kempty[i], 1);
      mbar_init(&bar_vempty[i], 1);
    }
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tslot + 256u * w;  // this pipeline's columns
  bool dead = false;  // a wait gave up: no further waits (the kernel still ends)
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    if (!dead) dead = !mbar_wait_bounded(bar, parity, p.err);
  };

  if (warp >= 8) {
    // ------------------------------------------------------ the issuers
    if ((tid & 31) == 0) {
      // the pipeline's key tiles in order: (query tile r, tile j of it, head)
      struct Cur {
        int r, j, n, head, qt;
        bool ok;
      };
      auto first = [&]() {
        Cur c{0, 0, 0, 0, 0, false};
        c.ok = attn_item(0, slot, nslots, bh, nq, c.head, c.qt);
        if (c.ok) c.n = tiles_of(c.qt);
        return c;
      };
      auto advance = [&](Cur& c) {
        if (++c.j == c.n) {
          c.j = 0;
          c.ok = attn_item(++c.r, slot, nslots, bh, nq, c.head, c.qt);
          if (c.ok) c.n = tiles_of(c.qt);
        }
      };
      Cur kc = first(), vc = first();  // next K / V tile to load
      int kt = 0, vt = 0;              // their numbers
      auto load_k = [&]() {
        const int s = kt & 1;
        mbar_arrive_expect_tx(&bar_kfull[s], C::kKVBytes);
#pragma unroll
        for (int b = 0; b < C::kBoxes; ++b)
          tma_load_3d(stage_k(s) + b * C::kKVBox, &tk, 64 * b, kc.j * BN, kc.head, &bar_kfull[s]);
        ++kt;
        advance(kc);
      };
      auto load_v = [&]() {
        const int s = vt & 1;
        mbar_arrive_expect_tx(&bar_vfull[s], C::kKVBytes);
#pragma unroll
        for (int b = 0; b < C::kBoxes; ++b)
          tma_load_3d(stage_v(s) + b * C::kKVBox, &tv, 64 * b, vc.j * BN, vc.head, &bar_vfull[s]);
        ++vt;
        advance(vc);
      };
      auto load_q = [&](const Cur& c) {
        mbar_arrive_expect_tx(bar_q, C::kQBytes);
#pragma unroll
        for (int b = 0; b < C::kBoxes; ++b)
          tma_load_3d(sq + b * kBoxBytes, &tq, 64 * b, c.qt * kBM, c.head, bar_q);
      };
      auto issue_s = [&](int t) {  // S = Q K^T of key tile t
        const uint32_t q_addr = smem_addr(sq), k_addr = smem_addr(stage_k(t & 1));
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t qo = (uint32_t)((kk >> 2) * kBoxBytes + (kk & 3) * 32);
          const uint32_t ko = (uint32_t)((kk >> 2) * C::kKVBox + (kk & 3) * 32);
          mma_ss(tm + C::kColS, sw128_desc(q_addr + qo, 16, 1024),
                 sw128_desc(k_addr + ko, 16, 1024), C::kIdescS, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar_s);
        mma_commit(&bar_kempty[t & 1]);
      };
      auto issue_pv = [&](int t, bool first_of_tile) {  // O (+)= P V of key tile t
        const uint32_t v_addr = smem_addr(stage_v(t & 1));
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts(tm + C::kColO, tm + C::kColP + (t % C::NPB) * (BN / 2) + 8 * kk,
                 sw128_desc(v_addr + kk * 2048, C::kKVBox, 1024), C::kIdescO,
                 (!first_of_tile || kk > 0) ? 1u : 0u);
        mma_commit(&bar_o[t % C::NPB]);
        mma_commit(&bar_vempty[t & 1]);
      };
      int qr = 0;  // the last query tile whose Q has been loaded
      // After S of key tile c (number t): if it is the last of its query tile,
      // the next query tile's Q loads as soon as that S is done.
      auto after_s = [&](const Cur& c, int t) {
        if (c.j != c.n - 1) return;
        Cur q2{c.r + 1, 0, 0, 0, 0, false};
        q2.ok = attn_item(q2.r, slot, nslots, bh, nq, q2.head, q2.qt);
        if (!q2.ok) return;
        wait_spin(bar_s, (uint32_t)(t & 1), dead, p.err);
        load_q(q2);
        qr = q2.r;
      };
      if (warp >= 10) {
        // warp 10 + w: V loads and O += P V.  O += P(t) V(t) as soon as the
        // softmax has written P(t) (the first of a query tile, which
        // overwrites O, once the softmax has read O); V(t + 1) loads into
        // the stage O += P V of t - 1 used once that is done
        Cur c = first();
        if (c.ok) {
          load_v();
          if (vc.ok) load_v();
        }
        for (int t = 0; c.ok; ++t) {
          if (vc.ok && vt == t + 1 && t >= 1) {
            wait_spin(&bar_vempty[(t - 1) & 1], (uint32_t)(((t - 1) >> 1) & 1), dead, p.err);
            load_v();
          }
          if (c.j == 0 && c.r > 0) wait_spin(bar_ofree, (uint32_t)((c.r - 1) & 1), dead, p.err);
          wait_spin(&bar_p[t % C::NPB], (uint32_t)((t / C::NPB) & 1), dead, p.err);
          wait_spin(&bar_vfull[t & 1], (uint32_t)((t >> 1) & 1), dead, p.err);
          issue_pv(t, c.j == 0);
          advance(c);
        }
      } else {
        // warp 8 + w: Q / K loads and S = Q K^T
        Cur cur = first();  // key tile t
        if (cur.ok) {
          load_q(cur);
          load_k();
          if (kc.ok) load_k();
          wait_spin(bar_q, 0, dead, p.err);
          wait_spin(&bar_kfull[0], 0, dead, p.err);
          issue_s(0);
          after_s(cur, 0);
        }
        for (int t = 0; cur.ok; ++t) {
          Cur nxt = cur;
          advance(nxt);
          if (nxt.ok) {
            // S(t + 1) once the softmax has read S(t); a new query tile's Q
            // was loaded after the current one's last S
            wait_spin(bar_sfree, (uint32_t)(t & 1), dead, p.err);
            if (nxt.r != cur.r) {
              if (qr < nxt.r) {  // not reached: after_s loaded it
                load_q(nxt);
                qr = nxt.r;
              }
              wait_spin(bar_q, (uint32_t)(nxt.r & 1), dead, p.err);
            }
            wait_spin(&bar_kfull[(t + 1) & 1], (uint32_t)(((t + 1) >> 1) & 1), dead, p.err);
            issue_s(t + 1);
            after_s(nxt, t + 1);
            // K(t + 2) into the stage S(t) used
            if (kc.ok && kt == t + 2) {
              wait_spin(&bar_kempty[t & 1], (uint32_t)((t >> 1) & 1), dead, p.err);
              load_k();
            }
          }
          cur = nxt;
        }
      }
    }
  } else {
    // ------------------------------------------------ softmax warpgroup
    const int t_row = tid & 127;  // row in the tile, TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tm + lane_base + C::kColS;
    const uint32_t tO = tm + lane_base + C::kColO;
    const float sc = p.scale_log2;
    int t = 0;
    int head = 0, qt = 0;
    for (int r = 0; attn_item(r, slot, nslots, bh, nq, head, qt); ++r) {
      const int n = tiles_of(qt);
      const int q0 = qt * kBM, row = q0 + t_row;
      const int lim = p.causal ? min(row, seq - 1) : seq - 1;  // last visible key
      float m = -INFINITY, l = 0.f;  // running maximum (log2 domain) and sum
      for (int j = 0; j < n; ++j, ++t) {
        wait(bar_s, (uint32_t)(t & 1));
        tc_fence_after();
        uint32_t v[BN / 32][32];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) tmem_ld32_nowait(tS + 32 * c, v[c]);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(bar_sfree);  // S may take the next tile
        const int key0 = j * BN;
        // keys to mask: after the query (causal, diagonal tiles) or past the end
        if (p.causal ? (key0 + BN - 1 > q0) : (key0 + BN > seq)) {
#pragma unroll
          for (int c = 0; c < BN / 32; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (key0 + 32 * c + i > lim) v[c][i] = __float_as_uint(-INFINITY);
        }
        // the tile's row maximum on the raw scores (scale > 0 keeps the order);
        // eight independent chains, so the reduction is not one long chain
        float mx[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mx[k] = -INFINITY;
#pragma unroll
        for (int c = 0; c < BN / 32; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) mx[i & 7] = fmaxf(mx[i & 7], __uint_as_float(v[c][i]));
        const float mx0 = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        const float mx1 = fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]));
        // The running maximum m moves only when the tile's maximum exceeds it
        // by more than 8 (log2 domain): otherwise P = 2^(s - m) stays below
        // 2^8 and O, l keep their scale, so O is rarely rescaled.  (Finite
        // after the first tile: key 0 is visible to every row.)
        const float mt = fmaxf(mx0, mx1) * sc;
        const float m_new = mt > m + 8.f ? mt : m;
        const float alpha = ex2(m - m_new);  // 1 if m stays, 0 on the first tile
        // P = 2^(s sc - m): packed exponent FMAs, the sum in four chains
        float l0 = 0.f, l1 = 0.f, l2 = 0.f, l3 = 0.f;
        uint32_t pk[BN / 32][16];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c)
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            float t0, t1, t2, t3;
            fma2(t0, t1, __uint_as_float(v[c][i]), __uint_as_float(v[c][i + 1]), sc, sc, -m_new,
                 -m_new);
            fma2(t2, t3, __uint_as_float(v[c][i + 2]), __uint_as_float(v[c][i + 3]), sc, sc,
                 -m_new, -m_new);
            const float p0 = ex2(t0), p1 = ex2(t1), p2 = ex2(t2), p3 = ex2(t3);
            add2(l0, l1, l0, l1, p0, p1);
            add2(l2, l3, l2, l3, p2, p3);
            pk[c][i >> 1] = pack_bf16(p0, p1);
            pk[c][(i >> 1) + 1] = pack_bf16(p2, p3);
          }
        l = l * alpha + ((l0 + l1) + (l2 + l3));
        m = m_new;
        // P(t) goes into buffer t % NPB once O += P V of tile t - NPB is done
        // with it; O is rescaled only after O += P V of tile t - 1
        if (t >= C::NPB) {
          wait(&bar_o[t % C::NPB], (uint32_t)((t / C::NPB - 1) & 1));
          tc_fence_after();
        }
        const uint32_t tP = tm + lane_base + C::kColP + (t % C::NPB) * (BN / 2);
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) tmem_st16(tP + 16 * c, pk[c]);
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          if constexpr (C::NPB > 1) {
            wait(&bar_o[(t - 1) % C::NPB], (uint32_t)(((t - 1) / C::NPB) & 1));
            tc_fence_after();
          }
          uint32_t o[D / 32][32];  // every load issued before the one wait
#pragma unroll
          for (int c = 0; c < D / 32; ++c) tmem_ld32_nowait(tO + 32 * c, o[c]);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              float a0, a1;
              mul2(a0, a1, __uint_as_float(o[c][i]), __uint_as_float(o[c][i + 1]), alpha, alpha);
              o[c][i] = __float_as_uint(a0);
              o[c][i + 1] = __float_as_uint(a1);
            }
            tmem_st32(tO + 32 * c, o[c]);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bar_p[t % C::NPB]);
      }
      // O / l in bf16: each warp writes its 32 rows, 64 columns at a time,
      // into its staging box (the 128-byte swizzled layout of the tensor map)
      // and stores the box with one TMA store (whole 128-byte lines, where
      // stores of a row per thread would each touch 32 lines)
      wait(&bar_o[(t - 1) % C::NPB], (uint32_t)(((t - 1) / C::NPB) & 1));
      tc_fence_after();
      const float inv = 1.f / l;
      uint32_t o[D / 32][32];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) tmem_ld32_nowait(tO + 32 * c, o[c]);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(bar_ofree);  // O read: the next query tile may overwrite it
      {
        const int lane = tid & 31, wq = warp & 3;
        unsigned char* box = smem + C::kOffStage + (4 * w + wq) * C::kStageWarp;
        const bool in_seq = q0 + 32 * wq < seq;  // seq is a multiple of 64: all or none
#pragma unroll
        for (int b = 0; b < D / 64; ++b) {
          if (lane == 0) bulk_wait_read();  // the box's previous store has read it
          __syncwarp();
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
              const uint32_t* oc = o[2 * b + c2];
              const uint4 q4 = make_uint4(
                  pack_bf16(__uint_as_float(oc[i]) * inv, __uint_as_float(oc[i + 1]) * inv),
                  pack_bf16(__uint_as_float(oc[i + 2]) * inv, __uint_as_float(oc[i + 3]) * inv),
                  pack_bf16(__uint_as_float(oc[i + 4]) * inv, __uint_as_float(oc[i + 5]) * inv),
                  pack_bf16(__uint_as_float(oc[i + 6]) * inv, __uint_as_float(oc[i + 7]) * inv));
              const int ch = 4 * c2 + (i >> 3);  // 16-byte chunk of the 128-byte row
              *reinterpret_cast<uint4*>(box + lane * 128 + ((ch ^ (lane & 7)) << 4)) = q4;
            }
          fence_proxy_async_smem();  // the writes are visible to the TMA store
          __syncwarp();
          if (lane == 0 && in_seq) tma_store_3d(&to, box, 64 * b, q0 + 32 * wq, head);
        }
      }
      if (p.lse != nullptr && row < seq)
        p.lse[(int64_t)head * seq + row] = (m + __log2f(l)) * 0.6931471805599453f;
    }
    if ((tid & 31) == 0) bulk_wait_all();  // the staging boxes are read, O written
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(*tslot), "r"(512u)
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
  if (d == 64) return AttnKernel{(const void*)attn_fwd_kernel<64>, AttnPL<64>::kSmem};
  if (d == 128) return AttnKernel{(const void*)attn_fwd_kernel<128>, AttnPL<128>::kSmem};
  return AttnKernel{nullptr, 0};
}

const char* attn_fwd_launch(const AttnParams& p, int d, int sms, cudaStream_t stream) {
  const AttnKernel ak = attn_fwd_kernel_for(d);
  if (ak.fn == nullptr) return "head_dim must be 64 or 128";
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return "cuTensorMapEncodeTiled is not available from the driver";
  // [bh][seq][d] bf16 as a 3-D tensor (d innermost); 128-byte swizzled boxes
  // of 64 columns x rows x 1 head (Q: 128 rows, K / V: the key tile); rows
  // past seq read as zeros
  const int bn = d == 64 ? AttnPL<64>::BN : AttnPL<128>::BN;
  CUtensorMap maps[4];
  const char* ptrs[4] = {p.q, p.k, p.v, p.o};
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)p.seq, (cuuint64_t)p.bh};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)p.seq * d * 2};
  const cuuint32_t es[3] = {1, 1, 1};
  for (int i = 0; i < 4; ++i) {  // q, k, v loads; o stores of 32 rows
    const cuuint32_t box[3] = {64, (cuuint32_t)(i == 0 ? kBM : i == 3 ? 32 : bn), 1};
    if (encode(&maps[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<char*>(ptrs[i]), dims,
               strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return "tensor map encoding failed";
  }
  AttnParams pc = p;
  void* args[] = {&maps[0], &maps[1], &maps[2], &maps[3], &pc};
  // persistent: one CTA per SM (two pipelines each), fewer for small problems
  const int64_t items = p.bh * ((p.seq + kBM - 1) / kBM);
  const int64_t grid = std::min<int64_t>(sms, (items + 1) / 2);
  if (cudaLaunchKernel(ak.fn, dim3((unsigned)grid), dim3(384), args, (size_t)ak.smem, stream) !=
      cudaSuccess)
    return "launch failed";
  return nullptr;
}

}  // namespace rr
