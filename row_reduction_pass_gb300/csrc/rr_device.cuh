// rr_device.cuh -- device-side building blocks shared by the row kernels:
// storage types, 16-byte chunk loads / stores with ragged heads and tails,
// ordered butterfly reductions, and the bulk-copy (TMA) / mbarrier / cluster
// primitives written as inline PTX for sm_103a.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace rr {

constexpr int kF32 = 0;
constexpr int kBF16 = 1;

template <int DT> struct DType;
template <> struct DType<kF32> { static constexpr int E = 4; static constexpr int V = 4; };
template <> struct DType<kBF16> { static constexpr int E = 2; static constexpr int V = 8; };

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// 2^x on the special-function unit (MUFU.EX2, flushes subnormal results).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Elementwise maximum of two packed bf16 pairs (exact; -inf is neutral).
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Packed two-lane float32 arithmetic (one FMA-pipe instruction for two
// values; each lane is an IEEE round-to-nearest operation like its scalar form).
__device__ __forceinline__ void fma2(float& dx, float& dy, float ax, float ay, float bx, float by,
                                     float cx, float cy) {
  asm("{\n\t.reg .b64 a, b, c, d;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
      "fma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(dx), "=f"(dy)
      : "f"(ax), "f"(ay), "f"(bx), "f"(by), "f"(cx), "f"(cy));
}
__device__ __forceinline__ void add2(float& dx, float& dy, float ax, float ay, float bx, float by) {
  asm("{\n\t.reg .b64 a, b, d;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "add.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(dx), "=f"(dy)
      : "f"(ax), "f"(ay), "f"(bx), "f"(by));
}
__device__ __forceinline__ void mul2(float& dx, float& dy, float ax, float ay, float bx, float by) {
  asm("{\n\t.reg .b64 a, b, d;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "mul.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(dx), "=f"(dy)
      : "f"(ax), "f"(ay), "f"(bx), "f"(by));
}

// ---------------------------------------------------------------- storage ---

__device__ __forceinline__ uint32_t word_of(const uint4& c, int k) {
  return k == 0 ? c.x : k == 1 ? c.y : k == 2 ? c.z : c.w;
}
__device__ __forceinline__ void set_word(uint4& c, int k, uint32_t w) {
  if (k == 0) c.x = w; else if (k == 1) c.y = w; else if (k == 2) c.z = w; else c.w = w;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h) { return __uint_as_float(h << 16); }

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  uint16_t h;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(f));
  return h;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Element v of a 16-byte chunk holding V values of type DT.
template <int DT> __device__ __forceinline__ float chunk_get(const uint4& c, int v);
template <> __device__ __forceinline__ float chunk_get<kF32>(const uint4& c, int v) {
  return __uint_as_float(word_of(c, v));
}
template <> __device__ __forceinline__ float chunk_get<kBF16>(const uint4& c, int v) {
  uint32_t w = word_of(c, v >> 1);
  return __uint_as_float((v & 1) ? (w & 0xffff0000u) : (w << 16));
}

// A chunk filled with one value (used for the ragged positions of a row).
template <int DT> __device__ __forceinline__ uint4 chunk_fill(float f);
template <> __device__ __forceinline__ uint4 chunk_fill<kF32>(float f) {
  uint32_t u = __float_as_uint(f);
  return make_uint4(u, u, u, u);
}
template <> __device__ __forceinline__ uint4 chunk_fill<kBF16>(float f) {
  uint32_t h = f32_to_bf16_bits(f);
  uint32_t u = h | (h << 16);
  return make_uint4(u, u, u, u);
}

template <int DT> __device__ __forceinline__ void chunk_set_bits(uint4& c, int v, uint32_t bits);
template <> __device__ __forceinline__ void chunk_set_bits<kF32>(uint4& c, int v, uint32_t bits) {
  set_word(c, v, bits);
}
template <> __device__ __forceinline__ void chunk_set_bits<kBF16>(uint4& c, int v, uint32_t bits) {
  uint32_t w = word_of(c, v >> 1);
  w = (v & 1) ? ((w & 0x0000ffffu) | (bits << 16)) : ((w & 0xffff0000u) | (bits & 0xffffu));
  set_word(c, v >> 1, w);
}

// Scalar element access at a byte address (streaming cache hints).
template <int DT> __device__ __forceinline__ uint32_t ld_elem_bits(const char* p);
template <> __device__ __forceinline__ uint32_t ld_elem_bits<kF32>(const char* p) {
  return __ldcs(reinterpret_cast<const unsigned int*>(p));
}
template <> __device__ __forceinline__ uint32_t ld_elem_bits<kBF16>(const char* p) {
  return __ldcs(reinterpret_cast<const unsigned short*>(p));
}
template <int DT> __device__ __forceinline__ float bits_to_f32(uint32_t b);
template <> __device__ __forceinline__ float bits_to_f32<kF32>(uint32_t b) { return __uint_as_float(b); }
template <> __device__ __forceinline__ float bits_to_f32<kBF16>(uint32_t b) { return bf16_bits_to_f32(b); }

template <int DT> __device__ __forceinline__ float ld_elem(const char* p) {
  return bits_to_f32<DT>(ld_elem_bits<DT>(p));
}
// Cached (L1) scalar load for small per-column vectors reused by every row.
template <int DT> __device__ __forceinline__ float ld_elem_cached(const char* p);
template <> __device__ __forceinline__ float ld_elem_cached<kF32>(const char* p) {
  return __ldg(reinterpret_cast<const float*>(p));
}
template <> __device__ __forceinline__ float ld_elem_cached<kBF16>(const char* p) {
  return bf16_bits_to_f32(__ldg(reinterpret_cast<const unsigned short*>(p)));
}
template <int DT> __device__ __forceinline__ float ld_smem_elem(const char* p);
template <> __device__ __forceinline__ float ld_smem_elem<kF32>(const char* p) {
  return *reinterpret_cast<const float*>(p);
}
template <> __device__ __forceinline__ float ld_smem_elem<kBF16>(const char* p) {
  return bf16_bits_to_f32(*reinterpret_cast<const unsigned short*>(p));
}

template <int DT> __device__ __forceinline__ void st_elem(char* p, float f);
template <> __device__ __forceinline__ void st_elem<kF32>(char* p, float f) {
  __stcs(reinterpret_cast<float*>(p), f);
}
template <> __device__ __forceinline__ void st_elem<kBF16>(char* p, float f) {
  __stcs(reinterpret_cast<unsigned short*>(p), f32_to_bf16_bits(f));
}

// Pack V floats into a chunk of DT.
template <int DT> __device__ __forceinline__ uint4 chunk_pack(const float* f);
template <> __device__ __forceinline__ uint4 chunk_pack<kF32>(const float* f) {
  return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                    __float_as_uint(f[3]));
}
template <> __device__ __forceinline__ uint4 chunk_pack<kBF16>(const float* f) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

__device__ __forceinline__ uint4 ld_chunk_stream(const char* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ uint4 ld_chunk_cached(const char* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void st_chunk_stream(char* p, uint4 v) {
  __stcs(reinterpret_cast<uint4*>(p), v);
}

// --- 16-byte accesses at addresses that are element-aligned but not 16-byte
// aligned (rows whose start is not 16-byte aligned, read in column-aligned
// chunks).  h = address % 16 (a multiple of the element size).

// Bytes [h, h + 16) of the 32-byte pair lo:hi.
__device__ __forceinline__ uint4 funnel16(const uint4& lo, const uint4& hi, int h) {
  const int sh = (h & 3) * 8;
  uint32_t a0, a1, a2, a3, a4;
  switch (h >> 2) {
    case 0: a0 = lo.x; a1 = lo.y; a2 = lo.z; a3 = lo.w; a4 = hi.x; break;
    case 1: a0 = lo.y; a1 = lo.z; a2 = lo.w; a3 = hi.x; a4 = hi.y; break;
    case 2: a0 = lo.z; a1 = lo.w; a2 = hi.x; a3 = hi.y; a4 = hi.z; break;
    default: a0 = lo.w; a1 = hi.x; a2 = hi.y; a3 = hi.z; a4 = hi.w; break;
  }
  return make_uint4(__funnelshift_r(a0, a1, sh), __funnelshift_r(a1, a2, sh),
                    __funnelshift_r(a2, a3, sh), __funnelshift_r(a3, a4, sh));
}

// Loads [p, p + 16) through the two aligned 16-byte chunks that hold it (read
// through L1, where the neighbouring lane's load of the same chunk hits).  The
// caller guarantees both aligned chunks lie inside the allocation.
__device__ __forceinline__ uint4 ld16_split(const char* p) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  const uint4* b = reinterpret_cast<const uint4*>(a & ~uintptr_t(15));
  return funnel16(__ldg(b), __ldg(b + 1), static_cast<int>(a & 15));
}

__device__ __forceinline__ void st_b16(char* p, uint32_t v) {
  asm volatile("st.global.cs.b16 [%0], %1;" ::"l"(p), "h"(static_cast<unsigned short>(v)) : "memory");
}
__device__ __forceinline__ void st_b32(char* p, uint32_t v) {
  asm volatile("st.global.cs.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_v2(char* p, uint32_t a, uint32_t b) {
  asm volatile("st.global.cs.v2.b32 [%0], {%1, %2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}

// Stores the 16 bytes v at p (p % 16 != 0, p % 2 == 0) as aligned pieces.
__device__ __forceinline__ void st16_split(char* p, const uint4& v) {
  const int h = static_cast<int>(reinterpret_cast<uintptr_t>(p) & 15);
  if ((h & 3) == 0) {
    if (h == 8) {
      st_v2(p, v.x, v.y);
      st_v2(p + 8, v.z, v.w);
    } else {  // h = 4 or 12: p + 4 is 8-byte aligned
      st_b32(p, v.x);
      st_v2(p + 4, v.y, v.z);
      st_b32(p + 12, v.w);
    }
  } else {  // h = 2 mod 4: the middle 12 bytes are v shifted by 16 bits
    const uint32_t u0 = __funnelshift_r(v.x, v.y, 16);
    const uint32_t u1 = __funnelshift_r(v.y, v.z, 16);
    const uint32_t u2 = __funnelshift_r(v.z, v.w, 16);
    st_b16(p, v.x & 0xffffu);
    if ((reinterpret_cast<uintptr_t>(p + 2) & 7) == 0) {
      st_v2(p + 2, u0, u1);
      st_b32(p + 10, u2);
    } else {
      st_b32(p + 2, u0);
      st_v2(p + 6, u1, u2);
    }
    st_b16(p + 14, v.w >> 16);
  }
}

// ------------------------------------------------------------- reductions ---

// Ordered butterfly over the lanes of a G-lane group (G a power of two <= 32):
// at each level the lane whose bit is clear passes its own value first, so both
// partners evaluate merge(lower, upper) identically and every lane of the group
// ends with the same bits.  S provides: static S shfl(const S&, int off).
template <class S, class M, int G>
__device__ __forceinline__ S group_reduce(S v, M merge) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = G / 2; off >= 1; off >>= 1) {
    S o = S::shfl_xor(v, off);
    v = (lane & off) ? merge(o, v) : merge(v, o);
  }
  return v;
}

// ------------------------------------------------- per-thread async copies --
// 16-byte global -> shared copies issued by one thread for itself (both
// addresses 16-byte aligned), grouped with commit and waited for by count; the
// issuing thread may read its own slots once the wait returns.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
               "l"(gsrc)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ------------------------------------------------- bulk copy and barriers ---

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
// One-dimensional bulk copy global -> this CTA's shared memory, completing
// `bytes` transaction bytes on `bar`.  dst, src 16-byte aligned; bytes % 16 == 0.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
// Arrival on an mbarrier of a CTA of this cluster (address from mapa), with
// release at cluster scope: this thread's earlier writes (to that CTA's shared
// memory, say) are visible to a thread that then sees the phase complete with
// a cluster-scope acquire.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cl_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cl_addr)
               : "memory");
}
__device__ __forceinline__ void st_cluster_f32x4(uint32_t cl_addr, float a, float b, float c,
                                                 float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(cl_addr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}
// try_wait with acquire at cluster scope (arrivals from other CTAs of the
// cluster).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait on an mbarrier phase: gives up after limit_ns of wall time
// (~1 s by default) and records RR_ERR_DEVICE_TIMEOUT (6) in *err instead of
// spinning forever.  The loop itself is bounded as well (2^32 polls), in case
// the global timer does not advance.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, int* err,
                                                  uint64_t limit_ns = 1000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  // plain polls: a suspend-time hint here slowed the engine's staged softmax
  // backward on 16384 x 50304 bf16 rows from 1.02 to 1.31 ms
  for (uint32_t it = 0; it != 0xffffffffu; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) break;
  }
  atomicCAS(err, 0, 6);
  return false;
}

// The same bounded wait for a phase completed by arrivals from other CTAs of
// the cluster (cluster-scope acquire).
__device__ __forceinline__ bool mbar_wait_bounded_cluster(uint64_t* bar, uint32_t parity, int* err,
                                                          uint64_t limit_ns = 1000000000ull) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0; it != 0xffffffffu; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) break;
  }
  atomicCAS(err, 0, 6);
  return false;
}

// Cluster primitives (distributed shared memory, no multicast).
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nrank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t map_to_rank(const void* local_smem, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_addr(local_smem)), "r"(rank));
  return out;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// Named barrier over `count` threads (ids 1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_bar(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

}  // namespace rr
