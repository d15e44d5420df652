// rr_kernels.h -- host-side view of the compiled kernel variants.
#pragma once

#include <cstdint>
#include <cuda_runtime_api.h>

namespace rr {

constexpr int kNumDirectG = 11;  // row groups of 1, 2, 4, ..., 1024 threads

// The variants of one operation for one storage type.  Index [m] is the mode:
// 0 = 16-byte chunks, 1 = single elements.
struct KernelSet {
  const void* direct[2][kNumDirectG];
  const void* staged[2];
  int nq_direct[2];
  int nq_staged[2];
  int maxt_direct;
  int maxt_staged;
};

// Row-group LayerNorm kernels (rr_ln.cuh).  Index [m][i]: m = 0 chunk mode
// with every row start 16-byte aligned, 1 chunk mode with any element
// alignment, 2 element mode; G = 2^i threads per row group.
constexpr int kNumLnG = 11;
struct LnKernelSet {
  const void* k[3][kNumLnG];
  int nq[3];  // chunks (elements in element mode) per thread
  // One chunk per thread, G <= 32 (backward: fewer registers, so more warps
  // per SM for short rows); null where not built.
  const void* k1[3][kNumLnG];
  // Forward rows split over a thread-block cluster: one group of 256 / 512 /
  // 1024 threads per block with nq chunks per thread, and [3] a 256-thread
  // group with 2 * nq; null where not built.
  const void* kc[3][4];
  // Chunk modes, rows of many chunks: nqd (> nq) chunks per thread so a row
  // needs fewer threads and each pays the per-row reductions over more data;
  // G >= 64 only, null where not built.
  const void* kd[2][kNumLnG];
  int nqd;
};

// Phase-aligned LayerNorm / RMSNorm kernels for long rows (rr_lnx.cuh):
// [rms][cluster]; nq_* chunks per thread.  Each function fills its half.
struct LnxKernels {
  const void* fwd[2][2];
  const void* bwd[2][2];
  const void* bwd2[2];  // backward, one block, at most 320 threads, two blocks per SM
  int nq_fwd, nq_bwd;
};
LnxKernels lnx_fwd_kernels_f32();
LnxKernels lnx_fwd_kernels_bf16();
LnxKernels lnx_bwd_kernels_f32();
LnxKernels lnx_bwd_kernels_bf16();

// Phase-aligned softmax-family kernels for long rows (rr_smx.cuh): [mode]
// [cluster], mode 0 softmax, 1 log-softmax, 2 cross-entropy; nq chunks per
// thread.
struct SmxKernels {
  const void* k[3][2];
  int nq;  // target chunks per thread
};
constexpr int kSmxMaxT = 512;  // threads per block

// Softmax / log-softmax backward for long rows (rr_smb.cuh): [log][cluster].
struct SmbKernels {
  const void* k[2][2];
};
SmbKernels smb_kernels_f32();
SmbKernels smb_kernels_bf16();

// Pipelined LayerNorm / RMSNorm kernels for long rows (rr_lnp.cuh): [rms]
// [cluster]; nq_bwd chunks per thread at most in the backward.
struct LnpKernels {
  const void* fwd[2][2];
  const void* bwd[2][2];
  const void* bwd2[2];  // backward, one block, at most 320 threads, two blocks per SM
  int nq_bwd;
};
LnpKernels lnp_fwd_kernels_f32();
LnpKernels lnp_fwd_kernels_bf16();
LnpKernels lnp_bwd_kernels_f32();
LnpKernels lnp_bwd_kernels_bf16();
SmxKernels smx_kernels_f32();
SmxKernels smx_kernels_bf16();

// Column-block LayerNorm / RMSNorm kernels for very long rows (rr_lnc.cuh):
// [rms].  Forward: stats, merge, norm launches; backward: part, dx launches
// (then the column reduce).  A work item (one block) is (class, column block,
// row group): item = cls + P * (b + nb * grp).
struct LncGeo {
  int64_t rows;
  int64_t cols;
  int32_t P;        // phase classes
  int32_t nb;       // column blocks of kCB chunks
  int32_t ng;       // row groups per class
  int32_t rg;       // rows per group (of its class)
  int32_t cb;       // chunks per column block (<= 32 * kLncWarps * CPL)
  int64_t rec_off;  // backward: floats from the workspace to the (S1, S2) records
};
constexpr int kLncWarps = 4;    // warps per block (128 threads)
constexpr int kLncCplFwd = 4;  // chunks per lane of a row, forward
constexpr int kLncCplBwd = 2;  // chunks per lane of a row, backward
constexpr int kLncDepth = 4;   // row stages of a block's copy ring (a pair of rows ahead)
// dynamic shared memory of a column-block kernel: its ring of row stages and
// their mbarriers
constexpr int lnc_ring_bytes(bool bwd) {
  return kLncDepth * (bwd ? 2 * kLncCplBwd : kLncCplFwd) * 32 * kLncWarps * 16 + 8 * kLncDepth;
}
struct LncKernels {
  const void* stats[2];
  const void* merge[2];
  const void* norm[2];
  const void* part[2];
  const void* dx[2];
};
LncKernels lnc_kernels_f32();
LncKernels lnc_kernels_bf16();

// LayerNorm / RMSNorm backward of short misaligned rows by phase class
// (rr_lns.cuh): bwd[rms][v], v = (lanes a row, chunks a lane): 0 (8, 1),
// 1 (16, 1), 2 (32, 1), and fp32 only (null for bf16) 3 (32, 2); a row of up
// to lanes x chunks 16-byte chunks, 32 / lanes rows a warp.  Blocks of
// kLnsWarps warps, one column partial ([planes][cols] floats) per block.
constexpr int kLnsWarps = 8;
struct LnsGeo {
  int64_t rows;
  int32_t cols;
  int32_t P;    // phase classes (divides kLnsWarps)
  int32_t hb0;  // byte of row 0 within its 16-byte block (x, dy and dx alike)
  int32_t rb;   // bytes per row
};
struct LnsKernels {
  const void* bwd[2][4];
};
LnsKernels lns_kernels_f32();
LnsKernels lns_kernels_bf16();

// Rows of one column (rr_one.cuh), elementwise: fwd [mode] 0 softmax,
// 1 log-softmax, 2 cross-entropy; bwd [log]; norm_fwd / norm_bwd [rms].
// Blocks of kOneThreads threads; the norm backward writes one partial
// (planes floats) per block.
constexpr int kOneThreads = 256;
struct OneKernels {
  const void* fwd[3];
  const void* bwd[2];
  const void* norm_fwd[2];
  const void* norm_bwd[2];
};
OneKernels one_kernels_f32();
OneKernels one_kernels_bf16();

// Short-row span kernels (rr_span.cuh): [dtype][mode], mode 0 softmax,
// 1 log-softmax, 2 cross-entropy, 3 softmax backward, 4 log-softmax backward,
// 5 LayerNorm forward, 6 RMSNorm forward, 7 LayerNorm backward, 8 RMSNorm
// backward.
struct SpanKernelSet {
  const void* k[2][9];
};
SpanKernelSet span_kernels();

KernelSet softmax_kernels_f32();
KernelSet softmax_kernels_bf16();
KernelSet softmax_bwd_kernels_f32();
KernelSet softmax_bwd_kernels_bf16();
KernelSet lnfwd_kernels_f32();
KernelSet lnfwd_kernels_bf16();
KernelSet lnbwd_kernels_f32();
KernelSet lnbwd_kernels_bf16();
LnKernelSet ln_fwd_rowgroup_kernels_f32();
LnKernelSet ln_fwd_rowgroup_kernels_bf16();
LnKernelSet ln_bwd_rowgroup_kernels_f32();
LnKernelSet ln_bwd_rowgroup_kernels_bf16();
LnKernelSet rms_fwd_rowgroup_kernels_f32();
LnKernelSet rms_fwd_rowgroup_kernels_bf16();
LnKernelSet rms_bwd_rowgroup_kernels_f32();
LnKernelSet rms_bwd_rowgroup_kernels_bf16();
// Scaled dot-product attention forward (k_attn.cu): bf16 [bh][seq][d]
// tensors, scores scaled by scale_log2 = scale * log2 e.
struct AttnParams {
  const char* q;
  const char* k;
  const char* v;
  char* o;
  float* lse;  // [bh][seq] natural-log sum of exp of the scaled scores, or null
  int* err;    // device error word (a bounded wait that gave up)
  int64_t bh;  // heads (batch x heads)
  int64_t seq;
  float scale_log2;
  int32_t causal;
};
struct AttnKernel {
  const void* fn;  // null for an unsupported head dimension
  int smem;        // dynamic shared memory bytes
};
AttnKernel attn_fwd_kernel_for(int d);
// Encodes the TMA tensor maps of q, k, v and launches the kernel for head
// dimension d on stream (persistent: at most `sms` CTAs): null on success,
// else a short reason (nothing launched, or the launch failed).
const char* attn_fwd_launch(const AttnParams& p, int d, int sms, cudaStream_t stream);
// The column reduce's split of its 32 warps over the P partial rows: the
// smallest power of two >= P / 16, at most 32 (the rest of the warps take
// further columns), so each warp sums about 16 partials.  A block covers
// 32 * (32 / split) columns.
inline __host__ __device__ int col_reduce_split(int64_t P) {
  int s = 1;
  while (s < 32 && (int64_t)s * 16 < P) s <<= 1;
  return s;
}
const void* col_reduce_kernel_ptr_f32();
const void* col_reduce_kernel_ptr_bf16();

}  // namespace rr
