// rr_api.cu -- the C ABI of librr.so: argument checks, per-device attribute
// cache, choice of kernel variant, and launches on the caller's stream.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <utility>

#include "../../include/rr.h"
#include "rr_kernels.h"
#include "rr_ln.cuh"
#include "rr_lnx.cuh"
#include "rr_span.cuh"
#include "rr_ops.cuh"

namespace {

using rr::KernelSet;

thread_local std::string g_detail;

rr_status fail(rr_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_detail = buf;
  return s;
}

rr_status ok() {
  g_detail.clear();
  return RR_OK;
}

// Error word written by bounded device-side waits that give up.
__device__ int g_rr_device_error;

struct DevInfo {
  bool init = false;
  int sms = 0;
  int smem_optin = 0;
  int* err = nullptr;
  std::map<const void*, int> smem_set;                   // kernel -> max dyn smem set
  std::map<std::pair<const void*, long long>, int> occ;  // (kernel, T<<32|smem) -> blocks/SM
  std::map<std::pair<const void*, long long>, int> ncl;  // (kernel, K<<32|smem) -> clusters
};

constexpr int kMaxDev = 64;
std::mutex g_mu;
DevInfo g_dev[kMaxDev];

rr_status device_info(DevInfo** out) {
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) return fail(RR_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (d < 0 || d >= kMaxDev) return fail(RR_ERR_CUDA, "device index %d out of range", d);
  DevInfo& di = g_dev[d];
  if (!di.init) {
    if ((e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, d)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&di.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, d)) !=
            cudaSuccess ||
        (e = cudaGetSymbolAddress(reinterpret_cast<void**>(&di.err), g_rr_device_error)) !=
            cudaSuccess)
      return fail(RR_ERR_CUDA, "device attributes: %s", cudaGetErrorString(e));
    di.init = true;
  }
  *out = &di;
  return RR_OK;
}

rr_status set_smem(DevInfo* di, const void* fn, size_t smem) {
  int& cur = di->smem_set[fn];
  if ((int)smem > cur) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
      return fail(RR_ERR_CUDA, "cudaFuncSetAttribute(%zu B smem): %s", smem, cudaGetErrorString(e));
    cur = (int)smem;
  }
  return RR_OK;
}

enum OpKind { kSoftmax = 0, kLnFwd = 1, kLnBwd = 2, kRmsFwd = 3, kRmsBwd = 4, kSoftmaxBwd = 5 };

// Row-engine kernel sets (the RMSNorm kinds have none: row-group kernels only).
const KernelSet& kernels(OpKind op, rr_dtype dt) {
  static KernelSet sets[4][2] = {
      {rr::softmax_kernels_f32(), rr::softmax_kernels_bf16()},
      {rr::lnfwd_kernels_f32(), rr::lnfwd_kernels_bf16()},
      {rr::lnbwd_kernels_f32(), rr::lnbwd_kernels_bf16()},
      {rr::softmax_bwd_kernels_f32(), rr::softmax_bwd_kernels_bf16()},
  };
  return sets[op == kSoftmaxBwd ? 3 : op][dt];
}

const rr::LnKernelSet& ln_kernels(OpKind op, rr_dtype dt) {
  static rr::LnKernelSet sets[4][2] = {
      {rr::ln_fwd_rowgroup_kernels_f32(), rr::ln_fwd_rowgroup_kernels_bf16()},
      {rr::ln_bwd_rowgroup_kernels_f32(), rr::ln_bwd_rowgroup_kernels_bf16()},
      {rr::rms_fwd_rowgroup_kernels_f32(), rr::rms_fwd_rowgroup_kernels_bf16()},
      {rr::rms_bwd_rowgroup_kernels_f32(), rr::rms_bwd_rowgroup_kernels_bf16()},
  };
  return sets[op - kLnFwd][dt];
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t a, int64_t b) { return cdiv(a, b) * b; }

struct Plan {
  int kind = 0;  // 0: row engine (rr::Geo), 1: row-group LayerNorm (rr::LnGeo), 2: rr::LnxGeo
  bool staged = false;
  int mode = 0;  // 0: 16-byte chunks, 1: elements
  int G = 0, T = 0, K = 1;
  const void* fn = nullptr;
  int64_t grid = 0;
  size_t smem = 0;
  int64_t partials = 0;  // LayerNorm backward: rows of column partials
  rr::Geo geo{};
  rr::LnGeo lgeo{};
  rr::LnxGeo xgeo{};
};

// Chooses the kernel variant and launch shape for (op, dtype, mode, rows, cols)
// on the current device.  head_free: every row starts 16-byte aligned, so a
// row needs no extra chunk for a ragged head.  max_partials caps the number of
// row groups (direct) or clusters (staged) that each leave a column partial.
// Deterministic for a given device, so the workspace size query and the launch agree.
// force: -1 any tier, 1 direct variants only, 2 staged one row per CTA only,
// 3 staged cluster-split rows only (K >= 2).
rr_status make_plan(OpKind op, rr_dtype dt, int mode, bool head_free, int64_t rows, int64_t cols,
                    Plan* pl, int64_t max_partials, int force) {
  std::lock_guard<std::mutex> lock(g_mu);
  DevInfo* di = nullptr;
  rr_status st = device_info(&di);
  if (st != RR_OK) return st;
  const KernelSet& ks = kernels(op, dt);
  const int E = dt == RR_BF16 ? 2 : 4;
  const int V = 16 / E;
  const int NT = (op == kLnBwd || op == kSoftmaxBwd) ? 2 : 1;
  pl->mode = mode;
  pl->geo.rows = rows;
  pl->geo.cols = cols;

  // Direct variants: the smallest row group whose threads hold the row.
  const int64_t units = mode == 0 ? cdiv(cols * E + (head_free ? 0 : 15), 16) : cols;
  int gi = -1;
  for (int i = 0; i < rr::kNumDirectG; ++i)
    if (cdiv(units, (int64_t)1 << i) <= ks.nq_direct[mode]) {
      gi = i;
      break;
    }
  if (gi >= 0 && ks.direct[mode][0] != nullptr && force != 2 && force != 3) {
    const int G = 1 << gi;
    const int T = ks.maxt_direct > G ? ks.maxt_direct : G;
    const int ngroups = T / G;
    size_t red = (size_t)(G > 32 ? ngroups * 1024 : 0) + 32;
    const int W = mode == 0 ? V : 1;
    size_t col = (op == kLnBwd) ? (size_t)ngroups * 2 * round_up(cols, W) * 4 : 0;
    size_t smem = round_up((int64_t)red, 16) + col;
    if ((int64_t)smem <= di->smem_optin) {
      const void* fn = ks.direct[mode][gi];
      if ((st = set_smem(di, fn, smem)) != RR_OK) return st;
      int& occ = di->occ[{fn, ((long long)T << 32) | (long long)smem}];
      if (occ == 0) {
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, T, smem);
        if (e != cudaSuccess || occ <= 0)
          return fail(RR_ERR_CUDA, "occupancy query: %s", cudaGetErrorString(e));
      }
      int64_t per_sm = op == kLnBwd ? (occ < 2 ? occ : 2) : occ;
      int64_t grid = cdiv(rows, ngroups);
      if (grid > (int64_t)di->sms * per_sm) grid = (int64_t)di->sms * per_sm;
      if (grid > max_partials) grid = max_partials;
      pl->staged = false;
      pl->G = G;
      pl->T = T;
      pl->K = 1;
      pl->fn = fn;
      pl->grid = grid;
      pl->smem = smem;
      pl->partials = grid;
      pl->geo.slice = cols;
      pl->geo.nbuf = 0;
      pl->geo.buf_bytes = 0;
      pl->geo.red_off = 0;
      pl->geo.col_off = (int32_t)round_up((int64_t)red, 16);
      return RR_OK;
    }
  }

  if (force == 1)
    return fail(RR_ERR_INVALID_ARG, "tier 1 (row in registers) cannot hold rows of %lld columns",
                (long long)cols);

  // Staged variants: one row (slice) per CTA, K-CTA clusters for long rows.
  const int T = ks.maxt_staged;
  const int nq = ks.nq_staged[mode];
  int K = 0;
  int64_t slice = 0;
  for (int k = force == 3 ? 2 : 1; k <= (force == 2 ? 1 : 8); k *= 2) {
    const int64_t sl = round_up(cdiv(cols, k), V);
    if (k > 1 && (k - 1) * sl >= cols) break;
    const int64_t su = mode == 0 ? cdiv(sl * E + (head_free ? 0 : 15), 16) : sl;
    if (cdiv(su, T) <= nq) {
      K = k;
      slice = sl;
      break;
    }
  }
  if (K == 0)
    return fail(RR_ERR_INVALID_ARG,
                force >= 2 ? "tier %d cannot hold rows of %lld columns"
                           : "cols=%lld is beyond the supported row length for this operation",
                force >= 2 ? force : (long long)cols, (long long)cols);
  const int64_t buf_bytes = round_up(slice * E + 32, 128);
  const int64_t colb = (op == kLnBwd) ? 2 * round_up(slice, mode == 0 ? V : 1) * 4 : 0;
  const int64_t fixed = 2 * 8 + 32 + 1024 + 32 + colb;
  int nbuf = 2;
  if (nbuf * NT * buf_bytes + fixed > di->smem_optin) nbuf = 1;
  if (nbuf * NT * buf_bytes + fixed > di->smem_optin)
    return fail(RR_ERR_INVALID_ARG, "row slice of %lld bytes does not fit shared memory",
                (long long)(slice * E));
  const int64_t red_off = round_up(nbuf * NT * buf_bytes + nbuf * 8, 16);
  const int64_t col_off = round_up(red_off + 1024 + 32, 16);
  const size_t smem = (size_t)(col_off + colb);
  const void* fn = ks.staged[mode];
  if ((st = set_smem(di, fn, smem)) != RR_OK) return st;
  int64_t grid;
  if (K == 1) {
    int& occ = di->occ[{fn, ((long long)T << 32) | (long long)smem}];
    if (occ == 0) {
      cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, T, smem);
      if (e != cudaSuccess || occ <= 0)
        return fail(RR_ERR_CUDA, "occupancy query: %s", cudaGetErrorString(e));
    }
    grid = rows < (int64_t)di->sms * occ ? rows : (int64_t)di->sms * occ;
    if (grid > max_partials) grid = max_partials;
  } else {
    int& ncl = di->ncl[{fn, ((long long)K << 32) | (long long)smem}];
    if (ncl == 0) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = K;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3((unsigned)(K * di->sms));
      cfg.blockDim = dim3((unsigned)T);
      cfg.dynamicSmemBytes = smem;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      cudaError_t e = cudaOccupancyMaxActiveClusters(&ncl, fn, &cfg);
      if (e != cudaSuccess || ncl <= 0)
        return fail(RR_ERR_CUDA, "cluster occupancy query (K=%d): %s", K, cudaGetErrorString(e));
    }
    int64_t nc = rows < ncl ? rows : ncl;
    if (nc > max_partials) nc = max_partials;
    grid = (int64_t)K * nc;
  }
  pl->staged = true;
  pl->G = T;
  pl->T = T;
  pl->K = K;
  pl->fn = fn;
  pl->grid = grid;
  pl->smem = smem;
  pl->partials = grid / K;
  pl->geo.slice = slice;
  pl->geo.nbuf = nbuf;
  pl->geo.buf_bytes = (int32_t)buf_bytes;
  pl->geo.red_off = (int32_t)red_off;
  pl->geo.col_off = (int32_t)col_off;
  return RR_OK;
}

// Row-group LayerNorm / RMSNorm plan (rr_ln.cuh): the smallest group G whose
// threads hold a row, G = 1 .. 1024, with gamma (/ beta, and the backward's
// column partials) in shared memory.  lmode: 0 chunks with aligned rows, 1 chunks
// with any row alignment, 2 elements.  RR_ERR_INVALID_ARG when the row does
// not fit one group (the caller then plans the staged engine kernels).
static rr_status ln_rowgroup_plan_impl(OpKind op, rr_dtype dt, int lmode, int64_t rows,
                                       int64_t cols, Plan* pl, int64_t max_partials,
                                       bool allow_deep, bool* used_deep) {
  std::lock_guard<std::mutex> lock(g_mu);
  DevInfo* di = nullptr;
  rr_status st = device_info(&di);
  if (st != RR_OK) return st;
  const rr::LnKernelSet& ls = ln_kernels(op, dt);
  const int E = dt == RR_BF16 ? 2 : 4;
  const int W = lmode == 2 ? 1 : 16 / E;
  const int64_t nfull = cols / W, rag = cols % W, nch = nfull + (rag > 0 ? 1 : 0);
  int nq = ls.nq[lmode];
  int gi = -1;
  for (int i = 0; i < rr::kNumLnG; ++i)
    if ((int64_t)nq << i >= nch) {
      gi = i;
      break;
    }
  // The deep variants where built (more chunks per thread, so the per-row
  // work is paid by fewer threads; the backward ones keep their column partials
  // in shared memory), chosen where they measured faster: forward rows the
  // standard variants would give 128 threads or more, RMSNorm backward rows
  // they would give 512, and LayerNorm backward rows longer than the standard
  // variants hold (two planes of shared-memory partials cost more than the
  // fewer threads save).  RR_LN_DEEP=0 keeps the standard ones (tuning aid).
  const bool fwdop = op == kLnFwd || op == kRmsFwd;
  const int deep_from = fwdop ? 7 : op == kRmsBwd ? 9 : 10;
  bool deep = allow_deep && lmode < 2 && ls.nqd > 0 && gi >= deep_from;
  if (const char* f = std::getenv("RR_LN_DEEP")) deep = deep && f[0] != '0';
  if (deep) {
    for (int i = 6; i < rr::kNumLnG; ++i)
      if ((int64_t)ls.nqd << i >= nch && ls.kd[lmode][i] != nullptr) {
        gi = i;
        nq = ls.nqd;
        break;
      }
    deep = nq == ls.nqd;
  }
  *used_deep = deep;
  if (gi < 0 || (deep ? ls.kd[lmode][gi] : ls.k[lmode][gi]) == nullptr)
    return fail(RR_ERR_INVALID_ARG, "row longer than one row group holds");
  const void* fn = deep ? ls.kd[lmode][gi] : ls.k[lmode][gi];
  // rows of at most 32 chunks: one chunk per thread where that variant exists
  for (int i = 0; i <= 5 && !deep; ++i)
    if (((int64_t)1 << i) >= nch) {
      if (ls.k1[lmode][i] != nullptr) {
        gi = i;
        fn = ls.k1[lmode][i];
      }
      break;
    }
  const int G = 1 << gi;
  const bool fwdk = fwdop;
  const int planes = (op == kLnFwd || op == kLnBwd) ? 2 : 1;  // gamma, beta / dgamma, dbeta
  const int M1 = fwdk ? 256 : deep ? 128 : 512;
  const int T = G > M1 ? G : M1;
  const int ngroups = T / G;
  const int64_t npad = nch * W;
  const int64_t red_off = round_up((fwdk ? planes : 1) * npad * 4, 16);
  const int64_t acc_off = round_up(red_off + (G > 32 ? (int64_t)ngroups * 1024 : 0), 16);
  const int64_t acc_end = acc_off + (fwdk ? 0 : (int64_t)ngroups * planes * npad * 4);
  // backward with aligned rows: per-thread prefetch slots [2][2][chunks per thread][T]
  const int nq_used = (fn == ls.k1[lmode][gi]) ? 1 : nq;
  const int64_t pf_off = round_up(acc_end, 16);
  // prefetch space: aligned rows, per-thread slots [2][tensors][chunks per thread][T];
  // misaligned rows (chunk mode), per-group row buffers [tensors][2][chunks + 2]
  const int ntens = fwdk ? 1 : 2;
  int64_t pf_bytes = 0;
  if (lmode == 0) pf_bytes = (int64_t)2 * ntens * nq_used * 16 * T;
  if (lmode == 1 && (fwdk ? G >= 32 : nq_used > 1))
    pf_bytes = (int64_t)ngroups * 2 * ntens * (nch + 2) * 16;
  const int64_t smem = pf_off + pf_bytes;
  if (smem > di->smem_optin) return fail(RR_ERR_INVALID_ARG, "row-group shared memory too large");
  if ((st = set_smem(di, fn, (size_t)smem)) != RR_OK) return st;
  int& occ = di->occ[{fn, ((long long)T << 32) | (long long)smem}];
  if (occ == 0) {
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, T, (size_t)smem);
    if (e != cudaSuccess || occ <= 0)
      return fail(RR_ERR_CUDA, "occupancy query: %s", cudaGetErrorString(e));
  }
  int64_t grid = cdiv(rows, ngroups);
  if (grid > (int64_t)di->sms * occ) grid = (int64_t)di->sms * occ;
  if (grid > max_partials) grid = max_partials;
  pl->kind = 1;
  pl->staged = false;
  pl->mode = lmode;
  pl->G = G;
  pl->T = T;
  pl->K = 1;
  pl->fn = fn;
  pl->grid = grid;
  pl->smem = (size_t)smem;
  pl->partials = grid;
  pl->lgeo = rr::LnGeo{rows,          (int32_t)cols,    (int32_t)nfull,   (int32_t)rag,
                       (int32_t)nch,  (int32_t)red_off, (int32_t)acc_off, (int32_t)pf_off,
                       (int32_t)cols, 0};
  return RR_OK;
}

// The plan above, falling back to the standard variants where a deep one does
// not fit shared memory (its per-group row buffers and partials grow with the
// row).
rr_status ln_rowgroup_plan(OpKind op, rr_dtype dt, int lmode, int64_t rows, int64_t cols, Plan* pl,
                           int64_t max_partials) {
  bool deep = false;
  rr_status st = ln_rowgroup_plan_impl(op, dt, lmode, rows, cols, pl, max_partials, true, &deep);
  if (st == RR_ERR_INVALID_ARG && deep)
    st = ln_rowgroup_plan_impl(op, dt, lmode, rows, cols, pl, max_partials, false, &deep);
  return st;
}

// Forward rows too long for one row group: the row is split over a cluster of K
// blocks (K = 2 .. 8), each one group of 256 / 512 / 1024 threads holding a
// slice of whole chunks (rr_ln.cuh, CL).  Among the (K, group size) pairs that
// fit: the wide 256-thread variant first, then the least estimated time, rounds
// of rows (rows / clusters resident on the device) x (chunks per thread + 2 for
// the per-row reductions).
rr_status ln_cluster_plan(OpKind op, rr_dtype dt, int lmode, int64_t rows, int64_t cols, Plan* pl,
                          int64_t max_partials = INT64_MAX) {
  std::lock_guard<std::mutex> lock(g_mu);
  DevInfo* di = nullptr;
  rr_status st = device_info(&di);
  if (st != RR_OK) return st;
  const rr::LnKernelSet& ls = ln_kernels(op, dt);
  const int E = dt == RR_BF16 ? 2 : 4;
  const int W = lmode == 2 ? 1 : 16 / E;
  const int nq = ls.nq[lmode];
  const bool fwdop = op == kLnFwd || op == kRmsFwd;
  const int planes = op == kLnFwd ? 2 : 1;           // gamma (, beta) staged as fp32
  const int kp = fwdop ? 0 : op == kLnBwd ? 2 : 1;  // backward: planes of column partials
  const int ntens = fwdop ? 1 : 2;
  // RR_LN_CLUSTER="K:v" forces cluster size K and variant v (0..3: 256, 512,
  // 1024 threads, or the wide 256-thread one) when that pair fits (tuning aid).
  int forceK = 0, forceV = -1;
  if (const char* f = std::getenv("RR_LN_CLUSTER")) std::sscanf(f, "%d:%d", &forceK, &forceV);
  struct Choice {
    int K = 0, T = 0, ncl = 0;
    int64_t S = 0, nchs = 0, smem = 0, red_off = 0, cl_off = 0, acc_off = 0, pf_off = 0;
    const void* fn = nullptr;
    double cost = 0.0;
  } best;
  for (int K = 2; K <= 8; ++K) {
    const int64_t S = round_up(cdiv(cols, K), W);
    if ((K - 1) * S >= cols) continue;  // every block of the cluster gets columns
    const int64_t nchs = S / W, npad = nchs * W;
    if (forceK > 0 && K != forceK) continue;
    for (int gi = 0; gi < 4; ++gi) {
      if (forceV >= 0 && gi != forceV) continue;
      const int T = gi < 3 ? 256 << gi : 256;
      // forward [3]: the wide 256-thread variant; backward: the deep chunk count
      const int nqv = fwdop ? (gi < 3 ? nq : 2 * nq) : ls.nqd;
      const void* fn = ls.kc[lmode][gi];
      if (fn == nullptr || (int64_t)nqv * T < nchs) continue;
      const int64_t red_off = round_up(planes * npad * 4, 16);
      const int64_t cl_off = round_up(red_off + 1024, 16);
      const int64_t acc_off = round_up(cl_off + 32, 16);
      const int64_t pf_off = round_up(acc_off + (int64_t)kp * npad * 4, 16);
      int64_t pf_bytes = 0;
      if (lmode == 0) pf_bytes = (int64_t)2 * ntens * nqv * 16 * T;
      if (lmode == 1) pf_bytes = (int64_t)2 * ntens * (nchs + 2) * 16;
      const int64_t smem = pf_off + pf_bytes;
      if (smem > di->smem_optin) continue;
      if ((st = set_smem(di, fn, (size_t)smem)) != RR_OK) return st;
      int& ncl = di->ncl[{fn, ((long long)K << 32) | (long long)smem}];
      if (ncl == 0) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = K;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3((unsigned)(K * di->sms));
        cfg.blockDim = dim3((unsigned)T);
        cfg.dynamicSmemBytes = (size_t)smem;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t e = cudaOccupancyMaxActiveClusters(&ncl, fn, &cfg);
        if (e != cudaSuccess)
          return fail(RR_ERR_CUDA, "cluster occupancy query (K=%d): %s", K, cudaGetErrorString(e));
        if (ncl <= 0) ncl = -1;  // cannot be resident: remembered, skipped
      }
      if (ncl <= 0) continue;
      // measured on 65537-column rows: the wide variant (fewer, fuller threads:
      // the per-row reductions are paid by half as many threads) beats the others
      // wherever it fits, so it is ranked first; among equals, rounds x chunks
      const double rounds = (double)cdiv(rows, ncl);
      const double cost = rounds * (double)(cdiv(nchs, T) + 2) + (fwdop && gi != 3 ? 1e9 : 0.0);
      if (best.K == 0 || cost < best.cost - 1e-9) {
        best.K = K;
        best.T = T;
        best.ncl = ncl;
        best.S = S;
        best.nchs = nchs;
        best.smem = smem;
        best.red_off = red_off;
        best.cl_off = cl_off;
        best.acc_off = acc_off;
        best.pf_off = pf_off;
        best.fn = fn;
        best.cost = cost;
      }
    }
  }
  if (best.K == 0) return fail(RR_ERR_INVALID_ARG, "row longer than a cluster of row groups holds");
  pl->kind = 1;
  pl->staged = false;
  pl->mode = lmode;
  pl->G = best.T;
  pl->T = best.T;
  pl->K = best.K;
  pl->fn = best.fn;
  int64_t nc = rows < best.ncl ? rows : best.ncl;
  if (nc > max_partials) nc = max_partials;  // the backward writes one partial row per cluster
  pl->grid = (int64_t)best.K * nc;
  pl->smem = (size_t)best.smem;
  pl->partials = pl->grid / best.K;
  pl->lgeo = rr::LnGeo{rows,
                       (int32_t)cols,
                       (int32_t)best.nchs,
                       0,
                       (int32_t)best.nchs,
                       (int32_t)best.red_off,
                       (int32_t)best.acc_off,
                       (int32_t)best.pf_off,
                       (int32_t)best.S,
                       (int32_t)best.cl_off};
  return RR_OK;
}

// Phase-class kernels for long rows: the plan (kernel, geometry, launch shape)
// of one call.  The row tensors must share their address modulo 16 (the caller
// checks); gamma / beta may have any alignment.  Rows of at least kLnxMinBytes
// (measured on 2^24-element rows, bf16, cold L2: the LayerNorm kernels beat the
// row-group ones from there — 4097 columns: backward 65.5 -> 55.5 us, RMSNorm
// forward 23.2 -> 19.3 us — and lose on shorter rows, 1000 columns: forward
// 16.9 against 28.6 us at best).  Kernels by op:
//   kLnFwd / kRmsFwd / kLnBwd / kRmsBwd: rr_lnx.cuh (rows in registers), or
//     with lnp the pipelined rr_lnp.cuh ones;
//   kSoftmax: rr_smx.cuh (smode 0 softmax, 1 log-softmax, 2 cross-entropy);
//   kSoftmaxBwd: rr_smb.cuh (smode 1: log-softmax).
// A block holds R row groups of G threads, or is one rank of a cluster of
// K = 2 .. 8 blocks splitting rows beyond one block (force: -1 any, 1 one
// block only, 3 clusters only).  Rows of each of the P phase classes go to
// bpc row owners; the norm backward writes one partial row per owner, at most
// max_partials.  RR_LNX=0 / RR_SMX=0 turn the kernels off (tuning aids).
constexpr int64_t kLnxMinBytes = 8192;

rr_status lnx_plan_impl(OpKind op, rr_dtype dt, int64_t rows, int64_t cols, Plan* pl,
                        int64_t max_partials, int force, int smode, bool lnp) {
  const bool smx = op == kSoftmax;
  const bool smb = op == kSoftmaxBwd;  // softmax / log-softmax backward (smode: log)
  if (const char* f = std::getenv(smx || smb ? "RR_SMX" : "RR_LNX"); f != nullptr && f[0] == '0')
    return fail(RR_ERR_INVALID_ARG, "phase-aligned kernels off");
  const bool pipe = smx || smb || lnp;  // rows held in shared memory, merges pipelined
  const int E = dt == RR_BF16 ? 2 : 4, W = 16 / E;
  // RR_LNX_MIN lowers (or raises) the row length these kernels take (bytes;
  // tuning aid)
  int64_t min_bytes = kLnxMinBytes;
  if (const char* f = std::getenv("RR_LNX_MIN")) min_bytes = std::max<int64_t>(16, std::atoll(f));
  if (cols * E < min_bytes || rows < 1) return fail(RR_ERR_INVALID_ARG, "short rows");
  const bool fwd = op == kLnFwd || op == kRmsFwd;
  const bool rms = op == kRmsFwd || op == kRmsBwd;
  std::lock_guard<std::mutex> lock(g_mu);
  DevInfo* di = nullptr;
  rr_status st = device_info(&di);
  if (st != RR_OK) return st;
  static const rr::LnxKernels fk[2] = {rr::lnx_fwd_kernels_f32(), rr::lnx_fwd_kernels_bf16()};
  static const rr::LnxKernels bk[2] = {rr::lnx_bwd_kernels_f32(), rr::lnx_bwd_kernels_bf16()};
  static const rr::SmxKernels sk[2] = {rr::smx_kernels_f32(), rr::smx_kernels_bf16()};
  static const rr::LnpKernels pf[2] = {rr::lnp_fwd_kernels_f32(), rr::lnp_fwd_kernels_bf16()};
  static const rr::LnpKernels pb[2] = {rr::lnp_bwd_kernels_f32(), rr::lnp_bwd_kernels_bf16()};
  static const rr::SmbKernels bb[2] = {rr::smb_kernels_f32(), rr::smb_kernels_bf16()};
  // chunks per thread: a target for the softmax family and the pipelined
  // forward; at most nq_bwd in the pipelined backward (register partials)
  const int NQ = smx || smb ? sk[dt].nq : (lnp && fwd) ? sk[dt].nq : lnp ? pb[dt].nq_bwd
                 : fwd ? fk[dt].nq_fwd : bk[dt].nq_bwd;
  const int NT = fwd || smx ? 1 : 2;
  const int vecs = smx || smb ? 0 : fwd ? (rms ? 1 : 2) : 1;  // gamma (, beta) planes
  const int64_t rb = (cols * E) % 16;
  int64_t P = 1;
  if (rb != 0) {
    int64_t a = 16, b = rb;
    while (b) { const int64_t t = a % b; a = b; b = t; }
    P = 16 / a;
  }
  const int64_t nch_min = cdiv(cols, W), nch_max = cdiv(cols + W - 1, W);
  // The LayerNorm forward split over a cluster measured slower than the
  // clusters of row groups (bf16 65537 columns: 65.9 against 49.4 us), so it
  // takes this path only when tier 3 is forced.
  const int kmax = force == 1 ? 1 : (op == kLnFwd && !lnp && force != 3) ? 1 : 8;
  // Pipelined kernels: the row stays in shared memory, so a thread holds no
  // row in registers; NQ is the target of chunks per thread and a block takes
  // up to kSmxMaxT threads.  A split that keeps three stages per ring is
  // preferred to one with two (more rows in flight); the others take any.
  const int maxT = pipe ? rr::kSmxMaxT : rr::kLnxMaxT;
  // the pipelined backward keeps at most NQ chunks a thread (no one-warp rows
  // beyond that)
  const bool cap = lnp && !fwd;
  int cpt = NQ, forceK = 0, blockT = pipe ? 512 : 256, solo_max = cap ? NQ : 40;
  bool force_cpt = cap;
  // RR_SMX_CPT (chunks per thread), RR_SMX_BT (threads per block, groups of
  // one-block rows), RR_SMX_SOLO (most chunks per lane of a row held by one
  // warp, 0: never) and RR_LNX_K (cluster size) force a shape (tuning aids)
  if (const char* f = std::getenv("RR_SMX_CPT"); pipe && !cap && f) {
    cpt = std::max(1, std::atoi(f));
    force_cpt = true;
  }
  if (const char* f = std::getenv("RR_SMX_BT"); pipe && f) blockT = std::max(32, std::atoi(f));
  if (const char* f = std::getenv("RR_SMX_SOLO"); f && !cap) solo_max = std::max(0, std::atoi(f));
  if (const char* f = std::getenv("RR_LNX_K")) forceK = std::atoi(f);
  // RR_LNX_2B=0 keeps the backward on the 128-register variant (tuning aid)
  bool two_blocks = true;
  if (const char* f = std::getenv("RR_LNX_2B"); f != nullptr && f[0] == '0') two_blocks = false;
  for (int minNS = pipe ? 3 : 2; minNS >= 2; --minNS)
  for (int K = force == 3 ? 2 : 1; K <= kmax; ++K) {
    const int64_t S = cdiv(nch_max, K);
    if (K > 1 && (K - 1) * S >= nch_min) break;  // every rank of every phase gets chunks
    if (forceK > 0 && K != forceK) continue;
    // Softmax family split over a cluster: only for a few rows per SM.  With
    // many rows the row engine's 1024-thread groups (the row and the next one
    // in registers) stream better: bf16 16384 x 50304 cross-entropy 554 us
    // there against 1050 us here; 256 rows of 65537 columns 33.9 against
    // 25.8 us.
    if ((smx || smb) && K > 1 && rows >= 4 * (int64_t)di->sms && forceK == 0 && force != 3) break;
    // softmax family: one warp per row where its lanes hold at most solo_max
    // chunks each (no merge across warps; two stages per ring suffice)
    const bool solo = pipe && K == 1 && S <= 32 * (int64_t)solo_max;
    // a cluster rank holds one group: as many threads as the block takes
    const int64_t kcpt = pipe && K > 1 && !force_cpt ? std::max<int64_t>(1, cdiv(S, maxT)) : cpt;
    const int64_t G = solo ? 32 : std::max<int64_t>(32, round_up(cdiv(S, kcpt), 32));
    if (G > maxT) continue;
    const void* fn1 = smx   ? sk[dt].k[smode][K > 1]
                      : smb ? bb[dt].k[smode][K > 1]
                      : lnp ? (fwd ? pf[dt].fwd[rms][K > 1] : pb[dt].bwd[rms][K > 1])
                      : fwd ? fk[dt].fwd[rms][K > 1]
                            : bk[dt].bwd[rms][K > 1];
    const int64_t planes = (int64_t)vecs * S * W * 4;
    // R row groups per block (one per block in a cluster), up to 256 threads;
    // NS stages per group's ring: the most that fit, four only where two blocks
    // still fit an SM
    int64_t rmax = K > 1 ? 1 : std::max<int64_t>(1, std::min<int64_t>(pipe ? 16 : 8, blockT / G));
    // RR_LNX_SHAPE="R:NS" forces the groups per block and the stages (tuning aid)
    int fR = 0, fNS = 0;
    if (const char* f = std::getenv("RR_LNX_SHAPE")) std::sscanf(f, "%d:%d", &fR, &fNS);
    if (fR > 0 && K == 1 && fR * G <= maxT) rmax = fR;
    for (int64_t R = rmax; R >= 1; --R) {
      // the row-in-registers RMSNorm backward, bf16: a variant capped at 96
      // registers (two blocks of up to 320 threads per SM) where the block is
      // that small (4097 columns: 47.2 -> 39.9 us).  The LayerNorm and fp32
      // variants spill at that cap and lost (bf16 LayerNorm 54.5 -> 90.5 us).
      const bool cap96 = !pipe && !fwd && rms && dt == RR_BF16 && K == 1 && R * G <= 320;
      // the pipelined backward (not routed by default): a 96-register variant
      // for blocks of <= 320 threads (no spills: its rows stay in shared
      // memory); bf16 4097 columns 66.0 -> 56.1 us, against 55.0 us for the
      // row-in-registers kernel
      const bool pcap96 = lnp && !fwd && K == 1 && R * G <= 320;
      const void* fn = (cap96 && two_blocks)    ? bk[dt].bwd2[rms]
                       : (pcap96 && two_blocks) ? pb[dt].bwd2[rms]
                                                : fn1;
      const bool two = solo && fNS == 0;  // one warp per row: two stages
      for (int NS = two ? 2 : 4; NS >= (two ? 2 : minNS); --NS) {
        if (fNS >= 2 && NS != fNS) continue;
        if (fR > 0 && R != rmax) continue;
        // pipelined kernels: partial slots [2][K][warps] and two merge
        // barriers per group; the others: reduction slots and one barrier
        // per stage
        const int64_t red_off = round_up(planes, 16);
        const int64_t bar_off = red_off + 1024 * R * (pipe ? K : 1);
        const int64_t ring_off = round_up(bar_off + 8 * (pipe ? 2 : NS) * R, 128);
        const int64_t cl_off = ring_off + R * NS * NT * S * 16;
        const int64_t smem = cl_off + 32;
        if (smem > di->smem_optin) continue;
        if (!pipe && NS > 2 && fNS == 0 && 2 * smem > di->smem_optin) continue;
        const int T = (int)(R * G);
        if ((st = set_smem(di, fn, (size_t)smem)) != RR_OK) return st;
        int owners = 0;
        if (K == 1) {
          int& occ = di->occ[{fn, ((long long)T << 32) | (long long)smem}];
          if (occ == 0) {
            cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, T, smem);
            if (e != cudaSuccess || occ <= 0)
              return fail(RR_ERR_CUDA, "occupancy query: %s", cudaGetErrorString(e));
          }
          owners = di->sms * occ;
        } else {
          int& ncl = di->ncl[{fn, ((long long)K << 32) | (long long)smem | ((long long)T << 48)}];
          if (ncl == 0) {
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = K;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3((unsigned)(K * di->sms));
            cfg.blockDim = dim3((unsigned)T);
            cfg.dynamicSmemBytes = (size_t)smem;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            cudaError_t e = cudaOccupancyMaxActiveClusters(&ncl, fn, &cfg);
            if (e != cudaSuccess)
              return fail(RR_ERR_CUDA, "cluster occupancy query (K=%d): %s", K,
                          cudaGetErrorString(e));
            if (ncl <= 0) ncl = -1;
          }
          if (ncl <= 0) continue;
          owners = ncl;
        }
        int64_t bpc = owners / P;
        if (bpc < 1) bpc = 1;
        const int64_t per_class = cdiv(cdiv(rows, P), R);  // blocks with a row for every group
        if (bpc > per_class) bpc = per_class;
        if (!fwd && !smx && !smb) {
          if (max_partials < P) return fail(RR_ERR_INVALID_ARG, "too few column partials allowed");
          if (bpc > max_partials / P) bpc = max_partials / P;
        }
        pl->kind = 2;
        pl->staged = true;
        pl->mode = 0;
        pl->G = (int)G;
        pl->T = T;
        pl->K = K;
        pl->fn = fn;
        pl->grid = P * bpc * K;
        pl->smem = (size_t)smem;
        pl->partials = P * bpc;
        pl->xgeo = rr::LnxGeo{rows,          (int32_t)cols,    (int32_t)P,
                              (int32_t)bpc,  (int32_t)S,       NS,
                              (int32_t)G,    0,                (int32_t)red_off,
                              (int32_t)bar_off, (int32_t)ring_off, (int32_t)cl_off};
        return RR_OK;
      }
    }
  }
  return fail(RR_ERR_INVALID_ARG, "row does not fit the phase-aligned kernels");
}

// LayerNorm / RMSNorm forward: the pipelined kernels of rr_lnp.cuh where a
// warp holds a row and at least eight such warps share a block (rows of up to
// ~8 KB), else the row-in-registers kernels of rr_lnx.cuh.  Measured on 2^24
// elements (cold L2): bf16 4097 columns LayerNorm 33.1 -> 26.2 us, RMSNorm
// 20.4 -> 18.4 us; where fewer warps fit (fp32 4097: six) or rows need several
// warps, the pipelined kernels lost (fp32 4097 LayerNorm 47.5 against 37.3
// us, bf16 65537 91.3 against 49.9 us), and so did the pipelined backward
// (bf16 4097 67.6 against 55.7 us), which is not routed.  RR_LNP=0 turns the
// pipelined kernels off, RR_LNP=1 takes them wherever they fit (tuning aids).
rr_status lnx_plan(OpKind op, rr_dtype dt, int64_t rows, int64_t cols, Plan* pl,
                   int64_t max_partials, int force, int smode = -1) {
  if (op == kSoftmax) return lnx_plan_impl(op, dt, rows, cols, pl, max_partials, force, smode, false);
  if (op == kSoftmaxBwd) {
    // Softmax / log-softmax backward: bf16 rows only, where measured faster
    // (4097 columns 39.5 -> 26.4 us, 65537 48.4 -> 45.3 us); fp32 rows, whose
    // two tensors leave room for few rows per SM, lost (4097: 37.8 against
    // 43.2 us, 65537: 73.0 against 141.6 us).  RR_SMB=1 takes them for fp32
    // too (tests, tuning).
    const char* f = std::getenv("RR_SMB");
    if (dt != RR_BF16 && !(f != nullptr && f[0] == '1'))
      return fail(RR_ERR_INVALID_ARG, "row engine for this dtype");
    return lnx_plan_impl(op, dt, rows, cols, pl, max_partials, force, smode, false);
  }
  const char* f = std::getenv("RR_LNP");
  const int mode = f == nullptr ? -1 : f[0] == '0' ? 0 : 1;
  const bool fwd = op == kLnFwd || op == kRmsFwd;
  if (mode == 1 || (mode < 0 && fwd)) {
    Plan tp;
    const rr_status st = lnx_plan_impl(op, dt, rows, cols, &tp, max_partials, force, smode, true);
    if (st == RR_OK && (mode == 1 || (tp.G == 32 && tp.T / tp.G >= 8))) {
      *pl = tp;
      return RR_OK;
    }
    if (st != RR_OK && st != RR_ERR_INVALID_ARG) return st;
  }
  return lnx_plan_impl(op, dt, rows, cols, pl, max_partials, force, smode, false);
}

// Column-block LayerNorm / RMSNorm kernels for very long rows (rr_lnc.cuh):
// statistics, then outputs, in separate launches over (class, column block,
// row group) items, so every SM streams from the first microsecond instead of
// waiting on a row per block or cluster.  Taken when no tier is forced for
// rows of at least 64 KB, and for the LayerNorm backward from 8 KB (bf16 4097
// columns 55.1 -> 49.5 us, fp32 63.1 -> 55.4 us; the forwards and the RMSNorm
// backward lost there to the phase-class kernels: bf16 LayerNorm forward 38.4
// against 26.6 us); RR_LNC=0 turns them off, RR_LNC_MIN (bytes) sets one
// threshold for all (tuning aids).  Items: as many row groups per class as keep the
// blocks within one wave (5 blocks per SM: registers, 32 KB copy rings), so each
// block streams as many rows as it can; each backward row group adds a
// column-partial row for the column reduce to read.
constexpr int64_t kLncMinBytes = 64 * 1024, kLncMinBytesLnBwd = 8192;

const rr::LncKernels& lnc_kernels(rr_dtype dt);

struct LncPlan {
  rr::LncGeo geo{};
  int64_t items = 0;
  int64_t partials = 0;   // backward: rows of column partials
  size_t rec_bytes = 0;   // (row, block) records
  size_t ws_bytes = 0;    // backward: partials + records
};

rr_status lnc_plan(bool bwd, bool rms, rr_dtype dt, int64_t rows, int64_t cols, LncPlan* lp,
                   int64_t max_partials = INT64_MAX, size_t ws_limit = SIZE_MAX) {
  if (const char* f = std::getenv("RR_LNC"); f != nullptr && f[0] == '0')
    return fail(RR_ERR_INVALID_ARG, "column-block kernels off");
  const int E = dt == RR_BF16 ? 2 : 4, W = 16 / E;
  int64_t min_bytes = bwd && !rms ? kLncMinBytesLnBwd : kLncMinBytes;
  if (const char* f = std::getenv("RR_LNC_MIN")) min_bytes = std::max<int64_t>(16, std::atoll(f));
  if (cols * E < min_bytes || rows < 1) return fail(RR_ERR_INVALID_ARG, "rows too short");
  int sms = 0;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    DevInfo* di = nullptr;
    rr_status st = device_info(&di);
    if (st != RR_OK) return st;
    sms = di->sms;
    // the streaming kernels' copy rings (dynamic shared memory)
    const rr::LncKernels& k = lnc_kernels(dt);
    const size_t ring = (size_t)rr::lnc_ring_bytes(bwd);
    const void* fns[2] = {bwd ? k.part[rms] : k.stats[rms], bwd ? k.dx[rms] : k.norm[rms]};
    for (const void* fn : fns)
      if ((st = set_smem(di, fn, ring)) != RR_OK) return st;
  }
  const int64_t rb = (cols * E) % 16;
  int64_t P = 1;
  if (rb != 0) {
    int64_t a = 16, b = rb;
    while (b) { const int64_t t = a % b; a = b; b = t; }
    P = 16 / a;
  }
  // column blocks of at most cbmax chunks, all of a row's blocks equal
  const int64_t cbmax = 32 * rr::kLncWarps * (bwd ? rr::kLncCplBwd : rr::kLncCplFwd);
  const int64_t nch_max = cdiv(cols + W - 1, W);
  const int64_t nb = cdiv(nch_max, cbmax);
  const int64_t cb = cdiv(nch_max, nb);
  const int64_t per_class = cdiv(rows, P);
  // RR_LNC_SLOTS: blocks per SM the item count aims at (tuning aid)
  int64_t per_sm = 5;
  if (const char* f = std::getenv("RR_LNC_SLOTS")) per_sm = std::max(1, std::atoi(f));
  const int64_t slots = per_sm * (int64_t)sms;
  int64_t ng = std::min<int64_t>(per_class, std::max<int64_t>(1, slots / (P * nb)));
  for (;; --ng) {
    const int64_t rg = cdiv(per_class, ng);
    const int64_t g2 = cdiv(per_class, rg);
    const int64_t planes = rms ? 1 : 2;
    const size_t rec = (size_t)rows * nb * (bwd ? 8 : rms ? 4 : 16);
    const size_t part = bwd ? (size_t)P * g2 * planes * cols * sizeof(float) : 0;
    const size_t ws = bwd ? ((part + 15) & ~size_t(15)) + rec : 0;
    if (ng > 1 && bwd && (P * g2 > max_partials || ws > ws_limit)) continue;
    if (P * nb * g2 > INT32_MAX) return fail(RR_ERR_INVALID_ARG, "too many column blocks");
    lp->geo = rr::LncGeo{rows, cols, (int32_t)P, (int32_t)nb, (int32_t)g2, (int32_t)rg, (int32_t)cb,
                         (int64_t)(((part + 15) & ~size_t(15)) / sizeof(float))};
    lp->items = P * nb * g2;
    lp->partials = P * g2;
    lp->rec_bytes = rec;
    lp->ws_bytes = ws;
    break;
  }
  if (bwd && (lp->partials > max_partials || lp->ws_bytes > ws_limit))
    return fail(RR_ERR_INVALID_ARG, "column-block partials exceed the workspace");
  return RR_OK;
}

const rr::LncKernels& lnc_kernels(rr_dtype dt) {
  static const rr::LncKernels k[2] = {rr::lnc_kernels_f32(), rr::lnc_kernels_bf16()};
  return k[dt == RR_BF16 ? 1 : 0];
}

// Forward launches (records in y, then mean / rstd, then y).
rr_status lnc_forward(bool rms, const LncPlan& lp, rr::LnFwdParams p, rr_dtype dt,
                      cudaStream_t stream) {
  const rr::LncKernels& k = lnc_kernels(dt);
  rr::LncGeo g = lp.geo;
  void* args[] = {&p, &g};
  const size_t ring = (size_t)rr::lnc_ring_bytes(false);
  cudaError_t e = cudaLaunchKernel(k.stats[rms], dim3((unsigned)lp.items), dim3(32 * rr::kLncWarps),
                                   args, ring, stream);
  if (e == cudaSuccess)
    e = cudaLaunchKernel(k.merge[rms], dim3((unsigned)cdiv(lp.geo.rows, 8)), dim3(256), args, 0,
                         stream);
  if (e == cudaSuccess)
    e = cudaLaunchKernel(k.norm[rms], dim3((unsigned)lp.items), dim3(32 * rr::kLncWarps), args,
                         ring, stream);
  if (e != cudaSuccess) return fail(RR_ERR_CUDA, "launch: %s", cudaGetErrorString(e));
  return RR_OK;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb);

// The forward's records live in y (rounded up to 16 bytes) until the last
// launch overwrites it: they must fit, and y must not overlap x.
bool lnc_fwd_fits(const LncPlan& lp, const void* x, const void* y, int64_t rows, int64_t cols,
                  size_t E) {
  const size_t n = (size_t)rows * cols * E;
  if (overlaps(x, n, y, n)) return false;
  const size_t pad = (16 - (reinterpret_cast<uintptr_t>(y) & 15)) & 15;
  return pad + lp.rec_bytes <= n;
}

// Plans in chunk mode when allowed, falling back to element mode (which holds
// longer rows per CTA) when the row does not fit the chunk-mode variants.
rr_status plan_any(OpKind op, rr_dtype dt, bool chunk_ok, bool head_free, int64_t rows,
                   int64_t cols, Plan* pl, int64_t max_partials = INT64_MAX, int force = -1) {
  if (chunk_ok) {
    rr_status st = make_plan(op, dt, 0, head_free, rows, cols, pl, max_partials, force);
    if (st != RR_ERR_INVALID_ARG) return st;
  }
  return make_plan(op, dt, 1, false, rows, cols, pl, max_partials, force);
}

// RR_FORCE_TIER = 0 .. 3 (or T0 .. T3) makes every call use one kernel tier,
// so tests can run each tier on any shape it can hold: 0 spans of short rows,
// 1 a row in registers (engine direct variants, LayerNorm / RMSNorm row
// groups), 2 staged rows, one per CTA, 3 cluster-split rows (LayerNorm /
// RMSNorm: clusters of row groups, the LayerNorm backward falling back to the
// staged engine with K >= 2; softmax family: the staged engine with K >= 2).
// A shape the forced tier cannot hold fails with RR_ERR_INVALID_ARG.
// Returns -1 when unset, -2 for a value outside those.
static int forced_tier() {
  const char* f = std::getenv("RR_FORCE_TIER");
  if (f == nullptr || *f == 0) return -1;
  if (*f == 'T' || *f == 't') ++f;
  if (f[0] >= '0' && f[0] <= '3' && f[1] == 0) return f[0] - '0';
  return -2;
}
static rr_status bad_tier() { return fail(RR_ERR_INVALID_ARG, "RR_FORCE_TIER must be 0..3 or T0..T3"); }
static rr_status no_span(int64_t cols) {
  return fail(RR_ERR_INVALID_ARG,
              "tier 0 (spans) takes 16-byte aligned tensors with short rows whose byte length "
              "is not a multiple of 16 (up to 448 bytes; 224 for the softmax backward, 64 "
              "(bf16 96) for the norm backward, fewer columns for some operations), not %lld "
              "columns",
              (long long)cols);
}

// Short misaligned rows (byte length not a multiple of 16, up to 448 bytes by
// operation, see span_plan; 16-byte aligned row tensors): the span kernels
// (rr_span.cuh), one warp per span of 32 x rpl rows of ~3 KB (at least 32
// rows).  mode 0
// softmax, 1 log-softmax, 2 cross-entropy, 3 softmax backward, 4 log-softmax
// backward, 5 LayerNorm forward, 6 RMSNorm forward, 7 LayerNorm backward,
// 8 RMSNorm backward.  aux_aligned: the labels (mode 2) or the row statistics
// (modes 7, 8) are 16-byte aligned and staged with the span.  The grid is at
// most max_grid blocks (the norm backward writes one column partial per block).
// RR_ERR_INVALID_ARG when not eligible.
struct SpanPlan {
  const void* fn = nullptr;
  int64_t smem = 0, grid = 0;
  rr::SpanGeo geo{};
};

static rr_status span_plan(rr_dtype dt, int mode, int64_t rows, int64_t cols, bool aux_aligned,
                           int64_t max_grid, SpanPlan* sp) {
  const int E = dt == RR_BF16 ? 2 : 4;
  // Rows whose byte length is not a multiple of 16.  Rows of whole 16-byte
  // chunks go to the row-group / direct kernels, which read them as chunks.
  // In the spans a lane per row puts the lanes a multiple of 16 bytes apart:
  // 8- to 32-way shared-memory bank conflicts at 32..128-byte rows (256-byte
  // rows took ten times the row-group time), and even with the lanes started
  // at staggered columns the row groups measured faster (bf16 64 columns:
  // cross-entropy 20.7 us against 27.5, softmax backward 12.5 against 29.9).
  // Odd multiples of 4 bytes are conflict-free, 8 mod 16 two-way.
  // Length limits, from timings of each operation on 2^24-element tensors
  // (cold L2) against the row-group / engine kernels for rows of 132 to 404
  // bytes (fp32 33..101 columns, bf16 65..199):
  //  - softmax / log-softmax: up to 448 bytes and 160 columns (fp32 33
  //    columns: log-softmax 46.0 -> 19.4 us; bf16 197 columns lost, 29.4 ->
  //    30.0 us);
  //  - cross-entropy: up to 448 bytes and 200 columns (fp32 33: 63.8 -> 22.6
  //    us, bf16 197: 36.9 -> 30.3 us);
  //  - softmax / log-softmax backward (two tensors per span): up to 224 bytes
  //    (fp32 33: 49.2 -> 29.6 us; even beyond);
  //  - LayerNorm / RMSNorm forward: up to 448 bytes, bf16 up to 128 columns
  //    (fp32 97: 41.5 -> 33.7 us; bf16 131 lost, 32.6 -> 34.9, and 197 lost,
  //    29.3 -> 38.6: a lane's serial pass over that many columns with one
  //    block of spans per SM);
  //  - LayerNorm / RMSNorm backward: up to 64 bytes, bf16 96 (two tensors,
  //    and the column partials' second pass).
  // RR_SPAN_MAX_BYTES replaces these limits by one byte limit for the
  // operations but the norm backward (tuning aid).
  // the norm backward: 64 bytes, bf16 96 (at most 48 columns, two column
  // slots a lane beyond 32; against the phase-class kernel bf16 33 columns
  // 69.7 -> 51.2 us, 47 columns 55.0 against 54.4 us, 63 columns lost, 53.1
  // against 66.6 us; fp32 25 and 31 columns were faster there too, 43.0 /
  // 65.8 against 58.4 / 80.3 us)
  int64_t lim = E == 2 ? 96 : 64, cmax = INT64_MAX;
  switch (mode) {
    case 0: case 1: lim = 448; cmax = 160; break;
    case 2: lim = 448; cmax = 200; break;
    case 3: case 4: lim = 224; break;
    case 5: case 6: lim = 448; cmax = E == 2 ? 128 : INT64_MAX; break;
    default: break;
  }
  if (const char* f = std::getenv("RR_SPAN_MAX_BYTES"); f != nullptr && mode < 7) {
    lim = std::atoll(f);
    cmax = INT64_MAX;
  }
  if (cols > cmax) return RR_ERR_INVALID_ARG;
  const int64_t rb = cols * E;
  if (rb > lim || rb % 16 == 0 || rows <= 0 || max_grid < 1) return RR_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  DevInfo* di = nullptr;
  rr_status st = device_info(&di);
  if (st != RR_OK) return st;
  static const rr::SpanKernelSet ks = rr::span_kernels();
  sp->fn = ks.k[dt][mode];
  // ~3 KB of row data (and staged labels or statistics) per span: large enough
  // per copy, small enough for 3-4 blocks (24-32 warps) per SM
  const bool two = mode == 3 || mode == 4 || mode >= 7;  // two row tensors in
  const int ntens = two ? 2 : 1;
  const int aux = mode == 2 ? 4 : mode >= 7 ? 8 : 0;  // label or statistics bytes per row
  int64_t rpl = 3072 / (32 * (ntens * cols * E + aux));
  if (rpl < 1) rpl = 1;
  const int64_t span_b = 32 * rpl * cols * E;  // a multiple of 16
  int64_t lab_b = (mode == 2 && aux_aligned) ? 32 * rpl * 4 : 0;
  if (mode >= 7) lab_b = 32 * rpl * 4;  // the statistics buffer is always there
  const int nstat = mode >= 7 ? 2 : 1;
  int64_t smem = (int64_t)rr::kSpanWarps * 2 * (ntens * span_b + nstat * lab_b);
  if (mode == 5 || mode == 6) smem += round_up(2 * cols * 4, 16);  // gamma, beta as fp32
  if (mode >= 7) smem += round_up(cols * 4, 16);                   // gamma as fp32
  if (smem > di->smem_optin) return RR_ERR_INVALID_ARG;
  if ((st = set_smem(di, sp->fn, (size_t)smem)) != RR_OK) return st;
  const int T = 32 * rr::kSpanWarps;
  int& occ = di->occ[{sp->fn, ((long long)T << 32) | (long long)smem}];
  if (occ == 0) {
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, sp->fn, T, (size_t)smem);
    if (e != cudaSuccess || occ <= 0)
      return fail(RR_ERR_CUDA, "occupancy query: %s", cudaGetErrorString(e));
  }
  const int64_t nspans = cdiv(rows, 32 * rpl);
  int64_t grid = cdiv(nspans, rr::kSpanWarps);
  if (grid > (int64_t)di->sms * occ) grid = (int64_t)di->sms * occ;
  if (grid > max_grid) grid = max_grid;
  sp->smem = smem;
  sp->grid = grid;
  sp->geo = rr::SpanGeo{rows, (int32_t)cols, (int32_t)rpl, (int32_t)span_b, (int32_t)lab_b,
                        (int32_t)(mode >= 7 && aux_aligned)};
  return RR_OK;
}

template <class P>
rr_status span_launch(const P& p, const SpanPlan& sp, cudaStream_t stream) {
  P pc = p;
  rr::SpanGeo geo = sp.geo;
  void* args[] = {&pc, &geo};
  cudaError_t e = cudaLaunchKernel(sp.fn, dim3((unsigned)sp.grid), dim3(32 * rr::kSpanWarps), args,
                                   (size_t)sp.smem, stream);
  if (e != cudaSuccess) return fail(RR_ERR_CUDA, "span launch: %s", cudaGetErrorString(e));
  return RR_OK;
}

template <class P>
rr_status span_launch(const P& p, rr_dtype dt, int mode, int64_t rows, int64_t cols,
                      bool aux_aligned, cudaStream_t stream) {
  SpanPlan sp;
  rr_status st = span_plan(dt, mode, rows, cols, aux_aligned, INT64_MAX, &sp);
  if (st != RR_OK) return st;
  return span_launch(p, sp, stream);
}

// Rows of one column (rr_one.cuh): elementwise kernels over tiles of
// kOneThreads x (16 / E) rows; as many blocks as are resident on the SMs at
// once (each takes further tiles in turn), at most max_grid (the norm backward
// writes one column partial per block).  Taken when no tier is forced; RR_ONE=0
// turns it off (tuning aid).
struct OnePlan {
  const void* fn = nullptr;
  int64_t grid = 0;
};

static const rr::OneKernels& one_kernels(rr_dtype dt) {
  static const rr::OneKernels f32 = rr::one_kernels_f32();
  static const rr::OneKernels bf16 = rr::one_kernels_bf16();
  return dt == RR_BF16 ? bf16 : f32;
}

static bool one_eligible(int64_t rows, int64_t cols) {
  if (cols != 1 || rows <= 0 || forced_tier() != -1) return false;
  const char* f = std::getenv("RR_ONE");
  return f == nullptr || f[0] != '0';
}

static rr_status one_plan(const void* fn, int64_t rows, int64_t max_grid, OnePlan* op) {
  if (max_grid < 1) return RR_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  DevInfo* di = nullptr;
  rr_status st = device_info(&di);
  if (st != RR_OK) return st;
  const int T = rr::kOneThreads;
  int& occ = di->occ[{fn, (long long)T << 32}];
  if (occ == 0) {
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, T, 0);
    if (e != cudaSuccess || occ <= 0)
      return fail(RR_ERR_CUDA, "occupancy query: %s", cudaGetErrorString(e));
  }
  // tiles of kOneThreads x U rows, U = 16 / E (the norm backward: 4); a
  // block without a tile just exits (the norm backward's partial is then 0)
  int64_t grid = cdiv(rows, T * 4);
  const int64_t resident = (int64_t)di->sms * occ;
  if (grid > resident) grid = resident;
  if (grid > max_grid) grid = max_grid;
  op->fn = fn;
  op->grid = grid;
  return RR_OK;
}

template <class P>
rr_status one_launch(const P& p, const OnePlan& op, int64_t rows, cudaStream_t stream) {
  P pc = p;
  int64_t n = rows;
  void* args[] = {&pc, &n};
  cudaError_t e =
      cudaLaunchKernel(op.fn, dim3((unsigned)op.grid), dim3(rr::kOneThreads), args, 0, stream);
  if (e != cudaSuccess) return fail(RR_ERR_CUDA, "launch: %s", cudaGetErrorString(e));
  return RR_OK;
}

template <class P>
rr_status one_run(const P& p, const void* fn, int64_t rows, cudaStream_t stream) {
  OnePlan op;
  rr_status st = one_plan(fn, rows, INT64_MAX, &op);
  if (st != RR_OK) return st;
  if ((st = one_launch(p, op, rows, stream)) != RR_OK) return st;
  return ok();
}

// LayerNorm / RMSNorm backward of short misaligned rows (rr_lns.cuh): byte
// length 65..1009 and not a multiple of 16 (shorter ones go to the spans; at
// most 64 chunks a row, whatever its offset),
// dy, x and dx at the same address modulo 16 (x's is hb0).  The variant is
// the narrowest that holds the longest chunk span of a row: four rows per warp
// up to 8 chunks, two up to 16, then one row per warp with one or two (fp32
// only) chunks a lane.  As
// many blocks as are resident, at most max_partials (one column partial each).
// RR_LNS=0 turns these kernels off; RR_LNS_V=0..3 forces a variant (tuning
// aids).
struct LnsPlan {
  const void* fn = nullptr;
  int64_t grid = 0;
  size_t smem = 0;
  rr::LnsGeo geo{};
};

static const rr::LnsKernels& lns_kernels(rr_dtype dt) {
  static const rr::LnsKernels f32 = rr::lns_kernels_f32();
  static const rr::LnsKernels bf16 = rr::lns_kernels_bf16();
  return dt == RR_BF16 ? bf16 : f32;
}

static rr_status lns_plan(bool rms, rr_dtype dt, int64_t rows, int64_t cols, int hb0,
                          int64_t max_partials, LnsPlan* lp) {
  if (const char* f = std::getenv("RR_LNS"); f != nullptr && f[0] == '0')
    return RR_ERR_INVALID_ARG;
  const int64_t E = dt == RR_BF16 ? 2 : 4;
  const int64_t rb = cols * E;
  if (rb % 16 == 0 || rb <= 64 || rb > 1024 || rows < 1 || max_partials < 1)
    return RR_ERR_INVALID_ARG;
  int64_t a = 16, b = rb % 16;
  while (b) {
    const int64_t t = a % b;
    a = b;
    b = t;
  }
  const int64_t P = 16 / a;  // 2, 4 or 8 for 2- and 4-byte elements: divides kLnsWarps
  const int64_t nch_max = (rb + 15 + 15) / 16;  // chunks a row touches at worst
  if (nch_max > 64) return RR_ERR_INVALID_ARG;
  static constexpr int64_t kCap[4] = {8, 16, 32, 64};  // chunks a row each variant holds
  static constexpr int64_t kRpw[4] = {4, 2, 1, 1};      // rows a warp holds at once
  int v = nch_max <= 8 ? 0 : nch_max <= 16 ? 1 : nch_max <= 32 ? 2 : 3;
  // Measured on 2^24-element tensors against the row-group kernels: fp32 rows
  // won at every length tried (17 columns 128.0 -> 118.5 us, 45: 91.6 -> 51.3,
  // 97: 76.1 -> 45.6, 127: 60.6 -> 57.1, 250: 58.6 -> 35.5; LayerNorm), so
  // fp32 takes every row that fits.  bf16 rows won where at least 3/4 of the
  // variant's chunk slots hold a chunk (97 columns, 14 of 16: 61.3 -> 51.8
  // us) and lost below (33 columns 85.7 -> 126.9 us, 59: 54.2 -> 79.1, 123,
  // 17 of 32: 52.2 -> 89.1): a bf16 chunk is eight columns, so the per-lane
  // arrays and the element-wise head and tail chunks cost twice as much.
  // bf16 rows of more than 32 chunks are left out: a two-chunk variant needs
  // ~170 registers there (500 columns 37.0 -> 62.8 us) and is not built.
  bool take = dt == RR_F32 || (4 * nch_max >= 3 * kCap[v] && v < 3);
  if (const char* f = std::getenv("RR_LNS_V"); f != nullptr && f[0] >= '0' && f[0] <= '3') {
    const int fv = f[0] - '0';
    if (nch_max <= kCap[fv] && !(dt == RR_BF16 && fv >= 3)) {
      v = fv;
      take = true;
    }
  }
  if (!take) return RR_ERR_INVALID_ARG;
  const void* fn = lns_kernels(dt).bwd[rms ? 1 : 0][v];
  const size_t smem = (size_t)rr::kLnsWarps * (rms ? 1 : 2) * (size_t)cols * sizeof(float);
  std::lock_guard<std::mutex> lock(g_mu);
  DevInfo* di = nullptr;
  rr_status st = device_info(&di);
  if (st != RR_OK) return st;
  if ((int64_t)smem > di->smem_optin) return RR_ERR_INVALID_ARG;
  if ((st = set_smem(di, fn, smem)) != RR_OK) return st;
  const int T = 32 * rr::kLnsWarps;
  int& occ = di->occ[{fn, ((long long)T << 32) | (long long)smem}];
  if (occ == 0) {
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, T, smem);
    if (e != cudaSuccess || occ <= 0)
      return fail(RR_ERR_CUDA, "occupancy query: %s", cudaGetErrorString(e));
  }
  const int64_t rpw = kRpw[v];
  int64_t grid = cdiv(rows, rpw * rr::kLnsWarps);
  if (grid > (int64_t)di->sms * occ) grid = (int64_t)di->sms * occ;
  if (grid > max_partials) grid = max_partials;
  lp->fn = fn;
  lp->grid = grid;
  lp->smem = smem;
  lp->geo = rr::LnsGeo{rows, (int32_t)cols, (int32_t)P, hb0, (int32_t)rb};
  return RR_OK;
}

template <class P>
rr_status launch(const Plan& pl, const P& params, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3((unsigned)pl.grid);
  cfg.blockDim = dim3((unsigned)pl.T);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = stream;
  cfg.numAttrs = 0;
  if (pl.K > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = pl.K;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  P pcopy = params;
  rr::Geo g = pl.geo;
  rr::LnGeo lg = pl.lgeo;
  rr::LnxGeo xg = pl.xgeo;
  void* args[] = {&pcopy, pl.kind == 2   ? static_cast<void*>(&xg)
                          : pl.kind == 1 ? static_cast<void*>(&lg)
                                         : static_cast<void*>(&g)};
  cudaError_t e = cudaLaunchKernelExC(&cfg, pl.fn, args);
  if (e != cudaSuccess)
    return fail(RR_ERR_CUDA, "launch (grid %lld, block %d, smem %zu, cluster %d): %s",
                (long long)pl.grid, pl.T, pl.smem, pl.K, cudaGetErrorString(e));
  return RR_OK;
}

// ------------------------------------------------------------- checks ----

// Whether [a, a + na) and [b, b + nb) share a byte (an absent, null, tensor
// overlaps nothing).
bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
  return a && b && na && nb && pa < pb + nb && pb < pa + na;
}
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

rr_status check_shape(int64_t rows, int64_t cols, rr_dtype dt) {
  if (dt != RR_F32 && dt != RR_BF16) return fail(RR_ERR_UNSUPPORTED_DTYPE, "dtype %d", (int)dt);
  if (rows < 0) return fail(RR_ERR_INVALID_ARG, "rows=%lld < 0", (long long)rows);
  if (cols < 1) return fail(RR_ERR_INVALID_ARG, "cols=%lld < 1", (long long)cols);
  if (cols > ((int64_t)1 << 31) || (rows > 0 && cols > (((int64_t)1 << 60) / rows)))
    return fail(RR_ERR_INVALID_ARG, "rows*cols too large");
  return RR_OK;
}

int* device_error_word() {
  std::lock_guard<std::mutex> lock(g_mu);
  DevInfo* di = nullptr;
  if (device_info(&di) != RR_OK) return nullptr;
  return di->err;
}

}  // namespace

// Lets the other translation units of the library report a detail string.
void rr_set_error_detail(const char* msg) { g_detail = msg ? msg : ""; }

extern "C" {

const char* rr_status_string(rr_status s) {
  switch (s) {
    case RR_OK: return "RR_OK";
    case RR_ERR_INVALID_ARG: return "RR_ERR_INVALID_ARG";
    case RR_ERR_UNSUPPORTED_DTYPE: return "RR_ERR_UNSUPPORTED_DTYPE";
    case RR_ERR_ALIASING: return "RR_ERR_ALIASING";
    case RR_ERR_WORKSPACE_TOO_SMALL: return "RR_ERR_WORKSPACE_TOO_SMALL";
    case RR_ERR_CUDA: return "RR_ERR_CUDA";
    case RR_ERR_DEVICE_TIMEOUT: return "RR_ERR_DEVICE_TIMEOUT";
  }
  return "RR_UNKNOWN_STATUS";
}

const char* rr_last_error_detail(void) { return g_detail.c_str(); }

static rr_status softmax_fwd_impl(const void* x, void* y, int64_t rows, int64_t cols,
                                  rr_dtype dtype, cudaStream_t stream, int32_t log) {
  rr_status st = check_shape(rows, cols, dtype);
  if (st != RR_OK) return st;
  if (rows == 0) return ok();
  if (!x || !y) return fail(RR_ERR_INVALID_ARG, "null pointer");
  const size_t E = dtype == RR_BF16 ? 2 : 4;
  if (!aligned(x, E) || !aligned(y, E)) return fail(RR_ERR_INVALID_ARG, "misaligned element pointer");
  const size_t n = (size_t)rows * cols * E;
  if (x != y && overlaps(x, n, y, n)) return fail(RR_ERR_ALIASING, "x and y partially overlap");
  const bool same = (reinterpret_cast<uintptr_t>(x) & 15) == (reinterpret_cast<uintptr_t>(y) & 15);
  const bool head_free = same && aligned(x, 16) && (cols * E) % 16 == 0;
  int* err = device_error_word();
  if (!err) return RR_ERR_CUDA;
  rr::SoftmaxParams p{static_cast<const char*>(x), static_cast<char*>(y), nullptr, nullptr, nullptr,
                      err, cols, 0, log};
  const int ft = forced_tier();
  if (ft == -2) return bad_tier();
  if (one_eligible(rows, cols))
    return one_run(p, one_kernels(dtype).fwd[log ? 1 : 0], rows, stream);
  if (ft <= 0 && aligned(x, 16) && aligned(y, 16)) {
    st = span_launch(p, dtype, log ? 1 : 0, rows, cols, false, stream);
    if (st != RR_ERR_INVALID_ARG) return st == RR_OK ? ok() : st;
  }
  if (ft == 0) return no_span(cols);
  Plan pl;
  // x and y at the same address modulo 16: phase-aligned kernels for long rows
  st = RR_ERR_INVALID_ARG;
  if (same && (ft < 0 || ft == 1 || ft == 3))
    st = lnx_plan(kSoftmax, dtype, rows, cols, &pl, INT64_MAX, ft, log ? 1 : 0);
  if (st == RR_ERR_INVALID_ARG)
    st = plan_any(kSoftmax, dtype, same, head_free, rows, cols, &pl, INT64_MAX, ft);
  if (st != RR_OK) return st;
  if ((st = launch(pl, p, stream)) != RR_OK) return st;
  return ok();
}

rr_status rr_softmax_fwd(const void* x, void* y, int64_t rows, int64_t cols, rr_dtype dtype,
                         cudaStream_t stream) {
  return softmax_fwd_impl(x, y, rows, cols, dtype, stream, 0);
}

rr_status rr_log_softmax_fwd(const void* x, void* z, int64_t rows, int64_t cols, rr_dtype dtype,
                             cudaStream_t stream) {
  return softmax_fwd_impl(x, z, rows, cols, dtype, stream, 1);
}

// Softmax (log = 0: y, dy) or log-softmax (log = 1: z, dz) backward.  dx may be
// either input exactly (each row is read whole before it is written).
static rr_status softmax_bwd_impl(const void* y, const void* dy, void* dx, int64_t rows,
                                  int64_t cols, rr_dtype dtype, cudaStream_t stream, int32_t log) {
  rr_status st = check_shape(rows, cols, dtype);
  if (st != RR_OK) return st;
  if (rows == 0) return ok();
  if (!y || !dy || !dx) return fail(RR_ERR_INVALID_ARG, "null pointer");
  const size_t E = dtype == RR_BF16 ? 2 : 4;
  if (!aligned(y, E) || !aligned(dy, E) || !aligned(dx, E))
    return fail(RR_ERR_INVALID_ARG, "misaligned element pointer");
  const size_t n = (size_t)rows * cols * E;
  if ((dx != y && overlaps(dx, n, y, n)) || (dx != dy && overlaps(dx, n, dy, n)))
    return fail(RR_ERR_ALIASING, "dx partially overlaps an input");
  // memory-aligned chunks hold the same columns of all three tensors only when
  // they share their alignment; otherwise element mode
  const uintptr_t a = reinterpret_cast<uintptr_t>(y) & 15;
  const bool same = a == (reinterpret_cast<uintptr_t>(dy) & 15) &&
                    a == (reinterpret_cast<uintptr_t>(dx) & 15);
  const bool head_free = same && a == 0 && (cols * E) % 16 == 0;
  int* err = device_error_word();
  if (!err) return RR_ERR_CUDA;
  rr::SoftmaxBwdParams p{static_cast<const char*>(y), static_cast<const char*>(dy),
                         static_cast<char*>(dx), err, cols, log};
  const int ft = forced_tier();
  if (ft == -2) return bad_tier();
  if (one_eligible(rows, cols))
    return one_run(p, one_kernels(dtype).bwd[log ? 1 : 0], rows, stream);
  if (ft <= 0 && same && a == 0) {
    st = span_launch(p, dtype, log ? 4 : 3, rows, cols, false, stream);
    if (st != RR_ERR_INVALID_ARG) return st == RR_OK ? ok() : st;
  }
  if (ft == 0) return no_span(cols);
  Plan pl;
  // the three tensors at the same address modulo 16: phase-class kernels for
  // long rows
  st = RR_ERR_INVALID_ARG;
  if (same && (ft < 0 || ft == 1 || ft == 3))
    st = lnx_plan(kSoftmaxBwd, dtype, rows, cols, &pl, INT64_MAX, ft, log ? 1 : 0);
  if (st == RR_ERR_INVALID_ARG)
    st = plan_any(kSoftmaxBwd, dtype, same, head_free, rows, cols, &pl, INT64_MAX, ft);
  if (st != RR_OK) return st;
  if ((st = launch(pl, p, stream)) != RR_OK) return st;
  return ok();
}

rr_status rr_softmax_bwd(const void* y, const void* dy, void* dx, int64_t rows, int64_t cols,
                         rr_dtype dtype, cudaStream_t stream) {
  return softmax_bwd_impl(y, dy, dx, rows, cols, dtype, stream, 0);
}

rr_status rr_log_softmax_bwd(const void* z, const void* dz, void* dx, int64_t rows, int64_t cols,
                             rr_dtype dtype, cudaStream_t stream) {
  return softmax_bwd_impl(z, dz, dx, rows, cols, dtype, stream, 1);
}

rr_status rr_softmax_xent_fwd_bwd(const void* logits, const int32_t* labels, float* loss,
                                  void* dlogits, int64_t rows, int64_t cols, int32_t ignore_index,
                                  int32_t* bad_label_count, rr_dtype dtype, cudaStream_t stream) {
  rr_status st = check_shape(rows, cols, dtype);
  if (st != RR_OK) return st;
  if (rows == 0) return ok();
  if (!logits || !labels || !loss || !dlogits) return fail(RR_ERR_INVALID_ARG, "null pointer");
  const size_t E = dtype == RR_BF16 ? 2 : 4;
  if (!aligned(logits, E) || !aligned(dlogits, E) || !aligned(labels, 4) || !aligned(loss, 4) ||
      (bad_label_count && !aligned(bad_label_count, 4)))
    return fail(RR_ERR_INVALID_ARG, "misaligned pointer");
  const size_t n = (size_t)rows * cols * E, nr = (size_t)rows * 4;
  if (logits != dlogits && overlaps(logits, n, dlogits, n))
    return fail(RR_ERR_ALIASING, "logits and dlogits partially overlap");
  if (overlaps(loss, nr, logits, n) || overlaps(loss, nr, dlogits, n) || overlaps(loss, nr, labels, nr) ||
      overlaps(labels, nr, dlogits, n))
    return fail(RR_ERR_ALIASING, "loss / labels overlap another tensor");
  if (bad_label_count && (overlaps(bad_label_count, 4, logits, n) || overlaps(bad_label_count, 4, dlogits, n) ||
                          overlaps(bad_label_count, 4, loss, nr) || overlaps(bad_label_count, 4, labels, nr)))
    return fail(RR_ERR_ALIASING, "bad_label_count overlaps another tensor");
  const bool same =
      (reinterpret_cast<uintptr_t>(logits) & 15) == (reinterpret_cast<uintptr_t>(dlogits) & 15);
  const bool head_free = same && aligned(logits, 16) && (cols * E) % 16 == 0;
  int* err = device_error_word();
  if (!err) return RR_ERR_CUDA;
  rr::SoftmaxParams p{static_cast<const char*>(logits), static_cast<char*>(dlogits), labels, loss,
                      bad_label_count, err, cols, ignore_index, 0};
  const int ft = forced_tier();
  if (ft == -2) return bad_tier();
  if (one_eligible(rows, cols)) return one_run(p, one_kernels(dtype).fwd[2], rows, stream);
  if (ft <= 0 && aligned(logits, 16) && aligned(dlogits, 16)) {
    st = span_launch(p, dtype, 2, rows, cols, aligned(labels, 16), stream);
    if (st != RR_ERR_INVALID_ARG) return st == RR_OK ? ok() : st;
  }
  if (ft == 0) return no_span(cols);
  Plan pl;
  st = RR_ERR_INVALID_ARG;
  if (same && (ft < 0 || ft == 1 || ft == 3))
    st = lnx_plan(kSoftmax, dtype, rows, cols, &pl, INT64_MAX, ft, 2);
  if (st == RR_ERR_INVALID_ARG)
    st = plan_any(kSoftmax, dtype, same, head_free, rows, cols, &pl, INT64_MAX, ft);
  if (st != RR_OK) return st;
  if ((st = launch(pl, p, stream)) != RR_OK) return st;
  return ok();
}

rr_status rr_layernorm_fwd(const void* x, const void* gamma, const void* beta, void* y, float* mean,
                           float* rstd, int64_t rows, int64_t cols, float eps, rr_dtype dtype,
                           cudaStream_t stream) {
  rr_status st = check_shape(rows, cols, dtype);
  if (st != RR_OK) return st;
  if (!(eps >= 0.f) || !std::isfinite(eps)) return fail(RR_ERR_INVALID_ARG, "eps must be finite and >= 0");
  if (rows == 0) return ok();
  if (!x || !gamma || !beta || !y || !mean || !rstd) return fail(RR_ERR_INVALID_ARG, "null pointer");
  const size_t E = dtype == RR_BF16 ? 2 : 4;
  if (!aligned(x, E) || !aligned(y, E) || !aligned(gamma, E) || !aligned(beta, E) || !aligned(mean, 4) ||
      !aligned(rstd, 4))
    return fail(RR_ERR_INVALID_ARG, "misaligned pointer");
  const size_t n = (size_t)rows * cols * E, nc = (size_t)cols * E, nr = (size_t)rows * 4;
  if (x != y && overlaps(x, n, y, n)) return fail(RR_ERR_ALIASING, "x and y partially overlap");
  if (overlaps(y, n, gamma, nc) || overlaps(y, n, beta, nc) || overlaps(mean, nr, rstd, nr) ||
      overlaps(mean, nr, x, n) || overlaps(mean, nr, y, n) || overlaps(rstd, nr, x, n) ||
      overlaps(rstd, nr, y, n) || overlaps(mean, nr, gamma, nc) || overlaps(mean, nr, beta, nc) ||
      overlaps(rstd, nr, gamma, nc) || overlaps(rstd, nr, beta, nc))
    return fail(RR_ERR_ALIASING, "outputs overlap inputs");
  // column-aligned chunks need 16-byte aligned gamma / beta; rows may have any alignment
  const bool al = aligned(gamma, 16) && aligned(beta, 16);
  const bool rows_al = (cols * (int64_t)E) % 16 == 0 && aligned(x, 16) && aligned(y, 16);
  Plan pl;
  const int lmode = al ? (rows_al ? 0 : 1) : 2;
  const int ft = forced_tier();
  if (ft == -2) return bad_tier();
  {
    int* err = device_error_word();
    if (!err) return RR_ERR_CUDA;
    rr::LnFwdParams p{static_cast<const char*>(x), static_cast<const char*>(gamma),
                      static_cast<const char*>(beta), static_cast<char*>(y), mean, rstd, err, cols,
                      eps, static_cast<float>(1.0 / static_cast<double>(cols))};
    if (one_eligible(rows, cols))
      return one_run(p, one_kernels(dtype).norm_fwd[0], rows, stream);
    if (ft <= 0 && aligned(x, 16) && aligned(y, 16)) {
      st = span_launch(p, dtype, 5, rows, cols, false, stream);
      if (st != RR_ERR_INVALID_ARG) return st == RR_OK ? ok() : st;
    }
  }
  if (ft == 0) return no_span(cols);
  // x and y at the same address modulo 16: phase-aligned kernels for long rows
  // (column blocks for the longest, when y is a separate tensor)
  const bool same16 = (reinterpret_cast<uintptr_t>(x) & 15) == (reinterpret_cast<uintptr_t>(y) & 15);
  if (same16 && ft < 0) {
    LncPlan lp;
    st = lnc_plan(false, false, dtype, rows, cols, &lp);
    if (st == RR_OK && lnc_fwd_fits(lp, x, y, rows, cols, E)) {
      int* err = device_error_word();
      if (!err) return RR_ERR_CUDA;
      rr::LnFwdParams p{static_cast<const char*>(x), static_cast<const char*>(gamma),
                        static_cast<const char*>(beta), static_cast<char*>(y), mean, rstd, err,
                        cols, eps, static_cast<float>(1.0 / static_cast<double>(cols))};
      if ((st = lnc_forward(false, lp, p, dtype, stream)) != RR_OK) return st;
      return ok();
    }
    if (st != RR_OK && st != RR_ERR_INVALID_ARG) return st;
  }
  st = RR_ERR_INVALID_ARG;
  if (same16 && (ft < 0 || ft == 1 || ft == 3))
    st = lnx_plan(kLnFwd, dtype, rows, cols, &pl, INT64_MAX, ft);
  if (st == RR_ERR_INVALID_ARG && (ft < 0 || ft == 1))
    st = ln_rowgroup_plan(kLnFwd, dtype, lmode, rows, cols, &pl, INT64_MAX);
  if (st == RR_ERR_INVALID_ARG && (ft < 0 || ft == 3))
    st = ln_cluster_plan(kLnFwd, dtype, lmode, rows, cols, &pl);
  if (st == RR_ERR_INVALID_ARG && (ft < 0 || ft == 2))
    st = plan_any(kLnFwd, dtype, al, true, rows, cols, &pl, INT64_MAX, ft < 0 ? -1 : 2);
  if (st != RR_OK) return st;
  int* err = device_error_word();
  if (!err) return RR_ERR_CUDA;
  rr::LnFwdParams p{static_cast<const char*>(x), static_cast<const char*>(gamma),
                    static_cast<const char*>(beta), static_cast<char*>(y), mean, rstd, err, cols, eps,
                    static_cast<float>(1.0 / static_cast<double>(cols))};
  if ((st = launch(pl, p, stream)) != RR_OK) return st;
  return ok();
}

rr_status rr_rmsnorm_fwd(const void* x, const void* gamma, void* y, float* rstd, int64_t rows,
                         int64_t cols, float eps, rr_dtype dtype, cudaStream_t stream) {
  rr_status st = check_shape(rows, cols, dtype);
  if (st != RR_OK) return st;
  if (!(eps >= 0.f) || !std::isfinite(eps)) return fail(RR_ERR_INVALID_ARG, "eps must be finite and >= 0");
  if (rows == 0) return ok();
  if (!x || !gamma || !y || !rstd) return fail(RR_ERR_INVALID_ARG, "null pointer");
  const size_t E = dtype == RR_BF16 ? 2 : 4;
  if (!aligned(x, E) || !aligned(y, E) || !aligned(gamma, E) || !aligned(rstd, 4))
    return fail(RR_ERR_INVALID_ARG, "misaligned pointer");
  const size_t n = (size_t)rows * cols * E, nc = (size_t)cols * E, nr = (size_t)rows * 4;
  if (x != y && overlaps(x, n, y, n)) return fail(RR_ERR_ALIASING, "x and y partially overlap");
  if (overlaps(y, n, gamma, nc) || overlaps(rstd, nr, x, n) || overlaps(rstd, nr, y, n) ||
      overlaps(rstd, nr, gamma, nc))
    return fail(RR_ERR_ALIASING, "outputs overlap inputs");
  const bool al = aligned(gamma, 16);
  const bool rows_al = (cols * (int64_t)E) % 16 == 0 && aligned(x, 16) && aligned(y, 16);
  Plan pl;
  const int lmode = al ? (rows_al ? 0 : 1) : 2;
  const int ft = forced_tier();
  if (ft == -2) return bad_tier();
  if (ft == 2) return fail(RR_ERR_INVALID_ARG, "tier 2 (staged rows) has no RMSNorm kernel");
  {
    int* err = device_error_word();
    if (!err) return RR_ERR_CUDA;
    rr::LnFwdParams p{static_cast<const char*>(x), static_cast<const char*>(gamma), nullptr,
                      static_cast<char*>(y), nullptr, rstd, err, cols, eps,
                      static_cast<float>(1.0 / static_cast<double>(cols))};
    if (one_eligible(rows, cols))
      return one_run(p, one_kernels(dtype).norm_fwd[1], rows, stream);
    if (ft <= 0 && aligned(x, 16) && aligned(y, 16)) {
      st = span_launch(p, dtype, 6, rows, cols, false, stream);
      if (st != RR_ERR_INVALID_ARG) return st == RR_OK ? ok() : st;
    }
  }
  if (ft == 0) return no_span(cols);
  const bool same16 = (reinterpret_cast<uintptr_t>(x) & 15) == (reinterpret_cast<uintptr_t>(y) & 15);
  if (same16 && ft < 0) {
    LncPlan lp;
    st = lnc_plan(false, true, dtype, rows, cols, &lp);
    if (st == RR_OK && lnc_fwd_fits(lp, x, y, rows, cols, E)) {
      int* err = device_error_word();
      if (!err) return RR_ERR_CUDA;
      rr::LnFwdParams p{static_cast<const char*>(x), static_cast<const char*>(gamma), nullptr,
                        static_cast<char*>(y), nullptr, rstd, err, cols, eps,
                        static_cast<float>(1.0 / static_cast<double>(cols))};
      if ((st = lnc_forward(true, lp, p, dtype, stream)) != RR_OK) return st;
      return ok();
    }
    if (st != RR_OK && st != RR_ERR_INVALID_ARG) return st;
  }
  st = RR_ERR_INVALID_ARG;
  if (same16 && (ft < 0 || ft == 1 || ft == 3))
    st = lnx_plan(kRmsFwd, dtype, rows, cols, &pl, INT64_MAX, ft);
  if (st == RR_ERR_INVALID_ARG && (ft < 0 || ft == 1))
    st = ln_rowgroup_plan(kRmsFwd, dtype, lmode, rows, cols, &pl, INT64_MAX);
  if (st == RR_ERR_INVALID_ARG && (ft < 0 || ft == 3))
    st = ln_cluster_plan(kRmsFwd, dtype, lmode, rows, cols, &pl);
  if (ft >= 1 && st != RR_OK) return st;
  if (st == RR_ERR_INVALID_ARG)
    return fail(RR_ERR_INVALID_ARG,
                "RMSNorm rows of %lld columns fit neither one row group nor a cluster of 8 of them",
                (long long)cols);
  if (st != RR_OK) return st;
  int* err = device_error_word();
  if (!err) return RR_ERR_CUDA;
  rr::LnFwdParams p{static_cast<const char*>(x), static_cast<const char*>(gamma), nullptr,
                    static_cast<char*>(y), nullptr, rstd, err, cols, eps,
                    static_cast<float>(1.0 / static_cast<double>(cols))};
  if ((st = launch(pl, p, stream)) != RR_OK) return st;
  return ok();
}

// Backward plan of LayerNorm (rms = false) or RMSNorm.  lmode as for
// ln_rowgroup_plan; LayerNorm rows too long for one row group go to the staged
// engine kernels (chunk mode unless lmode == 2).  ws_bytes: the column
// partials, [partials][planes][cols] floats.
static rr_status norm_bwd_plan(bool rms, int64_t rows, int64_t cols, rr_dtype dtype, int lmode,
                               bool lnx_ok, Plan* pl, size_t* ws_bytes,
                               int64_t max_partials = INT64_MAX) {
  const int ft = forced_tier();
  if (ft == -2) return bad_tier();
  if (ft == 0) return no_span(cols);
  if (rms && ft == 2)
    return fail(RR_ERR_INVALID_ARG, "tier 2 (staged rows) has no RMSNorm backward kernel");
  rr_status st = RR_ERR_INVALID_ARG;
  // dy, x and dx at the same address modulo 16: phase-aligned kernels for long rows
  if (lnx_ok && (ft < 0 || ft == 1 || ft == 3))
    st = lnx_plan(rms ? kRmsBwd : kLnBwd, dtype, rows, cols, pl, max_partials, ft);
  if (st == RR_ERR_INVALID_ARG && (ft < 0 || ft == 1))
    st = ln_rowgroup_plan(rms ? kRmsBwd : kLnBwd, dtype, lmode, rows, cols, pl, max_partials);
  // rows longer than one row group: clusters of row groups (chunk mode)
  if (st == RR_ERR_INVALID_ARG && (ft < 0 || ft == 3))
    st = ln_cluster_plan(rms ? kRmsBwd : kLnBwd, dtype, lmode, rows, cols, pl, max_partials);
  if (st == RR_ERR_INVALID_ARG && ft != 1) {
    if (rms)
      return fail(RR_ERR_INVALID_ARG,
                  "RMSNorm backward rows of %lld columns fit neither one row group nor a "
                  "cluster of them (16-byte aligned gamma)", (long long)cols);
    st = plan_any(kLnBwd, dtype, lmode != 2, true, rows, cols, pl, max_partials, ft < 0 ? -1 : ft);
  }
  if (st != RR_OK) return st;
  *ws_bytes = (size_t)pl->partials * (rms ? 1 : 2) * (size_t)cols * sizeof(float);
  return RR_OK;
}

static size_t norm_bwd_workspace_size(bool rms, int64_t rows, int64_t cols, rr_dtype dtype) {
  if (check_shape(rows, cols, dtype) != RR_OK) return 0;
  if (rows == 0) return (rms ? 1 : 2) * (size_t)cols * sizeof(float);
  // The caller does not know which mode the pointers will select (aligned or
  // misaligned chunks, elements: different shared memory, so different
  // occupancy and grid), so report the largest of the three.
  size_t best = 0;
  for (int lnx = 0; lnx < 2; ++lnx)
    for (int m = 0; m < 3; ++m) {
      Plan pl;
      size_t ws = 0;
      if (norm_bwd_plan(rms, rows, cols, dtype, m, lnx == 1, &pl, &ws) == RR_OK && ws > best)
        best = ws;
    }
  if (forced_tier() < 0) {  // the column-block kernels (partials and row records)
    LncPlan lp;
    if (lnc_plan(true, rms, dtype, rows, cols, &lp) == RR_OK && lp.ws_bytes > best) best = lp.ws_bytes;
  }
  LnsPlan sp2;  // short misaligned rows by phase class: one partial per block
  if (forced_tier() < 0 && lns_plan(rms, dtype, rows, cols, 0, INT64_MAX, &sp2) == RR_OK) {
    const size_t ws = (size_t)sp2.grid * (rms ? 1 : 2) * (size_t)cols * sizeof(float);
    if (ws > best) best = ws;
  }
  OnePlan op;  // rows of one column: one partial per block
  if (one_eligible(rows, cols) &&
      one_plan(one_kernels(dtype).norm_bwd[rms], rows, INT64_MAX, &op) == RR_OK) {
    const size_t ws = (size_t)op.grid * (rms ? 1 : 2) * sizeof(float);
    if (ws > best) best = ws;
  }
  SpanPlan sp;  // short rows with 16-byte aligned tensors: one partial per span block
  if (forced_tier() <= 0 && span_plan(dtype, rms ? 8 : 7, rows, cols, false, INT64_MAX, &sp) == RR_OK) {
    const size_t ws = (size_t)sp.grid * (rms ? 1 : 2) * (size_t)cols * sizeof(float);
    if (ws > best) best = ws;
  }
  return best;
}

size_t rr_layernorm_bwd_workspace_size(int64_t rows, int64_t cols, rr_dtype dtype) {
  return norm_bwd_workspace_size(false, rows, cols, dtype);
}

size_t rr_rmsnorm_bwd_workspace_size(int64_t rows, int64_t cols, rr_dtype dtype) {
  return norm_bwd_workspace_size(true, rows, cols, dtype);
}

}  // extern "C"

// Host-side argument checks of the LayerNorm (rms = false) or RMSNorm
// backward: shape, dtype, null pointers, alignment and overlap.  No device
// call.  check_ws = false skips the workspace (the no-allocation entry point's
// scratch lives inside the library and cannot overlap a caller's tensor).
static rr_status norm_bwd_check(bool rms, const void* dy, const void* x, const float* mean,
                                const float* rstd, const void* gamma, const void* dx,
                                const void* dgamma, const void* dbeta, const void* workspace,
                                size_t workspace_bytes, int64_t rows, int64_t cols, rr_dtype dtype,
                                bool check_ws) {
  rr_status st = check_shape(rows, cols, dtype);
  if (st != RR_OK) return st;
  if (!dy || !x || (!rms && !mean) || !rstd || !gamma || !dx || !dgamma || (!rms && !dbeta) ||
      (check_ws && !workspace))
    return fail(RR_ERR_INVALID_ARG, "null pointer");
  const size_t E = dtype == RR_BF16 ? 2 : 4;
  if (!aligned(dy, E) || !aligned(x, E) || !aligned(dx, E) || !aligned(gamma, E) || !aligned(dgamma, E) ||
      !aligned(dbeta, E) || !aligned(mean, 4) || !aligned(rstd, 4) ||
      (check_ws && !aligned(workspace, 16)))
    return fail(RR_ERR_INVALID_ARG, "misaligned pointer (workspace needs 16 bytes)");
  const size_t n = (size_t)rows * cols * E, nc = (size_t)cols * E, nr = (size_t)rows * 4;
  if (dx != dy && overlaps(dx, n, dy, n)) return fail(RR_ERR_ALIASING, "dx and dy partially overlap");
  if (dx != x && overlaps(dx, n, x, n)) return fail(RR_ERR_ALIASING, "dx and x partially overlap");
  const void* outs[] = {dgamma, dbeta, check_ws ? workspace : nullptr};
  const size_t outn[] = {nc, nc, workspace_bytes};
  const void* ins[] = {dy, x, mean, rstd, gamma, dx};
  const size_t inn[] = {n, n, nr, nr, nc, n};
  for (int i = 0; i < 3; ++i) {
    for (int j = 0; j < 6; ++j)
      if (overlaps(outs[i], outn[i], ins[j], inn[j])) return fail(RR_ERR_ALIASING, "output overlaps an input");
    for (int j = i + 1; j < 3; ++j)
      if (overlaps(outs[i], outn[i], outs[j], outn[j])) return fail(RR_ERR_ALIASING, "outputs overlap");
  }
  if (overlaps(dx, n, mean, nr) || overlaps(dx, n, rstd, nr) || overlaps(dx, n, gamma, nc))
    return fail(RR_ERR_ALIASING, "dx overlaps mean / rstd / gamma");
  return RR_OK;
}

// LayerNorm (rms = false) or RMSNorm backward with at most max_partials column
// partials (the no-allocation entry point sizes this to its fixed scratch).
// RMSNorm has no mean and no dbeta (both null).
static rr_status norm_bwd(bool rms, const void* dy, const void* x, const float* mean,
                          const float* rstd, const void* gamma, void* dx, void* dgamma, void* dbeta,
                          void* workspace, size_t workspace_bytes, int64_t rows, int64_t cols,
                          rr_dtype dtype, cudaStream_t stream, int64_t max_partials) {
  rr_status st = norm_bwd_check(rms, dy, x, mean, rstd, gamma, dx, dgamma, dbeta, workspace,
                                workspace_bytes, rows, cols, dtype, true);
  if (st != RR_OK) return st;
  const size_t E = dtype == RR_BF16 ? 2 : 4;
  const int64_t planes = rms ? 1 : 2;
  const bool al = aligned(gamma, 16);
  Plan pl;
  size_t need = 0;
  if (rows == 0) {
    // Nothing to read: dgamma = dbeta = 0 through a one-partial workspace.
    need = planes * (size_t)cols * sizeof(float);
    if (workspace_bytes < need)
      return fail(RR_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu bytes", workspace_bytes, need);
    cudaError_t e = cudaMemsetAsync(workspace, 0, need, stream);
    if (e != cudaSuccess) return fail(RR_ERR_CUDA, "memset: %s", cudaGetErrorString(e));
    pl.partials = 1;
  } else {
    const bool rows_al = (cols * (int64_t)E) % 16 == 0 && aligned(dy, 16) && aligned(x, 16) &&
                         aligned(dx, 16);
    const int lmode = al ? (rows_al ? 0 : 1) : 2;
    int* err = device_error_word();
    if (!err) return RR_ERR_CUDA;
    rr::LnBwdParams p{static_cast<const char*>(dy), static_cast<const char*>(x), mean, rstd,
                      static_cast<const char*>(gamma), static_cast<char*>(dx),
                      static_cast<float*>(workspace), err, cols,
                      static_cast<float>(1.0 / static_cast<double>(cols))};
    SpanPlan sp;
    st = RR_ERR_INVALID_ARG;
    const int ft = forced_tier();
    // rows of one column: elementwise, one partial per block
    OnePlan op;
    const bool one = one_eligible(rows, cols);
    if (one &&
        (st = one_plan(one_kernels(dtype).norm_bwd[rms], rows, max_partials, &op)) != RR_OK)
      return st;
    if (!one && ft <= 0 && aligned(dy, 16) && aligned(x, 16) && aligned(dx, 16)) {
      const bool stats_al = aligned(rstd, 16) && (rms || aligned(mean, 16));
      st = span_plan(dtype, rms ? 8 : 7, rows, cols, stats_al, max_partials, &sp);
      if (st != RR_OK && st != RR_ERR_INVALID_ARG) return st;
    }
    if (one) {
      need = (size_t)op.grid * planes * sizeof(float);
      if (workspace_bytes < need)
        return fail(RR_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu bytes", workspace_bytes, need);
      if ((st = one_launch(p, op, rows, stream)) != RR_OK) return st;
      pl.partials = op.grid;
    } else if (st == RR_OK) {
      need = (size_t)sp.grid * planes * (size_t)cols * sizeof(float);
      if (workspace_bytes < need)
        return fail(RR_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu bytes", workspace_bytes, need);
      if ((st = span_launch(p, sp, stream)) != RR_OK) return st;
      pl.partials = sp.grid;
    } else {
      const uintptr_t a16 = reinterpret_cast<uintptr_t>(x) & 15;
      const bool same16 = a16 == (reinterpret_cast<uintptr_t>(dy) & 15) &&
                          a16 == (reinterpret_cast<uintptr_t>(dx) & 15);
      // short misaligned rows: phase-class warps (one partial per block)
      LnsPlan sp2;
      st = RR_ERR_INVALID_ARG;
      if (same16 && ft < 0) {
        st = lns_plan(rms, dtype, rows, cols, (int)a16, max_partials, &sp2);
        if (st != RR_OK && st != RR_ERR_INVALID_ARG) return st;
      }
      // the longest rows: column-block kernels, where their partials and
      // records fit the workspace
      LncPlan lp;
      const bool lns = st == RR_OK;
      if (!lns && same16 && ft < 0) {
        st = lnc_plan(true, rms, dtype, rows, cols, &lp, max_partials, workspace_bytes);
        if (st != RR_OK && st != RR_ERR_INVALID_ARG) return st;
      }
      if (lns) {
        need = (size_t)sp2.grid * planes * (size_t)cols * sizeof(float);
        if (workspace_bytes < need)
          return fail(RR_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu bytes", workspace_bytes, need);
        rr::LnsGeo g = sp2.geo;
        void* args[] = {&p, &g};
        cudaError_t e = cudaLaunchKernel(sp2.fn, dim3((unsigned)sp2.grid),
                                         dim3(32 * rr::kLnsWarps), args, sp2.smem, stream);
        if (e != cudaSuccess) return fail(RR_ERR_CUDA, "launch: %s", cudaGetErrorString(e));
        pl.partials = sp2.grid;
      } else if (st == RR_OK) {
        const rr::LncKernels& k = lnc_kernels(dtype);
        rr::LncGeo g = lp.geo;
        void* args[] = {&p, &g};
        const size_t ring = (size_t)rr::lnc_ring_bytes(true);
        cudaError_t e = cudaLaunchKernel(k.part[rms], dim3((unsigned)lp.items),
                                         dim3(32 * rr::kLncWarps), args, ring, stream);
        if (e == cudaSuccess)
          e = cudaLaunchKernel(k.dx[rms], dim3((unsigned)lp.items), dim3(32 * rr::kLncWarps),
                               args, ring, stream);
        if (e != cudaSuccess) return fail(RR_ERR_CUDA, "launch: %s", cudaGetErrorString(e));
        pl.partials = lp.partials;
      } else {
        if ((st = norm_bwd_plan(rms, rows, cols, dtype, lmode, same16, &pl, &need, max_partials)) !=
            RR_OK)
          return st;
        if (workspace_bytes < need)
          return fail(RR_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu bytes", workspace_bytes, need);
        if ((st = launch(pl, p, stream)) != RR_OK) return st;
      }
    }
  }
  const void* cr = dtype == RR_BF16 ? rr::col_reduce_kernel_ptr_bf16() : rr::col_reduce_kernel_ptr_f32();
  const float* ws = static_cast<const float*>(workspace);
  int64_t P = pl.partials;
  char* dg = static_cast<char*>(dgamma);
  char* db = static_cast<char*>(dbeta);
  int64_t pl_n = planes;
  void* args[] = {&ws, &P, &cols, &pl_n, &dg, &db};
  cudaError_t e =
      cudaLaunchKernel(cr, dim3((unsigned)cdiv(planes * cols, 32 * (32 / rr::col_reduce_split(P)))),
                       dim3(1024), args, 0, stream);
  if (e != cudaSuccess) return fail(RR_ERR_CUDA, "column reduce launch: %s", cudaGetErrorString(e));
  return ok();
}

// The LayerNorm backward's argument checks without a workspace (no device
// call), for the no-allocation entry point.
rr_status layernorm_bwd_check_args(const void* dy, const void* x, const float* mean,
                                   const float* rstd, const void* gamma, const void* dx,
                                   const void* dgamma, const void* dbeta, int64_t rows,
                                   int64_t cols, rr_dtype dtype) {
  return norm_bwd_check(false, dy, x, mean, rstd, gamma, dx, dgamma, dbeta, nullptr, 0, rows, cols,
                        dtype, false);
}

// rr_layernorm_bwd with at most max_partials column partials (the no-allocation
// entry point sizes this to its fixed scratch).
rr_status layernorm_bwd_capped(const void* dy, const void* x, const float* mean, const float* rstd,
                               const void* gamma, void* dx, void* dgamma, void* dbeta,
                               void* workspace, size_t workspace_bytes, int64_t rows, int64_t cols,
                               rr_dtype dtype, cudaStream_t stream, int64_t max_partials) {
  return norm_bwd(false, dy, x, mean, rstd, gamma, dx, dgamma, dbeta, workspace, workspace_bytes,
                  rows, cols, dtype, stream, max_partials);
}

extern "C" {

rr_status rr_layernorm_bwd(const void* dy, const void* x, const float* mean, const float* rstd,
                           const void* gamma, void* dx, void* dgamma, void* dbeta, void* workspace,
                           size_t workspace_bytes, int64_t rows, int64_t cols, rr_dtype dtype,
                           cudaStream_t stream) {
  return norm_bwd(false, dy, x, mean, rstd, gamma, dx, dgamma, dbeta, workspace, workspace_bytes,
                  rows, cols, dtype, stream, INT64_MAX);
}

rr_status rr_rmsnorm_bwd(const void* dy, const void* x, const float* rstd, const void* gamma,
                         void* dx, void* dgamma, void* workspace, size_t workspace_bytes,
                         int64_t rows, int64_t cols, rr_dtype dtype, cudaStream_t stream) {
  return norm_bwd(true, dy, x, nullptr, rstd, gamma, dx, dgamma, nullptr, workspace,
                  workspace_bytes, rows, cols, dtype, stream, INT64_MAX);
}

rr_status rr_attention_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                           int64_t bh, int64_t seq, int64_t head_dim, float scale, int causal,
                           rr_dtype dtype, cudaStream_t stream) {
  if (dtype != RR_BF16)
    return fail(RR_ERR_UNSUPPORTED_DTYPE, "attention takes bf16 q, k, v (tensor-core path)");
  if (bh < 0 || seq < 0) return fail(RR_ERR_INVALID_ARG, "negative size");
  if (bh == 0 || seq == 0) return ok();
  if (seq % 64 != 0) return fail(RR_ERR_INVALID_ARG, "seq must be a multiple of 64");
  if (bh > INT32_MAX) return fail(RR_ERR_INVALID_ARG, "too many heads per call");
  if (seq > (int64_t)64 * 65535) return fail(RR_ERR_INVALID_ARG, "seq too long");
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(RR_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (!q || !k || !v || !o) return fail(RR_ERR_INVALID_ARG, "null pointer");
  const rr::AttnKernel ak = rr::attn_fwd_kernel_for((int)head_dim);
  if (ak.fn == nullptr) return fail(RR_ERR_INVALID_ARG, "head_dim must be 64 or 128");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      (lse != nullptr && !aligned(lse, 4)))
    return fail(RR_ERR_INVALID_ARG, "q, k, v, o must be 16-byte aligned");
  const size_t n = (size_t)bh * seq * head_dim * 2, nl = (size_t)bh * seq * 4;
  if (overlaps(o, n, q, n) || overlaps(o, n, k, n) || overlaps(o, n, v, n))
    return fail(RR_ERR_ALIASING, "o overlaps q, k or v");
  if (lse != nullptr && (overlaps(lse, nl, q, n) || overlaps(lse, nl, k, n) ||
                         overlaps(lse, nl, v, n) || overlaps(lse, nl, o, n)))
    return fail(RR_ERR_ALIASING, "lse overlaps a tensor");
  int sms = 0;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    DevInfo* di = nullptr;
    rr_status st = device_info(&di);
    if (st != RR_OK) return st;
    if (ak.smem > di->smem_optin) return fail(RR_ERR_INVALID_ARG, "attention tile exceeds shared memory");
    if ((st = set_smem(di, ak.fn, (size_t)ak.smem)) != RR_OK) return st;
    sms = di->sms;
  }
  int* err = device_error_word();
  if (!err) return RR_ERR_CUDA;
  rr::AttnParams p{static_cast<const char*>(q), static_cast<const char*>(k),
                   static_cast<const char*>(v), static_cast<char*>(o), lse, err, bh, seq,
                   scale * 1.4426950408889634f, causal ? 1 : 0};
  if (const char* why = rr::attn_fwd_launch(p, (int)head_dim, sms, stream)) {
    cudaError_t e = cudaGetLastError();
    return fail(RR_ERR_CUDA, "attention: %s (%s)", why, cudaGetErrorString(e));
  }
  return ok();
}

}  // extern "C"

namespace {

// One thread arms an mbarrier for 16 transaction bytes that no copy delivers
// and waits on it with the kernels' bounded wait; the wait gives up after
// limit_ns, records RR_ERR_DEVICE_TIMEOUT in *err and the block returns.
__global__ void selftest_wait_kernel(int* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  rr::mbar_init(&bar, 1);
  rr::fence_mbar_init();
  rr::mbar_arrive_expect_tx(&bar, 16);
  rr::mbar_wait_bounded(&bar, 0, err, limit_ns);
}

}  // namespace

extern "C" {

rr_status rr_selftest_bounded_wait(int64_t limit_ns, cudaStream_t stream) {
  if (limit_ns < 1 || limit_ns > 1000000000LL)
    return fail(RR_ERR_INVALID_ARG, "limit_ns must be in [1, 1e9]");
  int* err = device_error_word();
  if (!err) return RR_ERR_CUDA;
  selftest_wait_kernel<<<1, 32, 0, stream>>>(err, (uint64_t)limit_ns);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(RR_ERR_CUDA, "self-test launch: %s", cudaGetErrorString(e));
  return ok();
}

rr_status rr_read_device_error(int device, int* value, int reset) {
  if (!value) return fail(RR_ERR_INVALID_ARG, "null pointer");
  int prev = 0;
  cudaError_t e = cudaGetDevice(&prev);
  if (e != cudaSuccess) return fail(RR_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if ((e = cudaSetDevice(device)) != cudaSuccess)
    return fail(RR_ERR_CUDA, "cudaSetDevice(%d): %s", device, cudaGetErrorString(e));
  rr_status st = RR_OK;
  int v = 0;
  if ((e = cudaDeviceSynchronize()) != cudaSuccess ||
      (e = cudaMemcpyFromSymbol(&v, g_rr_device_error, sizeof v)) != cudaSuccess) {
    st = fail(RR_ERR_CUDA, "reading the error word: %s", cudaGetErrorString(e));
  } else if (reset) {
    const int zero = 0;
    if ((e = cudaMemcpyToSymbol(g_rr_device_error, &zero, sizeof zero)) != cudaSuccess)
      st = fail(RR_ERR_CUDA, "clearing the error word: %s", cudaGetErrorString(e));
  }
  cudaSetDevice(prev);
  *value = v;
  return st == RR_OK ? ok() : st;
}

}  // extern "C"
