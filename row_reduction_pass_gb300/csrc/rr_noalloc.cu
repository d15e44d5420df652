// rr_noalloc.cu -- rr_layernorm_bwd_noalloc: the LayerNorm backward for
// callers that cannot allocate device memory when they call it.
//
// rr_layernorm_bwd needs a caller-provided workspace for its column partials.
// Some callers have no way to provide one: code that runs under a framework's
// memory planner which owns every device allocation, plugin interfaces that
// hand the operation only its input and output buffers, or latency-critical
// paths where a cudaMalloc (and the synchronisation it may imply) is not
// allowed.  This entry point takes the same inputs and outputs and uses a
// fixed scratch array that lives in the library instead.
//
// The scratch is a file-scope __device__ array of kNoAllocScratchBytes
// (8 MiB).  Every GPU that loads the library holds it until the process
// exits.  In host code the array's name is only a host-side stand-in, so the
// device address is resolved with cudaGetSymbolAddress, once per device, with
// that device current, on the first call made on that device.
#include <mutex>

#include "../../include/rr.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;

// The shared scratch: column partials of the most recent call.  Every call
// overwrites what it reads, so nothing in it must start at zero.
static __device__ __align__(256) float g_rr_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

constexpr int kMaxDev = 64;
std::mutex g_mu;
void* g_ptr[kMaxDev];

}  // namespace

// Sets the detail string returned by rr_last_error_detail (defined in rr_api.cu).
void rr_set_error_detail(const char* msg);
// rr_layernorm_bwd's argument checks, workspace aside; no device call (rr_api.cu).
rr_status layernorm_bwd_check_args(const void* dy, const void* x, const float* mean,
                                   const float* rstd, const void* gamma, const void* dx,
                                   const void* dgamma, const void* dbeta, int64_t rows,
                                   int64_t cols, rr_dtype dtype);
// rr_layernorm_bwd with at most max_partials column partials (rr_api.cu).
rr_status layernorm_bwd_capped(const void* dy, const void* x, const float* mean, const float* rstd,
                               const void* gamma, void* dx, void* dgamma, void* dbeta,
                               void* workspace, size_t workspace_bytes, int64_t rows, int64_t cols,
                               rr_dtype dtype, cudaStream_t stream, int64_t max_partials);

extern "C" rr_status rr_layernorm_bwd_noalloc(const void* dy, const void* x, const float* mean,
                                              const float* rstd, const void* gamma, void* dx,
                                              void* dgamma, void* dbeta, int64_t rows,
                                              int64_t cols, rr_dtype dtype, cudaStream_t stream) {
  // Every argument is checked on the host before the device is touched, with
  // the same statuses as rr_layernorm_bwd (cols is then in [1, 2^31]).
  rr_status st =
      layernorm_bwd_check_args(dy, x, mean, rstd, gamma, dx, dgamma, dbeta, rows, cols, dtype);
  if (st != RR_OK) return st;
  // One column partial is a row of dgamma and a row of dbeta sums in fp32; the
  // launch is planned with no more partials than the scratch holds (fewer
  // row groups than rr_layernorm_bwd would use when the columns are many).
  const int64_t per_partial_floats = 2;  // per column
  if (cols > (int64_t)(kNoAllocScratchBytes / sizeof(float)) / per_partial_floats) {
    rr_set_error_detail(
        "rr_layernorm_bwd_noalloc: one column partial (2 * cols * 4 bytes) exceeds the "
        "library's fixed 8 MiB scratch; use rr_layernorm_bwd with a caller-provided workspace");
    return RR_ERR_WORKSPACE_TOO_SMALL;
  }
  const int64_t max_partials =
      (int64_t)kNoAllocScratchBytes / (per_partial_floats * cols * (int64_t)sizeof(float));
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDev) {
    rr_set_error_detail("rr_layernorm_bwd_noalloc: no usable current device");
    return RR_ERR_CUDA;
  }
  void* ptr = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_ptr[dev] == nullptr) {
      // first call on this device: resolve the scratch's device address
      e = cudaGetSymbolAddress(&g_ptr[dev], g_rr_noalloc_scratch);
      if (e != cudaSuccess) {
        g_ptr[dev] = nullptr;
        rr_set_error_detail("rr_layernorm_bwd_noalloc: cudaGetSymbolAddress of the scratch failed");
        return RR_ERR_CUDA;
      }
    }
    ptr = g_ptr[dev];
  }
  return layernorm_bwd_capped(dy, x, mean, rstd, gamma, dx, dgamma, dbeta, ptr,
                              kNoAllocScratchBytes, rows, cols, dtype, stream, max_partials);
}
