/*
 * rr.h -- C ABI of librr.so: single-pass fused row reductions for GB300 (sm_103a).
 *
 * Operations (definitions from "Engineering a CUDA Machine Learning Framework
 * from Scratch", sec. 3.1 "Online FlashSoftmax", sec. 3.2 "Welford
 * Single-Pass Normalization", sec. 2.1 (loss gradients fused into registers)
 * and sec. 2.2 (pre-derived analytic backward); cross-entropy as in the
 * "gpu-ml-learning" README, Module 3):
 *   rr_softmax_fwd           y = softmax(x) per row
 *   rr_softmax_xent_fwd_bwd  per-row cross-entropy loss and dlogits = softmax - onehot
 *   rr_layernorm_fwd         y = (x - mean) * rstd * gamma + beta, saving mean / rstd
 *   rr_layernorm_bwd         dx, dgamma, dbeta from the saved mean / rstd
 * and, built on the same machinery:
 *   rr_log_softmax_fwd, rr_softmax_bwd, rr_log_softmax_bwd   the softmax pair
 *   rr_rmsnorm_fwd, rr_rmsnorm_bwd                           RMSNorm
 *   rr_attention_fwd         causal scaled dot-product attention on the online softmax
 *   rr_layernorm_bwd_noalloc the LayerNorm backward without a caller workspace
 *   rr_selftest_bounded_wait, rr_read_device_error   the bounded device waits
 *
 * Common conventions
 *   - Every tensor is dense, row-major [rows x cols] with row stride = cols
 *     (per-column vectors are [cols], per-row vectors are [rows]).
 *   - Every pointer is a DEVICE pointer on the current CUDA device, allocated
 *     and owned by the caller; the library allocates nothing and keeps no state
 *     beyond a per-device cache of attributes (and the fixed scratch array of
 *     rr_layernorm_bwd_noalloc).  Any alignment is accepted;
 *     16-byte aligned bases and rows whose byte length is a multiple of 16 take
 *     the vectorised path.
 *   - `dtype` (RR_F32 or RR_BF16) is the storage type of x, y, logits, dlogits,
 *     gamma, beta, dy, dx, dgamma and dbeta.  mean, rstd and loss are always
 *     float32 and labels int32.  Arithmetic is float32 on the GPU.
 *   - Calls are asynchronous on `stream` (0 = legacy default stream).
 *     Argument errors are returned synchronously and nothing is launched;
 *     launch errors are returned as RR_ERR_CUDA (detail string from
 *     rr_last_error_detail()); faults during execution surface at the caller's
 *     next synchronisation.  No C++ exception crosses this ABI.
 *   - rows == 0 is a no-op returning RR_OK.  cols must be >= 1.
 *   - Per-device state (attributes, the device addresses of the library's
 *     error word and scratch array) is resolved on the first call on a device
 *     and kept for the life of the process: it assumes the device's primary
 *     context lives that long.  After cudaDeviceReset of a device, do not call
 *     the library on that device again in the same process.
 *   - Waits inside the kernels are bounded; a wait that gives up records
 *     RR_ERR_DEVICE_TIMEOUT in a per-device error word read by
 *     rr_read_device_error(), and the kernel returns instead of hanging.
 *   - The kernel tier is chosen per call from the row's byte length, the
 *     pointers' alignment and the device.  The environment variable
 *     RR_FORCE_TIER (read at every call; for tests and tuning) forces one:
 *     0 spans of short rows through shared memory, 1 a row in registers,
 *     2 staged rows (one per CTA, bulk copies to shared memory), 3 rows split
 *     over a thread-block cluster.  A shape the forced tier cannot hold returns
 *     RR_ERR_INVALID_ARG; so does a value other than 0..3 (or T0..T3).
 *   - Rows of at least 8 KB whose row tensors share their address modulo 16
 *     run on kernels that group the rows by their start offset within a
 *     16-byte block (every chunk then an aligned 16-byte block), where measured
 *     faster.  RR_SMX=0 (softmax family) and RR_LNX=0 (LayerNorm / RMSNorm)
 *     turn them off, RR_LNP=0/1 and RR_SMB=1 choose among their variants (tests
 *     and tuning; read at every call).  LayerNorm / RMSNorm rows of at least
 *     64 KB (LayerNorm backward: 8 KB) with no forced tier run on column-block
 *     kernels (row statistics in one launch, the outputs in the next; the
 *     forward keeps its per-block statistics in y until it writes y, so it
 *     takes them only when y does not overlap x); RR_LNC=0 turns those off and
 *     RR_LNC_MIN (bytes) sets their threshold.  Rows of one column with no
 *     forced tier run on elementwise kernels (a one-element row is its own
 *     maximum, sum and moments); RR_ONE=0 turns those off.  Results agree
 *     within the tolerances of the operation whichever kernel runs; they are
 *     not bit-identical across kernels.
 *   - Softmax family range: the exponentials are taken as
 *     2^(x log2 e - fl(m log2 e)) times 2^(-r), r the rounding residual of
 *     fl(m log2 e) (m the row maximum).  For |m| >= 2^30 that residual can
 *     leave the float32 exponent range, and the row's outputs can then be NaN;
 *     finite logits below 2^30 in magnitude are always in range.
 */
#ifndef RR_H
#define RR_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { RR_F32 = 0, RR_BF16 = 1 } rr_dtype;

typedef enum {
    RR_OK = 0,
    RR_ERR_INVALID_ARG = 1,         /* null pointer, negative size, cols == 0, bad eps */
    RR_ERR_UNSUPPORTED_DTYPE = 2,
    RR_ERR_ALIASING = 3,            /* partial overlap of an input and an output */
    RR_ERR_WORKSPACE_TOO_SMALL = 4,
    RR_ERR_CUDA = 5,                /* a CUDA runtime call failed */
    RR_ERR_DEVICE_TIMEOUT = 6       /* a bounded device-side wait gave up */
} rr_status;

/* Static, human-readable name of a status. */
const char *rr_status_string(rr_status status);

/* Detail of the last error returned on the calling host thread ("" if none). */
const char *rr_last_error_detail(void);

/*
 * Softmax forward ("Online FlashSoftmax", sec. 3.1): for each row,
 *   y_j = exp(x_j - m) / d,  m = max_j x_j,  d = sum_j exp(x_j - m),
 * with (m, d) computed in one pass over global memory by the online
 * normaliser and merged across threads with its pairwise rule.
 *   x, y : [rows x cols] dtype.  y == x (in place) is allowed; any other
 *          overlap returns RR_ERR_ALIASING.
 * A row whose maximum is -inf (fully masked) produces y = 0.
 */
rr_status rr_softmax_fwd(const void *x, void *y, int64_t rows, int64_t cols,
                         rr_dtype dtype, cudaStream_t stream);

/*
 * Log-softmax forward of each row: z_j = (x_j - m) - ln d with m = max_j x_j
 * and d = sum_j exp(x_j - m), from the same one-pass online normaliser as
 * rr_softmax_fwd (sec. 3.1).  x, z : [rows x cols] dtype (z == x allowed).
 * A fully masked row (maximum -inf) gives z = 0; a -inf entry of a live row
 * gives -inf.
 */
rr_status rr_log_softmax_fwd(const void *x, void *z, int64_t rows, int64_t cols,
                             rr_dtype dtype, cudaStream_t stream);

/*
 * Softmax backward, the vector-Jacobian product of y = softmax(x) (the
 * Softmax layer of the "NexusGrad" README's layer stack):
 *   dx_j = y_j * (dy_j - sum_k y_k dy_k).
 *   y : the forward's output, dy : upstream gradient, dx : [rows x cols] dtype.
 * dx may equal y or dy exactly (partial overlap is RR_ERR_ALIASING).  A fully
 * masked row (y = 0) gets dx = 0.
 */
rr_status rr_softmax_bwd(const void *y, const void *dy, void *dx, int64_t rows,
                         int64_t cols, rr_dtype dtype, cudaStream_t stream);

/*
 * Log-softmax backward, the vector-Jacobian product of z = log_softmax(x):
 *   dx_j = dz_j - exp(z_j) * sum_k dz_k.
 *   z : the forward's output, dz : upstream gradient, dx : [rows x cols] dtype.
 * dx may equal z or dz exactly.  The formula is applied to every row (a row
 * the forward masked to z = 0 has no derivative of its own).
 */
rr_status rr_log_softmax_bwd(const void *z, const void *dz, void *dx, int64_t rows,
                             int64_t cols, rr_dtype dtype, cudaStream_t stream);

/*
 * Fused softmax cross-entropy, forward and backward in one pass (sec. 2.1
 * and sec. 3.1; cross-entropy as in Module 3 of "gpu-ml-learning"):
 *   loss_r      = m + log d - logits[r, label_r]           (float32, [rows])
 *   dlogits_r,j = softmax(logits_r)_j - [j == label_r]     ([rows x cols] dtype)
 *   logits  : [rows x cols] dtype.   labels : [rows] int32.
 *   dlogits : may equal logits (written in place); other overlap is an error.
 *   ignore_index : a row whose label equals it gets loss 0 and dlogits 0 and
 *           its logits are not read (PyTorch's default is -100).
 *   bad_label_count : nullable device int32; each row whose label is outside
 *           [0, cols) and is not ignore_index adds 1.  Such a row gets loss NaN
 *           and dlogits equal to the plain softmax.  There is no trap.
 * A fully masked row (max = -inf) gets loss 0 and dlogits 0.
 * dlogits is not divided by the number of rows (loss is per row).
 */
rr_status rr_softmax_xent_fwd_bwd(const void *logits, const int32_t *labels,
                                  float *loss, void *dlogits, int64_t rows,
                                  int64_t cols, int32_t ignore_index,
                                  int32_t *bad_label_count, rr_dtype dtype,
                                  cudaStream_t stream);

/*
 * LayerNorm forward ("Welford Single-Pass Normalization", sec. 3.2): per row,
 *   mean = (1/C) sum_j x_j,  var = (1/C) sum_j (x_j - mean)^2 (biased),
 *   rstd = 1 / sqrt(var + eps),  y_j = (x_j - mean) * rstd * gamma_j + beta_j,
 * the moments from one pass over global memory: with the row (or its slice)
 * held on chip, an exact mean from a compensated sum and then the squared
 * deviations about it (row groups, clusters of them, spans); the staged
 * engine kernels, left for rows no row group or cluster of them takes, merge
 * per-thread moments with the Chan/Welford update.
 *   x, y : [rows x cols] dtype (y == x allowed).  gamma, beta : [cols] dtype.
 *   mean, rstd : [rows] float32 outputs, saved for rr_layernorm_bwd.
 *   eps : >= 0 and finite.
 * A row holding a non-finite value is masked: y = 0, mean = 0, rstd = 0.
 */
rr_status rr_layernorm_fwd(const void *x, const void *gamma, const void *beta,
                           void *y, float *mean, float *rstd, int64_t rows,
                           int64_t cols, float eps, rr_dtype dtype,
                           cudaStream_t stream);

/* Bytes of device workspace rr_layernorm_bwd needs for (rows, cols, dtype);
 * 0 if the arguments are invalid.  Depends on the current device. */
size_t rr_layernorm_bwd_workspace_size(int64_t rows, int64_t cols, rr_dtype dtype);

/*
 * LayerNorm backward (analytic derivative, sec. 2.2): with
 * xhat = (x - mean) * rstd and g = dy * gamma,
 *   dx_j     = rstd * (g_j - mean_j(g) - xhat_j * mean_j(g * xhat)),
 *   dgamma_j = sum_r dy_rj * xhat_rj,   dbeta_j = sum_r dy_rj.
 *   dy, x, dx : [rows x cols] dtype (dx may equal dy or x).  gamma, dgamma,
 *   dbeta : [cols] dtype.  mean, rstd : [rows] float32 from rr_layernorm_fwd.
 *   workspace : device scratch of workspace_bytes >= the size query's answer
 *   (16-byte aligned), owned by the caller; its contents on entry are ignored.
 * A row with rstd == 0 (masked by the forward) gets dx = 0 and adds nothing to
 * dgamma / dbeta.  dgamma / dbeta are summed over rows in a fixed order, so the
 * result is deterministic for a given device and shape.
 */
rr_status rr_layernorm_bwd(const void *dy, const void *x, const float *mean,
                           const float *rstd, const void *gamma, void *dx,
                           void *dgamma, void *dbeta, void *workspace,
                           size_t workspace_bytes, int64_t rows, int64_t cols,
                           rr_dtype dtype, cudaStream_t stream);

/*
 * RMSNorm forward ("NexusGrad" README, "Core Capabilities", which lists
 * RMSNorm among its transformer components without a formula; this library
 * takes the standard definition):
 *   ms = (1/C) sum_j x_j^2,  rstd = 1 / sqrt(ms + eps),  y_j = x_j * rstd * gamma_j.
 *   x, y : [rows x cols] dtype (y == x allowed).  gamma : [cols] dtype.
 *   rstd : [rows] float32 output, saved for rr_rmsnorm_bwd.  eps : >= 0, finite.
 * A row whose mean square is not finite is masked: y = 0, rstd = 0.  Rows of
 * any length run where x and y share their address modulo 16 and do not
 * overlap (the column-block kernels); otherwise rows must fit one row group of
 * threads or a thread-block cluster of up to 8 row groups (at least 65537
 * columns for fp32 and bf16, in every alignment), and longer rows return
 * RR_ERR_INVALID_ARG.
 */
rr_status rr_rmsnorm_fwd(const void *x, const void *gamma, void *y, float *rstd,
                         int64_t rows, int64_t cols, float eps, rr_dtype dtype,
                         cudaStream_t stream);

/* Bytes of device workspace rr_rmsnorm_bwd needs for (rows, cols, dtype); 0 if
 * the arguments are invalid or no kernel holds the rows.  Depends on the
 * current device. */
size_t rr_rmsnorm_bwd_workspace_size(int64_t rows, int64_t cols, rr_dtype dtype);

/*
 * RMSNorm backward (analytic derivative of rr_rmsnorm_fwd): with
 * xhat = x * rstd and g = dy * gamma,
 *   dx_j = rstd * (g_j - xhat_j * mean_j(g * xhat)),  dgamma_j = sum_r dy_rj * xhat_rj.
 *   dy, x, dx : [rows x cols] dtype (dx may equal dy or x).  gamma, dgamma : [cols]
 *   dtype.  rstd : [rows] float32 from rr_rmsnorm_fwd.
 *   workspace : device scratch of workspace_bytes >= the size query's answer
 *   (16-byte aligned), owned by the caller; its contents on entry are ignored.
 * A row with rstd == 0 gets dx = 0 and adds nothing to dgamma, which is summed
 * over rows in a fixed order (deterministic for a given device and shape).
 * Rows of any length run where dy, x and dx share their address modulo 16
 * (the column-block kernels); otherwise rows must fit one row group (at least
 * 8192 columns) or, with 16-byte aligned gamma, a thread-block cluster of up
 * to 8 row groups (beyond 65536 columns for fp32 and bf16), and longer rows
 * return RR_ERR_INVALID_ARG (the size query returns 0 when no kernel holds
 * them).
 */
rr_status rr_rmsnorm_bwd(const void *dy, const void *x, const float *rstd,
                         const void *gamma, void *dx, void *dgamma, void *workspace,
                         size_t workspace_bytes, int64_t rows, int64_t cols,
                         rr_dtype dtype, cudaStream_t stream);

/*
 * LayerNorm backward without a caller-provided workspace (this entry point has
 * no counterpart in the pages; it is a convenience of this library).
 * For callers that cannot allocate device memory at call time -- code under a
 * framework's memory planner that owns every allocation, plugin interfaces
 * that receive only input and output buffers, latency-critical paths where an
 * allocation is not allowed.  Same arguments, results and error behaviour as
 * rr_layernorm_bwd, minus the workspace: the column partials go to a scratch
 * array of 8 MiB inside the library, held on every GPU that loads the library
 * until the process exits.  This entry point allocates nothing (no cudaMalloc,
 * cudaFree or allocating library routine).
 *   - The launch is planned with no more column partials (2 * cols fp32 each)
 *     than 8 MiB holds, so shapes whose rr_layernorm_bwd plan would need more
 *     run with fewer row groups.  Rows too long for even one partial
 *     (cols > 1048576) return RR_ERR_WORKSPACE_TOO_SMALL.
 *   - Arguments are checked on the host first, with the same statuses as
 *     rr_layernorm_bwd; only then is the device touched.
 *   - The first call on each device resolves the scratch's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - Every call on a device shares the one scratch array, which keeps the last
 *     call's contents.  Calls that overlap on the GPU (e.g. on two streams
 *     without ordering between them) race on it and give wrong dgamma / dbeta.
 */
rr_status rr_layernorm_bwd_noalloc(const void *dy, const void *x, const float *mean,
                                   const float *rstd, const void *gamma, void *dx,
                                   void *dgamma, void *dbeta, int64_t rows, int64_t cols,
                                   rr_dtype dtype, cudaStream_t stream);

/*
 * Scaled dot-product attention forward, causal or not, built on the online
 * softmax: the extension the source names for it ("Engineering a CUDA Machine
 * Learning Framework from Scratch", sec. 6.4, FlashAttention-style fusion of
 * the sec. 3.1 online normaliser; attention as defined by Vaswani et al.
 * 2017).  For each head b and query row i:
 *   s_j = scale * q_i . k_j over the keys j it may see (j <= i when causal),
 *   o_i = sum_j softmax(s)_j v_j,   lse_i = log sum_j exp(s_j).
 *   q, k, v, o : [bh x seq x head_dim] bf16 (dtype must be RR_BF16), 16-byte
 *   aligned, o must not overlap q, k or v.  lse : [bh x seq] float32, or NULL.
 *   head_dim : 64 or 128;  seq : a multiple of 64;  scale > 0 (usually
 *   1 / sqrt(head_dim)).
 * Products on the tensor cores (bf16 in, fp32 accumulate), softmax in fp32,
 * P rounded to bf16 for P V.  Other shapes or dtypes return
 * RR_ERR_INVALID_ARG / RR_ERR_UNSUPPORTED_DTYPE; bh == 0 or seq == 0 is a no-op.
 */
rr_status rr_attention_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                           int64_t bh, int64_t seq, int64_t head_dim, float scale, int causal,
                           rr_dtype dtype, cudaStream_t stream);

/*
 * Self-test of the bounded device-side waits (a diagnostic of this library;
 * the pages have no counterpart).  Launches one block that arms an mbarrier
 * for 16 bytes of bulk-copy data that no copy ever delivers and waits on it
 * with the same bounded wait the kernels use, giving up after limit_ns
 * nanoseconds of device time (1 .. 10^9; otherwise RR_ERR_INVALID_ARG).  The
 * wait gives up, RR_ERR_DEVICE_TIMEOUT is recorded in the current device's
 * error word (see rr_read_device_error) and the block returns; no memory of
 * the caller is touched and the context stays usable.  Asynchronous on
 * `stream`.
 */
rr_status rr_selftest_bounded_wait(int64_t limit_ns, cudaStream_t stream);

/*
 * Reads (and if `reset` is non-zero clears) the error word of `device` that
 * the kernels set when a bounded wait gives up.  *value receives 0 or an
 * rr_status such as RR_ERR_DEVICE_TIMEOUT.  Synchronous: it waits for the
 * device's outstanding work.
 */
rr_status rr_read_device_error(int device, int *value, int reset);

#ifdef __cplusplus
}
#endif

#endif /* RR_H */
