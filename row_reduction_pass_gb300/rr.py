"""Thin ctypes binding of ``librr.so`` (the C ABI declared in ``include/rr.h``).

Argument marshalling only: every function takes torch tensors (device memory),
passes their pointers, sizes, the dtype code and the current CUDA stream to the
C entry point of the same name, and raises :class:`RRError` on a non-zero
status.  No arithmetic of the method happens here, and there is no fallback:
if the library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIBNAME = "librr.so"
_lock = threading.Lock()
_lib = None

RR_F32 = 0
RR_BF16 = 1

_STATUS = {
    0: "RR_OK", 1: "RR_ERR_INVALID_ARG", 2: "RR_ERR_UNSUPPORTED_DTYPE",
    3: "RR_ERR_ALIASING", 4: "RR_ERR_WORKSPACE_TOO_SMALL", 5: "RR_ERR_CUDA",
    6: "RR_ERR_DEVICE_TIMEOUT",
}


class RRError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed: {_STATUS.get(status, status)} ({msg})")
        self.status = status


def library_path() -> str:
    return os.path.join(_HERE, _LIBNAME)


def load_library():
    """Load librr.so (built by ``__graft_entry__.build()``); raises if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(path)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
        st = ctypes.c_int
        lib.rr_status_string.argtypes = [st]
        lib.rr_status_string.restype = ctypes.c_char_p
        lib.rr_softmax_fwd.argtypes = [vp, vp, i64, i64, st, vp]
        lib.rr_softmax_fwd.restype = st
        lib.rr_softmax_xent_fwd_bwd.argtypes = [vp, vp, vp, vp, i64, i64, i32, vp, st, vp]
        lib.rr_softmax_xent_fwd_bwd.restype = st
        lib.rr_log_softmax_fwd.argtypes = [vp, vp, i64, i64, st, vp]
        lib.rr_log_softmax_fwd.restype = st
        lib.rr_softmax_bwd.argtypes = [vp, vp, vp, i64, i64, st, vp]
        lib.rr_softmax_bwd.restype = st
        lib.rr_log_softmax_bwd.argtypes = [vp, vp, vp, i64, i64, st, vp]
        lib.rr_log_softmax_bwd.restype = st
        lib.rr_layernorm_fwd.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, ctypes.c_float,
                                         st, vp]
        lib.rr_layernorm_fwd.restype = st
        lib.rr_layernorm_bwd_workspace_size.argtypes = [i64, i64, st]
        lib.rr_layernorm_bwd_workspace_size.restype = ctypes.c_size_t
        lib.rr_layernorm_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t,
                                         i64, i64, st, vp]
        lib.rr_layernorm_bwd.restype = st
        lib.rr_rmsnorm_fwd.argtypes = [vp, vp, vp, vp, i64, i64, ctypes.c_float, st, vp]
        lib.rr_rmsnorm_fwd.restype = st
        lib.rr_rmsnorm_bwd_workspace_size.argtypes = [i64, i64, st]
        lib.rr_rmsnorm_bwd_workspace_size.restype = ctypes.c_size_t
        lib.rr_rmsnorm_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, i64, i64, st,
                                       vp]
        lib.rr_rmsnorm_bwd.restype = st
        lib.rr_layernorm_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, st, vp]
        lib.rr_layernorm_bwd_noalloc.restype = st
        lib.rr_last_error_detail.argtypes = []
        lib.rr_last_error_detail.restype = ctypes.c_char_p
        lib.rr_read_device_error.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_int), st]
        lib.rr_read_device_error.restype = st
        lib.rr_selftest_bounded_wait.argtypes = [i64, vp]
        lib.rr_selftest_bounded_wait.restype = st
        lib.rr_attention_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, ctypes.c_float,
                                         ctypes.c_int, st, vp]
        lib.rr_attention_fwd.restype = st
        _lib = lib
        return lib


def rr_status_string(status: int) -> str:
    return load_library().rr_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != 0:
        detail = load_library().rr_last_error_detail()
        raise RRError(fn, status, (detail or b"").decode())


def _dtype(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return RR_F32
    if t.dtype == torch.bfloat16:
        return RR_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _contig(*ts):
    for t in ts:
        if t is not None and not t.is_contiguous():
            raise ValueError("tensors must be contiguous row-major")


def rr_softmax_fwd(x, y, stream=None):
    """y[r, :] = softmax(x[r, :]); y may be x (in place)."""
    _contig(x, y)
    rows, cols = x.shape
    _check("rr_softmax_fwd", load_library().rr_softmax_fwd(
        _p(x), _p(y), rows, cols, _dtype(x), _stream(stream)))


def rr_softmax_xent_fwd_bwd(logits, labels, loss, dlogits, ignore_index=-100,
                            bad_label_count=None, stream=None):
    """Per-row loss (fp32) and dlogits = softmax - onehot; dlogits may be logits."""
    _contig(logits, labels, loss, dlogits)
    rows, cols = logits.shape
    _check("rr_softmax_xent_fwd_bwd", load_library().rr_softmax_xent_fwd_bwd(
        _p(logits), _p(labels), _p(loss), _p(dlogits), rows, cols, int(ignore_index),
        _p(bad_label_count), _dtype(logits), _stream(stream)))


def rr_log_softmax_fwd(x, z, stream=None):
    """z = log_softmax(x) per row (z may be x)."""
    _contig(x, z)
    rows, cols = x.shape
    _check("rr_log_softmax_fwd", load_library().rr_log_softmax_fwd(
        _p(x), _p(z), rows, cols, _dtype(x), _stream(stream)))


def rr_softmax_bwd(y, dy, dx, stream=None):
    """dx = y * (dy - sum(y * dy)) per row, y the softmax output."""
    _contig(y, dy, dx)
    rows, cols = y.shape
    _check("rr_softmax_bwd", load_library().rr_softmax_bwd(
        _p(y), _p(dy), _p(dx), rows, cols, _dtype(y), _stream(stream)))


def rr_log_softmax_bwd(z, dz, dx, stream=None):
    """dx = dz - exp(z) * sum(dz) per row, z the log-softmax output."""
    _contig(z, dz, dx)
    rows, cols = z.shape
    _check("rr_log_softmax_bwd", load_library().rr_log_softmax_bwd(
        _p(z), _p(dz), _p(dx), rows, cols, _dtype(z), _stream(stream)))


def rr_attention_fwd(q, k, v, o, lse=None, scale=None, causal=True, stream=None):
    """Scaled dot-product attention of [bh, seq, head_dim] bf16 tensors:
    o = softmax(scale * q k^T (causal mask)) v, lse (fp32 [bh, seq]) optional;
    scale defaults to 1 / sqrt(head_dim)."""
    _contig(q, k, v, o)
    if lse is not None:
        _contig(lse)
    bh, seq, d = q.shape
    if scale is None:
        scale = 1.0 / float(d) ** 0.5
    _check("rr_attention_fwd", load_library().rr_attention_fwd(
        _p(q), _p(k), _p(v), _p(o), _p(lse), bh, seq, d, ctypes.c_float(scale),
        1 if causal else 0, _dtype(q), _stream(stream)))


def rr_layernorm_fwd(x, gamma, beta, y, mean, rstd, eps=1e-5, stream=None):
    """y = (x - mean) * rstd * gamma + beta; saves mean and rstd (fp32)."""
    _contig(x, gamma, beta, y, mean, rstd)
    rows, cols = x.shape
    _check("rr_layernorm_fwd", load_library().rr_layernorm_fwd(
        _p(x), _p(gamma), _p(beta), _p(y), _p(mean), _p(rstd), rows, cols,
        ctypes.c_float(eps), _dtype(x), _stream(stream)))


def rr_layernorm_bwd_workspace_size(rows: int, cols: int, dtype) -> int:
    import torch
    code = {torch.float32: RR_F32, torch.bfloat16: RR_BF16}.get(dtype, dtype)
    return int(load_library().rr_layernorm_bwd_workspace_size(rows, cols, int(code)))


def rr_layernorm_bwd(dy, x, mean, rstd, gamma, dx, dgamma, dbeta, workspace=None,
                     stream=None):
    """dx, dgamma, dbeta of LayerNorm from the saved mean / rstd.

    ``workspace`` is a uint8 CUDA tensor of at least
    ``rr_layernorm_bwd_workspace_size`` bytes; it is allocated here if omitted."""
    import torch
    _contig(dy, x, mean, rstd, gamma, dx, dgamma, dbeta)
    rows, cols = x.shape
    need = rr_layernorm_bwd_workspace_size(rows, cols, x.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=x.device)
    _check("rr_layernorm_bwd", load_library().rr_layernorm_bwd(
        _p(dy), _p(x), _p(mean), _p(rstd), _p(gamma), _p(dx), _p(dgamma), _p(dbeta),
        _p(workspace), workspace.numel() * workspace.element_size(), rows, cols,
        _dtype(x), _stream(stream)))


def rr_layernorm_bwd_noalloc(dy, x, mean, rstd, gamma, dx, dgamma, dbeta, stream=None):
    """rr_layernorm_bwd without a workspace argument: the library's fixed 8 MiB
    scratch holds the column partials (for callers that cannot allocate).
    Calls on one device must not overlap on the GPU."""
    _contig(dy, x, mean, rstd, gamma, dx, dgamma, dbeta)
    rows, cols = x.shape
    _check("rr_layernorm_bwd_noalloc", load_library().rr_layernorm_bwd_noalloc(
        _p(dy), _p(x), _p(mean), _p(rstd), _p(gamma), _p(dx), _p(dgamma), _p(dbeta), rows, cols,
        _dtype(x), _stream(stream)))


def rr_rmsnorm_fwd(x, gamma, y, rstd, eps=1e-5, stream=None):
    """y = x * rstd * gamma with rstd = 1/sqrt(mean(x^2) + eps) (fp32, saved)."""
    _contig(x, gamma, y, rstd)
    rows, cols = x.shape
    _check("rr_rmsnorm_fwd", load_library().rr_rmsnorm_fwd(
        _p(x), _p(gamma), _p(y), _p(rstd), rows, cols, ctypes.c_float(eps), _dtype(x),
        _stream(stream)))


def rr_rmsnorm_bwd_workspace_size(rows: int, cols: int, dtype) -> int:
    import torch
    code = {torch.float32: RR_F32, torch.bfloat16: RR_BF16}.get(dtype, dtype)
    return int(load_library().rr_rmsnorm_bwd_workspace_size(rows, cols, int(code)))


def rr_rmsnorm_bwd(dy, x, rstd, gamma, dx, dgamma, workspace=None, stream=None):
    """dx and dgamma of RMSNorm from the saved rstd.

    ``workspace`` is a uint8 CUDA tensor of at least
    ``rr_rmsnorm_bwd_workspace_size`` bytes; it is allocated here if omitted."""
    import torch
    _contig(dy, x, rstd, gamma, dx, dgamma)
    rows, cols = x.shape
    need = rr_rmsnorm_bwd_workspace_size(rows, cols, x.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=x.device)
    _check("rr_rmsnorm_bwd", load_library().rr_rmsnorm_bwd(
        _p(dy), _p(x), _p(rstd), _p(gamma), _p(dx), _p(dgamma), _p(workspace),
        workspace.numel() * workspace.element_size(), rows, cols, _dtype(x), _stream(stream)))


def rr_read_device_error(device: int = 0, reset: bool = True) -> int:
    """Device-side error word (0 = none, else an RR status such as a timed-out wait)."""
    out = ctypes.c_int(0)
    _check("rr_read_device_error", load_library().rr_read_device_error(
        int(device), ctypes.byref(out), int(bool(reset))))
    return out.value


def rr_selftest_bounded_wait(limit_ns: int, stream=None):
    """Launch the bounded-wait self-test: one block waits on an mbarrier that
    nothing completes, gives up after ``limit_ns`` and records
    RR_ERR_DEVICE_TIMEOUT in the device error word (read it with
    :func:`rr_read_device_error`)."""
    _check("rr_selftest_bounded_wait", load_library().rr_selftest_bounded_wait(
        int(limit_ns), _stream(stream)))
