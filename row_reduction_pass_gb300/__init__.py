"""GB300-native fused row reductions: online softmax and log-softmax (forward and
backward), fused softmax cross-entropy (loss and dlogits in one pass),
one-pass LayerNorm forward (moments from a compensated sum and the squared
deviations of the row held on chip) and backward, RMSNorm forward / backward,
and causal scaled dot-product attention built on
the online softmax (bf16, tensor cores).

The compute path is the C-ABI library ``librr.so`` built from ``csrc/`` for
sm_103a; :mod:`row_reduction_pass_gb300.rr` binds its entry points by name.
"""
from .rr import (RRError, rr_attention_fwd, rr_layernorm_bwd, rr_layernorm_bwd_noalloc,  # noqa: F401
                 rr_layernorm_bwd_workspace_size,
                 rr_layernorm_fwd, rr_log_softmax_bwd, rr_log_softmax_fwd,
                 rr_rmsnorm_bwd, rr_rmsnorm_bwd_workspace_size,
                 rr_rmsnorm_fwd, rr_selftest_bounded_wait, rr_softmax_bwd, rr_softmax_fwd,
                 rr_softmax_xent_fwd_bwd, rr_read_device_error,
                 rr_status_string, library_path, load_library)
