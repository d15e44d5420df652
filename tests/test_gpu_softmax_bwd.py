"""GPU parity of the log-softmax forward and of the softmax / log-softmax
backward (rr_log_softmax_fwd, rr_softmax_bwd, rr_log_softmax_bwd) against the
float64 oracle, through the C ABI: row lengths across every row tier (row
groups, staged rows, cluster-split rows), ragged tails, +-1e4 outliers and
fully masked rows, misaligned and in-place layouts.  The backward's forward
outputs are the oracle's, stored in the tensor's dtype."""
import numpy as np
import pytest

import oracle
from row_reduction_pass_gb300 import synth

from parity import check_log_softmax, check_softmax_bwd, store

pytestmark = pytest.mark.gpu

COLS = [1, 2, 3, 8, 31, 33, 97, 256, 1000, 2049, 4097, 8192, 16385, 30000, 50304, 65537]


def rows_for(cols: int) -> int:
    if cols >= 4097:
        return 160 if cols <= 16385 else 64
    return int(max(3, min(2000, (1 << 20) // cols)))


def logits(rows, cols, dtype, seed):
    x, _ = synth.xent_inputs(rows, cols, dtype, 3.0, seed, ignore_frac=0.0, outlier_frac=0.01,
                             masked_row_every=37)
    return x


def upstream(rows, cols, dtype, seed):
    rng = np.random.default_rng(seed)
    return store(rng.standard_normal((rows, cols)), dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cols", COLS)
def test_log_softmax_fwd(cols, dtype):
    check_log_softmax(logits(rows_for(cols), cols, dtype, 600 + cols), dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cols", COLS)
def test_softmax_bwd(cols, dtype):
    R = rows_for(cols)
    x = logits(R, cols, dtype, 700 + cols)
    y = store(oracle.softmax(x), dtype)
    check_softmax_bwd(y, upstream(R, cols, dtype, 701 + cols), dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cols", COLS)
def test_log_softmax_bwd(cols, dtype):
    R = rows_for(cols)
    x = logits(R, cols, dtype, 800 + cols)
    z = store(oracle.log_softmax(x), dtype)
    check_softmax_bwd(z, upstream(R, cols, dtype, 801 + cols), dtype, log=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cols", [1, 33, 1000, 4097, 50304])
@pytest.mark.parametrize("layout", ["inplace", "misaligned", "out_misaligned"])
def test_log_softmax_fwd_layouts(cols, dtype, layout):
    x = logits(rows_for(cols) // 2 + 1, cols, dtype, 650 + cols)
    if layout == "inplace":
        check_log_softmax(x, dtype, pad_in=1, inplace=True)
    elif layout == "misaligned":
        check_log_softmax(x, dtype, pad_in=1, pad_out=1)
    else:
        check_log_softmax(x, dtype, pad_in=0, pad_out=1)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cols", [1, 33, 1000, 4097, 50304])
@pytest.mark.parametrize("log", [False, True])
@pytest.mark.parametrize("layout", ["dx_is_y", "dx_is_dy", "all_misaligned", "mixed"])
def test_softmax_bwd_layouts(cols, dtype, log, layout):
    R = rows_for(cols) // 2 + 1
    x = logits(R, cols, dtype, 750 + cols)
    y = store(oracle.log_softmax(x) if log else oracle.softmax(x), dtype)
    dy = upstream(R, cols, dtype, 751 + cols)
    if layout == "dx_is_y":
        check_softmax_bwd(y, dy, dtype, log=log, inplace="y")
    elif layout == "dx_is_dy":
        check_softmax_bwd(y, dy, dtype, log=log, pads=(1, 1, 0), inplace="dy")
    elif layout == "all_misaligned":
        check_softmax_bwd(y, dy, dtype, log=log, pads=(1, 1, 1))
    else:
        # different alignments: element mode
        check_softmax_bwd(y, dy, dtype, log=log, pads=(0, 1, 0))


def test_log_softmax_fwd_masked_rows_are_zero_and_minus_inf_stays():
    x = np.full((3, 9), -np.inf, np.float32)
    x[1, :4] = [1.0, 2.0, 3.0, 4.0]
    x[2] = 0.5
    check_log_softmax(x, "f32")
    assert np.isinf(oracle.log_softmax(x)[1, 5])
