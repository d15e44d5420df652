"""GPU parity: every operation through the C ABI against the float64 oracle on
the same seeded inputs, over row lengths that exercise every kernel variant
(one thread per row up to clusters of CTAs per row), ragged tails, misaligned
bases (element mode), in-place outputs, masked and ignored rows."""
import numpy as np
import pytest

import oracle
from row_reduction_pass_gb300 import synth

from parity import (check_ln, check_log_softmax, check_norm_bwd, check_rms, check_softmax,
                    check_softmax_bwd, check_xent, store)

pytestmark = pytest.mark.gpu

COLS = [1, 2, 3, 5, 8, 31, 32, 33, 97, 127, 256, 512, 768, 1000, 1023, 2049, 4097, 8192,
        12289, 16385, 50304, 65537]


def rows_for(cols: int) -> int:
    if cols >= 4097:
        return 320 if cols <= 16385 else 160
    return int(max(3, min(3000, (1 << 21) // cols)))


def logits(rows, cols, dtype, seed, sigma=3.0, outliers=0.01, masked_every=37):
    x, lab = synth.xent_inputs(rows, cols, dtype, sigma, seed, ignore_frac=0.05,
                               outlier_frac=outliers, masked_row_every=masked_every)
    return x, lab


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cols", COLS)
def test_softmax(cols, dtype):
    x, _ = logits(rows_for(cols), cols, dtype, 100 + cols)
    check_softmax(x, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cols", [1, 3, 33, 97, 1000, 4097, 50304])
@pytest.mark.parametrize("layout", ["both_misaligned", "out_misaligned", "inplace"])
def test_softmax_layouts(cols, dtype, layout):
    x, _ = logits(rows_for(cols) // 2 + 1, cols, dtype, 200 + cols)
    if layout == "both_misaligned":
        check_softmax(x, dtype, pad_in=1, pad_out=1)
    elif layout == "out_misaligned":
        check_softmax(x, dtype, pad_in=0, pad_out=1)
    else:
        check_softmax(x, dtype, pad_in=1, inplace=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cols", COLS)
def test_xent(cols, dtype):
    x, lab = logits(rows_for(cols), cols, dtype, 300 + cols)
    lab[1::50] = cols + 3          # out of range -> NaN loss, counted
    lab[2::97] = -7                # negative, not the ignore index
    check_xent(x, lab, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cols", [1, 5, 31, 1000, 4097, 50304, 65537])
@pytest.mark.parametrize("layout", ["inplace", "misaligned_inplace", "out_misaligned"])
def test_xent_layouts(cols, dtype, layout):
    x, lab = logits(rows_for(cols) // 2 + 1, cols, dtype, 400 + cols)
    if layout == "inplace":
        check_xent(x, lab, dtype, inplace=True)
    elif layout == "misaligned_inplace":
        check_xent(x, lab, dtype, pad_in=3, inplace=True)
    else:
        check_xent(x, lab, dtype, pad_in=0, pad_out=1)


def test_xent_custom_ignore_index():
    x, lab = logits(50, 77, "f32", 5)
    lab[::3] = 7                   # a valid class used as the ignore index
    check_xent(x, lab, "f32", ignore_index=7)


LN_COLS = [1, 2, 3, 8, 31, 32, 97, 128, 256, 768, 1000, 1024, 2049, 4096, 4097, 6145, 8192, 8193,
           12289, 16384, 32768, 65537]


def ln_case(rows, cols, dtype, seed):
    return synth.ln_inputs(rows, cols, dtype, seed, row_offset=10.0, gamma_std=0.1,
                           beta_std=0.1, outlier_frac=0.005, masked_row_every=41)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cols", LN_COLS)
def test_layernorm(cols, dtype):
    x, g, b, dy = ln_case(rows_for(cols), cols, dtype, 500 + cols)
    check_ln(x, g, b, dy, 1e-5, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cols", [1, 31, 768, 1000, 4097, 16384, 40000])
@pytest.mark.parametrize("pad", [(1, 1, 1, 1, 1), (0, 0, 1, 0, 0), (0, 1, 0, 0, 1)])
def test_layernorm_misaligned(cols, dtype, pad):
    x, g, b, dy = ln_case(rows_for(cols) // 2 + 1, cols, dtype, 600 + cols)
    check_ln(x, g, b, dy, 1e-5, dtype, pad=pad)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_layernorm_chain_uses_gpu_stats(dtype):
    """fwd -> bwd with the GPU's own float32 mean / rstd."""
    x, g, b, dy = ln_case(1000, 768, dtype, 7)
    check_ln(x, g, b, dy, 1e-5, dtype, oracle_stats=False)


def test_layernorm_eps_zero_and_large():
    x, g, b, dy = ln_case(64, 100, "f32", 8)
    check_ln(x, g, b, dy, 0.0, "f32")
    check_ln(x, g, b, dy, 10.0, "f32")


SHORT = [("f32", c) for c in (1, 3, 17, 31, 32)] + \
        [("bf16", c) for c in (1, 5, 32, 33, 47, 63, 64)]


@pytest.mark.parametrize("dtype,cols", SHORT)
@pytest.mark.parametrize("rows", [1, 37, 4099, 60001, 1000003])
@pytest.mark.parametrize("layout", ["plain", "stats_misaligned", "dx_over_dy", "dx_over_x"])
def test_layernorm_bwd_short_rows(dtype, cols, rows, layout):
    """Short rows: spans of rows per warp up to 64 bytes, bf16 96 (a million
    rows: several spans per warp through both stages; bf16 rows of 33..47
    columns hold two column slots a lane), the phase-class kernel beyond,
    ragged last span, statistics staged with the span (16-byte aligned) or
    loaded, dx in place."""
    if rows * cols > 400000 and layout != "plain":
        pytest.skip("large shapes run in the plain layout only")
    if rows > 100000 and cols > 5:
        pytest.skip("a million rows for the shortest rows only")
    x, g, b, dy = ln_case(rows, cols, dtype, 700 + cols + rows)
    check_norm_bwd(x, g, b, dy, dtype, stat_pad=1 if layout == "stats_misaligned" else 0,
                   inplace={"dx_over_dy": "dy", "dx_over_x": "x"}.get(layout))


# Rows of 130..448 bytes that are not whole 16-byte chunks: the span kernels
# take the softmax family, its backward (up to 224 bytes) and the norm forward
# (bf16 up to 128 columns), with one row per lane (32 rows per span); around
# the limits in bytes and columns on both sides.
SPAN_LONG = [("f32", c) for c in (33, 35, 50, 63, 101, 111, 113)] + \
            [("bf16", c) for c in (65, 99, 111, 127, 131, 150, 161, 199, 201)]


@pytest.mark.parametrize("dtype,cols", SPAN_LONG)
@pytest.mark.parametrize("rows", [1, 33, 5003, 70001])
def test_span_rows_up_to_448_bytes(dtype, cols, rows):
    """Several spans per warp (70001 rows), a ragged last span, one row; every
    operation routed as without a forced tier, against the oracle."""
    x, lab = logits(rows, cols, dtype, 900 + cols + rows)
    lab[1::50] = cols + 3
    check_softmax(x, dtype)
    check_log_softmax(x, dtype)
    check_xent(x, lab, dtype)
    check_xent(x, lab, dtype, inplace=True)
    y = store(oracle.softmax(x), dtype)
    dy = store(np.random.default_rng(cols + rows).standard_normal((rows, cols)), dtype)
    check_softmax_bwd(y, dy, dtype)
    check_softmax_bwd(store(oracle.log_softmax(x), dtype), dy, dtype, log=True, inplace="dy")
    xl, g, b, dyl = ln_case(rows, cols, dtype, 950 + cols + rows)
    check_ln(xl, g, b, dyl, 1e-5, dtype)
    check_rms(xl, g, dyl, 1e-5, dtype)
