"""GPU parity of RMSNorm forward / backward (rr_rmsnorm_fwd, rr_rmsnorm_bwd)
against the float64 oracle, through the C ABI: row lengths across the
row-group sizes and their boundaries, ragged last chunks, misaligned tensors,
masked rows and +-1e4 outliers, a chained GPU-forward-into-backward check,
rows of any length on the column-block kernels, and the rejection of rows
beyond a cluster of row groups where those kernels are off."""
import numpy as np
import pytest
import torch

import oracle
import row_reduction_pass_gb300 as rr
from row_reduction_pass_gb300 import synth

from parity import (TOL, TOL_F32_OUT, check_guards, check_norm_bwd, check_rms, compare,
                    empty_like_dev, host, out_f32, to_dev)

pytestmark = pytest.mark.gpu

RMS_COLS = [1, 2, 3, 8, 31, 32, 97, 128, 768, 1000, 1024, 2049, 4096, 4097, 6144, 8192, 8193]


def rows_for(cols: int) -> int:
    return 320 if cols >= 4096 else int(max(3, min(3000, (1 << 21) // cols)))


def case(rows, cols, dtype, seed):
    x, g, _, dy = synth.ln_inputs(rows, cols, dtype, seed, row_offset=2.0, gamma_std=0.1,
                                  outlier_frac=0.005, masked_row_every=41)
    return x, g, dy


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cols", RMS_COLS)
def test_rmsnorm(cols, dtype):
    x, g, dy = case(rows_for(cols), cols, dtype, 900 + cols)
    check_rms(x, g, dy, 1e-5, dtype)


def test_rmsnorm_bf16_rows_beyond_8192():
    """bf16 rows of 12289 columns: the deep backward (shared-memory partials)."""
    x, g, dy = case(200, 12289, "bf16", 912289)
    check_rms(x, g, dy, 1e-5, "bf16")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cols", [1, 31, 768, 1000, 4097])
@pytest.mark.parametrize("pad", [(1, 1, 1, 1, 1), (0, 0, 1, 0, 0), (0, 1, 0, 0, 1)])
def test_rmsnorm_misaligned(cols, dtype, pad):
    x, g, dy = case(rows_for(cols) // 2 + 1, cols, dtype, 950 + cols)
    check_rms(x, g, dy, 1e-5, dtype, pad=pad)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_rmsnorm_chained_gpu_statistics(dtype):
    x, g, _, dy = synth.ln_inputs(512, 1000, dtype, 77, row_offset=1.0)
    check_rms(x, g, dy, 1e-5, dtype, oracle_stats=False)


@pytest.mark.parametrize("kern", ["routed", "clusters"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cols", [16385, 40000, 65537])
@pytest.mark.parametrize("pad", [(0, 0, 0, 0, 0), (1, 1, 0, 0, 0), (0, 0, 1, 0, 0)])
def test_rmsnorm_fwd_clustered_rows(cols, dtype, pad, kern, monkeypatch):
    """Forward rows longer than one row group: split over a thread-block
    cluster (RR_LNC=0), or routed (the column-block kernels for rows of 64 KB
    and more whose x and y share their address modulo 16)."""
    if kern == "clusters":
        monkeypatch.setenv("RR_LNC", "0")
    x, g, _ = case(64, cols, dtype, 990 + cols)
    xd, gd = to_dev(x, pad[0]), to_dev(g, pad[2])
    y = empty_like_dev(x.shape, dtype, pad[1])
    rstd = out_f32(x.shape[0])
    rr.rr_rmsnorm_fwd(xd, gd, y, rstd, eps=1e-5)
    torch.cuda.synchronize()
    check_guards()
    ry, rrstd = oracle.rms_fwd(x, g, 1e-5)
    rtol, atol = TOL[dtype]
    compare("rms y (clustered)", host(y), ry, rtol, atol)
    compare("rms rstd (clustered)", host(rstd), rrstd, *TOL_F32_OUT)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_rmsnorm_rows_beyond_a_cluster(dtype):
    """Rows beyond a cluster of 8 row groups (300000 columns): the column-block
    kernels take them, forward and backward, against the oracle."""
    x, g, dy = case(5, 300000, dtype, 1300)
    check_rms(x, g, dy, 1e-5, dtype)


def test_rmsnorm_rejects_rows_beyond_its_kernels(monkeypatch):
    """With the column-block kernels off, rows beyond a cluster of row groups
    are refused (and the workspace query answers 0)."""
    monkeypatch.setenv("RR_LNC", "0")
    dev = torch.device("cuda", 0)
    x = torch.zeros(2, 300000, device=dev)          # beyond a cluster of 8 row groups
    g = torch.ones(300000, device=dev)
    with pytest.raises(rr.RRError):
        rr.rr_rmsnorm_fwd(x, g, torch.empty_like(x), torch.empty(2, device=dev))
    x = torch.zeros(4, 300000, device=dev)           # nor a cluster of backward row groups
    g = torch.ones(300000, device=dev)
    assert rr.rr_rmsnorm_bwd_workspace_size(4, 300000, torch.float32) == 0
    with pytest.raises(rr.RRError):
        rr.rr_rmsnorm_bwd(x, x, torch.ones(4, device=dev), g, torch.empty_like(x),
                          torch.empty_like(g), workspace=torch.empty(1 << 20, dtype=torch.uint8,
                                                                      device=dev))


SHORT = [("f32", c) for c in (1, 3, 17, 32)] + [("bf16", c) for c in (1, 5, 33, 64)]


@pytest.mark.parametrize("dtype,cols", SHORT)
@pytest.mark.parametrize("rows", [1, 37, 4099, 60001, 1000003])
@pytest.mark.parametrize("layout", ["plain", "stats_misaligned", "dx_over_x"])
def test_rmsnorm_bwd_short_rows(dtype, cols, rows, layout):
    """The RMSNorm backward of rows of at most 128 bytes (spans of rows per warp)."""
    if rows * cols > 400000 and layout != "plain":
        pytest.skip("large shapes run in the plain layout only")
    if rows > 100000 and cols > 5:
        pytest.skip("a million rows for the shortest rows only")
    x, g, dy = case(rows, cols, dtype, 950 + cols + rows)
    check_norm_bwd(x, g, None, dy, dtype, rms=True,
                   stat_pad=1 if layout == "stats_misaligned" else 0,
                   inplace={"dx_over_x": "x"}.get(layout))
