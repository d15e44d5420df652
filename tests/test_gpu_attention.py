"""GPU parity of the scaled dot-product attention forward (rr_attention_fwd,
bf16 tensor cores) against the float64 oracle on the same seeded inputs:
head dimensions 64 and 128, one to several key tiles, causal and not, sharp
score distributions; the full 8 x 16 heads x 512 shape on sampled heads; the
shapes and dtypes the call refuses.

Tolerance, from the arithmetic: the products are exact bf16 x bf16 in fp32,
the softmax weights p_j are rounded to bf16 (relative 2^-9) before P V and the
output is rounded to bf16 (2^-9 |o|), so |o_gpu - o_ref| <= 2^-8 sum_j p_j |v_j|;
the test allows twice that.  lse is fp32: 1e-5 relative plus 1e-5."""
import numpy as np
import pytest
import torch

import oracle
import row_reduction_pass_gb300 as rr
from row_reduction_pass_gb300 import synth

from parity import TOL_F32_OUT, check_guards, compare, empty_like_dev, host, out_f32, to_dev

pytestmark = pytest.mark.gpu


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def run_attention(bh, seq, d, seed, causal=True, sigma=1.0, heads_checked=None):
    q, k, v = synth.attn_inputs(bh, seq, d, seed, sigma)
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    o = empty_like_dev((bh, seq, d), "bf16")
    lse = out_f32(bh * seq).view(bh, seq)
    scale = 1.0 / np.sqrt(d)
    rr.rr_attention_fwd(qd, kd, vd, o, lse, scale=scale, causal=causal)
    torch.cuda.synchronize()
    check_guards()
    heads = range(bh) if heads_checked is None else heads_checked
    for h in heads:
        sl = slice(h, h + 1)
        ro, rl = oracle.attention(q[sl], k[sl], v[sl], scale, causal)
        vabs = synth.bf16_bits(np.abs(synth.bf16_to_f32(v[sl])))
        mag, _ = oracle.attention(q[sl], k[sl], vabs, scale, causal)  # sum_j p_j |v_j|
        compare(f"attention o (head {h})", host(o[sl]), ro, 0.0, 1e-6, scale=mag,
                scale_rtol=2.0 ** -7)
        compare(f"attention lse (head {h})", host(lse[sl]), rl, *TOL_F32_OUT)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("seq", [64, 128, 256])
@pytest.mark.parametrize("causal", [True, False])
def test_attention(d, seq, causal):
    run_attention(3, seq, d, 100 + seq + d, causal)


@pytest.mark.parametrize("d", [64, 128])
def test_attention_sharp_scores(d):
    # sigma 3 on q and k: scores ~ 9 sqrt(d) / sqrt(d) wide, near one-hot rows
    run_attention(2, 192, d, 7 + d, True, sigma=3.0)


def test_attention_full_shape_sampled_heads():
    # 8 batches x 16 heads x 512 queries, head_dim 64, every head computed;
    # eight heads spread over the batch compared against the oracle
    run_attention(128, 512, 64, 2024, True, heads_checked=[0, 17, 35, 54, 71, 90, 109, 127])


@pytest.mark.parametrize("d", [64, 128])
def test_attention_several_query_tiles_per_pipeline(d):
    # 64 heads x 1024 keys, not causal: 512 query tiles, several per pipeline
    # of the persistent kernel (query tile changes: Q reloads, O hand-over)
    run_attention(64, 1024, d, 77 + d, False, heads_checked=[0, 21, 42, 63])


@pytest.mark.parametrize("d", [64, 128])
def test_attention_long_causal_sequence(d):
    # 4 heads x 2048 queries, causal: 32 key tiles on the longest query rows
    # (the compute-bound regime the tensor-core timing lines use)
    run_attention(4, 2048, d, 91 + d, True, heads_checked=[0, 3])


def test_attention_lse_optional_and_empty():
    q, k, v = (dev_bf16(a) for a in synth.attn_inputs(2, 64, 64, 5))
    o = torch.empty_like(q)
    rr.rr_attention_fwd(q, k, v, o, None)
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all()
    e = torch.empty((0, 64, 64), dtype=torch.bfloat16, device="cuda")
    rr.rr_attention_fwd(e, e, e, torch.empty_like(e), None)


def test_attention_refuses_unsupported_shapes():
    q = torch.zeros((1, 96, 64), dtype=torch.bfloat16, device="cuda")  # seq not a multiple of 64
    with pytest.raises(rr.RRError, match="INVALID_ARG"):
        rr.rr_attention_fwd(q, q, q, torch.empty_like(q))
    q = torch.zeros((1, 64, 96), dtype=torch.bfloat16, device="cuda")  # head_dim 96
    with pytest.raises(rr.RRError, match="INVALID_ARG"):
        rr.rr_attention_fwd(q, q, q, torch.empty_like(q))
    q = torch.zeros((1, 64, 64), dtype=torch.float32, device="cuda")   # fp32: no tensor-core path here
    with pytest.raises(rr.RRError, match="UNSUPPORTED_DTYPE"):
        rr.rr_attention_fwd(q, q, q, torch.empty_like(q))
    q = torch.zeros((1, 64, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(rr.RRError, match="ALIASING"):
        rr.rr_attention_fwd(q, q, q, q)
