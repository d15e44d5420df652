"""Seeded synthetic inputs for the row reductions.

This module is the one piece shared by the GPU path's tests/benchmark and the
float64 oracle: it draws the inputs and holds none of the method's arithmetic
(no softmax, no moments).  Everything is numpy on the host; float32 values are
rounded to bfloat16 with round-to-nearest-even when a bf16 workload asks for it,
and both sides consume the same stored bits.

Random streams: ``numpy.random.PCG64`` children of ``SeedSequence(seed)``, one
child per fixed block of 2**22 elements, so a given seed gives the same array
however many threads draw it.
"""
from __future__ import annotations

import concurrent.futures as _cf
import os

import numpy as np

SEED_BASE = 20261202
IGNORE_INDEX = -100
_BLOCK = 1 << 22


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even).

    Returns the uint16 bit patterns.  NaN stays NaN (quiet); infinities stay."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    out = np.empty(a.shape, np.uint16)
    flat_u = u.reshape(-1)
    flat_o = out.reshape(-1)
    step = 1 << 24
    for s in range(0, flat_u.size, step):
        v = flat_u[s:s + step]
        nan = (v & 0x7FFFFFFF) > 0x7F800000
        r = (v + (np.uint32(0x7FFF) + ((v >> 16) & 1))) >> 16
        r = r.astype(np.uint16)
        if nan.any():
            r[nan] = ((v[nan] >> 16) | 0x40).astype(np.uint16)
        flat_o[s:s + step] = r
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def _threads() -> int:
    try:
        return max(1, min(16, len(os.sched_getaffinity(0))))
    except AttributeError:  # pragma: no cover
        return max(1, min(16, os.cpu_count() or 1))


def standard_normal(n: int, seed: int, stream: int = 0) -> np.ndarray:
    """n float32 N(0,1) draws; block-seeded so the result is thread-count free."""
    ss = np.random.SeedSequence([seed, stream])
    nblk = (n + _BLOCK - 1) // _BLOCK
    kids = ss.spawn(nblk)
    out = np.empty(n, np.float32)

    def fill(b):
        lo, hi = b * _BLOCK, min(n, (b + 1) * _BLOCK)
        np.random.Generator(np.random.PCG64(kids[b])).standard_normal(
            hi - lo, dtype=np.float32, out=out[lo:hi])

    if nblk == 1:
        fill(0)
    else:
        with _cf.ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, range(nblk)))
    return out


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream])))


def _store(a32: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.ascontiguousarray(a32, np.float32)
    if dtype == "bf16":
        return bf16_bits(a32)
    raise ValueError(f"unknown dtype {dtype!r}")


def _outliers(a: np.ndarray, frac: float, value: float, rng) -> None:
    """Set a Bernoulli(frac) subset of entries to +-value (signs 50/50)."""
    if frac <= 0:
        return
    flat = a.reshape(-1)
    n = flat.size
    k = rng.binomial(n, frac)
    idx = rng.choice(n, size=k, replace=False) if n < (1 << 26) else \
        np.unique(rng.integers(0, n, size=k))
    sign = np.where(rng.random(idx.size) < 0.5, -1.0, 1.0).astype(np.float32)
    flat[idx] = sign * np.float32(value)


def xent_inputs(rows: int, cols: int, dtype: str, sigma: float, seed: int,
                ignore_frac: float = 0.0, outlier_frac: float = 0.0,
                outlier_value: float = 1e4, masked_row_every: int = 0):
    """Logits ~ N(0, sigma^2) and labels ~ U{0..cols-1} (int32).

    ignore_frac: Bernoulli fraction of labels replaced by IGNORE_INDEX.
    outlier_frac: fraction of entries set to +-outlier_value.
    masked_row_every: rows r with r % k == 0 are set entirely to -inf."""
    a = standard_normal(rows * cols, seed, 0).reshape(rows, cols)
    if sigma != 1.0:
        a *= np.float32(sigma)
    rng = _rng(seed, 1)
    _outliers(a, outlier_frac, outlier_value, rng)
    if masked_row_every:
        a[::masked_row_every, :] = -np.inf
    labels = rng.integers(0, cols, size=rows, dtype=np.int64).astype(np.int32)
    if ignore_frac > 0:
        labels[rng.random(rows) < ignore_frac] = IGNORE_INDEX
    return _store(a, dtype), labels


def causal_scores(batch: int, heads: int, queries: int, keys: int, dtype: str,
                  sigma: float, seed: int) -> np.ndarray:
    """Attention scores ~ N(0, sigma^2) as [batch*heads*queries, keys] rows,
    with the upper triangle (key > query) set to -inf."""
    rows = batch * heads * queries
    a = standard_normal(rows * keys, seed, 0).reshape(batch * heads, queries, keys)
    if sigma != 1.0:
        a *= np.float32(sigma)
    upper = np.arange(keys)[None, :] > np.arange(queries)[:, None]
    a[:, upper] = -np.inf
    return _store(a.reshape(rows, keys), dtype)


def attn_inputs(bh: int, seq: int, head_dim: int, seed: int, sigma: float = 1.0):
    """Attention q, k, v ~ N(0, sigma^2) as [bh, seq, head_dim] bfloat16 bits
    (three independent streams of one seed)."""
    n = bh * seq * head_dim
    out = []
    for stream in range(3):
        a = standard_normal(n, seed, 10 + stream).reshape(bh, seq, head_dim)
        if sigma != 1.0:
            a *= np.float32(sigma)
        out.append(_store(a, "bf16"))
    return tuple(out)


def ln_inputs(rows: int, cols: int, dtype: str, seed: int, row_offset: float = 0.0,
              gamma_mean: float = 1.0, gamma_std: float = 0.1, beta_std: float = 0.1,
              outlier_frac: float = 0.0, outlier_value: float = 1e4,
              masked_row_every: int = 0):
    """LayerNorm inputs: x = N(0,1) + per-row offset U(-row_offset, row_offset),
    gamma ~ N(gamma_mean, gamma_std^2), beta ~ N(0, beta_std^2), dy ~ N(0,1).

    Returns (x, gamma, beta, dy) in the storage dtype."""
    x = standard_normal(rows * cols, seed, 0).reshape(rows, cols)
    rng = _rng(seed, 1)
    if row_offset:
        x += rng.uniform(-row_offset, row_offset, size=(rows, 1)).astype(np.float32)
    _outliers(x, outlier_frac, outlier_value, rng)
    if masked_row_every:
        x[::masked_row_every, :] = -np.inf
    gamma = (gamma_mean + gamma_std * rng.standard_normal(cols)).astype(np.float32)
    beta = (beta_std * rng.standard_normal(cols)).astype(np.float32)
    dy = standard_normal(rows * cols, seed, 2).reshape(rows, cols)
    return _store(x, dtype), _store(gamma, dtype), _store(beta, dtype), _store(dy, dtype)


# -- the workloads the library is measured and checked on -----------------------
# Each recipe is a plain dict; ``make(name, **overrides)`` draws it.

SWEEP_COLS = (1, 31, 97, 1000, 4097, 65537)


def sweep_rows(cols: int) -> int:
    return (1 << 24) // cols


WORKLOADS = {
    # softmax-cross-entropy fwd+bwd, fp32, 64 x 1000, logits ~ N(0, 2^2)
    "xent_f32_64x1000": dict(kind="xent", rows=64, cols=1000, dtype="f32", sigma=2.0,
                             seed=SEED_BASE + 0),
    # LayerNorm fwd+bwd, fp32, 4096 x 768, x = N(0,1) + U(-10,10) per row
    "ln_f32_4096x768": dict(kind="ln", rows=4096, cols=768, dtype="f32", seed=SEED_BASE + 1,
                            row_offset=10.0, gamma_mean=1.0, gamma_std=0.1, beta_std=0.1,
                            eps=1e-5),
    # causal attention-score softmax fwd, bf16, 8x16x512 rows x 512 keys, N(0, 4^2)
    "softmax_bf16_causal_65536x512": dict(kind="causal", batch=8, heads=16, queries=512,
                                          keys=512, dtype="bf16", sigma=4.0,
                                          seed=SEED_BASE + 2),
    # LM-head softmax-cross-entropy fwd+bwd, bf16, 16384 x 50304, N(0, 3^2), 5% ignored
    "xent_bf16_16384x50304": dict(kind="xent", rows=16384, cols=50304, dtype="bf16",
                                  sigma=3.0, ignore_frac=0.05, seed=SEED_BASE + 3),
}
for _dt in ("f32", "bf16"):
    for _c in SWEEP_COLS:
        WORKLOADS[f"sweep_xent_{_dt}_c{_c}"] = dict(
            kind="xent", rows=sweep_rows(_c), cols=_c, dtype=_dt, sigma=1.0,
            outlier_frac=0.01, masked_row_every=1024, seed=SEED_BASE + 4)
        WORKLOADS[f"sweep_ln_{_dt}_c{_c}"] = dict(
            kind="ln", rows=sweep_rows(_c), cols=_c, dtype=_dt, seed=SEED_BASE + 4,
            row_offset=0.0, gamma_mean=1.0, gamma_std=0.0, beta_std=0.0,
            outlier_frac=0.01, masked_row_every=1024, eps=1e-5)


def make(name: str, rows: int | None = None, **over):
    """Draw workload ``name``; ``rows`` (if given) truncates / resizes the row count
    while keeping every other property of the recipe."""
    spec = dict(WORKLOADS[name])
    spec.update(over)
    kind = spec.pop("kind")
    if rows is not None:
        if kind == "causal":
            raise ValueError("causal workload is sized by batch/heads")
        spec["rows"] = rows
    if kind == "xent":
        logits, labels = xent_inputs(spec["rows"], spec["cols"], spec["dtype"], spec["sigma"],
                                     spec["seed"], spec.get("ignore_frac", 0.0),
                                     spec.get("outlier_frac", 0.0), 1e4,
                                     spec.get("masked_row_every", 0))
        return dict(kind=kind, dtype=spec["dtype"], logits=logits, labels=labels,
                    ignore_index=IGNORE_INDEX)
    if kind == "causal":
        x = causal_scores(spec["batch"], spec["heads"], spec["queries"], spec["keys"],
                          spec["dtype"], spec["sigma"], spec["seed"])
        return dict(kind=kind, dtype=spec["dtype"], x=x)
    if kind == "ln":
        x, g, b, dy = ln_inputs(spec["rows"], spec["cols"], spec["dtype"], spec["seed"],
                                spec.get("row_offset", 0.0), spec.get("gamma_mean", 1.0),
                                spec.get("gamma_std", 0.1), spec.get("beta_std", 0.1),
                                spec.get("outlier_frac", 0.0), 1e4,
                                spec.get("masked_row_every", 0))
        return dict(kind=kind, dtype=spec["dtype"], x=x, gamma=g, beta=b, dy=dy,
                    eps=spec["eps"])
    raise ValueError(kind)
