"""Benchmark of the fused row reductions on one GB300 (or N weak-scaled replicas).

One step = one pass of the whole hot path over one batch of synthetic input,
every input already resident in HBM:
  1. LayerNorm forward,  fp32, 4096 x 768  (x = N(0,1) + U(-10,10) per row)
  2. causal attention-score softmax, bf16, 65536 x 512 (scores ~ N(0, 4^2), key > query = -inf)
  3. LayerNorm backward, fp32, 4096 x 768 (+ the fixed-order dgamma / dbeta pass)
  4. LM-head softmax cross-entropy fwd+bwd, bf16, 16384 x 50304 (logits ~ N(0, 3^2),
     5% labels = -100), per-row fp32 loss, dlogits written in place
The metric is achieved HBM bandwidth: algorithmic (minimum) bytes of the step
divided by its device time.  The 3.3 GB cross-entropy pass streams far more
than the 129 MB L2 through the chip every step, so each step starts with a
cold L2 for its inputs.

Prints one JSON line (rank 0).  --impl reference times the float64 CPU oracle
(the reference implementation of the same arithmetic) on a bounded sample.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from row_reduction_pass_gb300 import synth  # noqa: E402

METRIC = "achieved HBM GB/s (% of GB300 peak) for softmax-xent & LayerNorm fwd+bwd"
FALLBACK_HBM_GBS = 6800.0
LN_BF16_COLS = (1000, 4097, 65537)   # the sweep's bf16 LayerNorm cases, 2^24 elements each
WORKLOAD = ("hot-path step: LN fwd+bwd fp32 4096x768 + causal softmax fwd bf16 65536x512 + "
            "LN fwd+bwd bf16 16777x1000, 4095x4097, 255x65537 (sweep cases) + "
            "softmax-xent fwd+bwd bf16 16384x50304 (in place, 5% ignored)")
XENT_IN_PLACE = ("dlogits are written over the logits (the configuration's in-place call), so "
                 "every step after the first reads the previous step's dlogits: the same bytes "
                 "and the same work (the kernel's time does not depend on the values; ignored "
                 "rows stay ignored)")


# ------------------------------------------------------------ byte counts ----

def ln_bytes(rows, cols, e):
    fwd = 2 * rows * cols * e + 2 * cols * e + 8 * rows          # x, y, gamma, beta, mean, rstd
    bwd = 3 * rows * cols * e + 3 * cols * e + 8 * rows          # dy, x, dx, gamma, dg, db, mean, rstd
    return fwd, bwd


def rms_bytes(rows, cols, e):
    fwd = 2 * rows * cols * e + cols * e + 4 * rows              # x, y, gamma, rstd
    bwd = 3 * rows * cols * e + 2 * cols * e + 4 * rows          # dy, x, dx, gamma, dg, rstd
    return fwd, bwd


def softmax_bytes(rows, cols, e):
    return 2 * rows * cols * e


def xent_bytes(rows, cols, e, n_ignored):
    """Minimum traffic: ignored rows are only written (zeros), others read + written."""
    return (2 * (rows - n_ignored) + n_ignored) * cols * e + 8 * rows


# ----------------------------------------------------------------- clocks ----

_REASON_BITS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
                0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
                0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
                0x100: "display_clock_setting"}


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[str] = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=clocks.sm,clocks.max.sm,"
                 "clocks_event_reasons.active", "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 3:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
                bits = int(parts[2], 16) if parts[2].startswith("0x") else int(parts[2])
            except ValueError:
                continue
            for b, name in _REASON_BITS.items():
                if bits & b and name != "gpu_idle":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ peaks ----

FALLBACK_BF16_TFLOPS = 1900.0


def bf16_peak(sustained: bool = False):
    """Dense bf16 tensor TFLOP/s: MEASURED_PEAKS.json (burst or sustained), else
    the fallback figure."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as f:
                d = json.load(f)
            k = "bf16_tflops_sustained" if sustained else "bf16_tflops"
            if d.get(k):
                return float(d[k]), "measured"
        except (OSError, ValueError):
            pass
    return FALLBACK_BF16_TFLOPS, "fallback"


def attn_flops(bh: int, seq: int, d: int, causal: bool) -> float:
    """Algorithmic flops of attention: two products of 2 * d flops per visible
    (query, key) pair."""
    pairs = seq * (seq + 1) // 2 if causal else seq * seq
    return 4.0 * bh * d * pairs


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as f:
                d = json.load(f)
            for k in ("hbm_gbs", "hbm_GBs", "hbm_gb_s"):
                if k in d and d[k]:
                    return float(d[k]), "measured"
        except (OSError, ValueError):
            pass
    return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(files=("rr_device.cuh", "rr_engine.cuh", "rr_ops.cuh",
                               "rr_instantiate.cuh", "k_softmax_bf16.cu")):
    """Hash of the sources the cross-entropy kernel is compiled from."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "row_reduction_pass_gb300", "csrc")
    for f in sorted(files):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(key: str):
    """DRAM bytes per launch of `key` from profiles/traffic.txt, if taken on the
    current kernel sources (a line: key bytes source-hash)."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    cur = kernel_source_hash()
    with open(p) as f:
        for ln in f:
            parts = ln.split()
            if len(parts) >= 3 and parts[0] == key and parts[2] == cur:
                return float(parts[1])
    return None


# ------------------------------------------------------------- the workload --

def make_inputs(scale_rows: float = 1.0):
    """Host arrays of the step's workloads (rows scaled for samples): config 2's
    LayerNorm, config 3's causal softmax, the sweep's bf16 LayerNorm cases and
    config 4's cross-entropy."""
    def rows(n):
        return max(1, int(n * scale_rows))
    w = {"ln": synth.make("ln_f32_4096x768", rows=rows(4096))}
    w["sm"] = synth.make("softmax_bf16_causal_65536x512")
    if scale_rows < 1.0:
        w["sm"]["x"] = w["sm"]["x"][:rows(65536)]
    for c in LN_BF16_COLS:
        w[f"lnb{c}"] = synth.make(f"sweep_ln_bf16_c{c}", rows=rows((1 << 24) // c))
    w["xe"] = synth.make("xent_bf16_16384x50304", rows=rows(16384))
    return w


def step_bytes(w):
    """Algorithmic bytes of every launch group of the step, in step order."""
    r, c = w["ln"]["x"].shape
    lf, lb = ln_bytes(r, c, 4)
    out = {"ln_fwd": lf, "softmax": softmax_bytes(*w["sm"]["x"].shape, 2), "ln_bwd": lb}
    for cc in LN_BF16_COLS:
        bf, bb = ln_bytes(*w[f"lnb{cc}"]["x"].shape, 2)
        out[f"ln_bf16_c{cc}_fwd"] = bf
        out[f"ln_bf16_c{cc}_bwd"] = bb
    xe = w["xe"]
    n_ign = int((xe["labels"] == synth.IGNORE_INDEX).sum())
    out["xent"] = xent_bytes(*xe["logits"].shape, 2, n_ign)
    return out


def oracle_step(w):
    """The float64 oracle over every workload of the step (CPU legs only)."""
    import oracle
    ln = w["ln"]
    _, mean, rstd = oracle.ln_fwd(ln["x"], ln["gamma"], ln["beta"], ln["eps"])
    oracle.softmax(w["sm"]["x"])
    oracle.ln_bwd(ln["dy"], ln["x"], mean, rstd, ln["gamma"])
    for c in LN_BF16_COLS:
        b = w[f"lnb{c}"]
        _, m, r = oracle.ln_fwd(b["x"], b["gamma"], b["beta"], b["eps"])
        oracle.ln_bwd(b["dy"], b["x"], m, r, b["gamma"])
    oracle.xent(w["xe"]["logits"], w["xe"]["labels"])


def run_ours(args, rank, world):
    import torch
    import row_reduction_pass_gb300 as rr

    torch.cuda.set_device(rank % max(1, torch.cuda.device_count()))
    dev = torch.device("cuda", torch.cuda.current_device())
    rr.load_library()
    w = make_inputs()
    nbytes = step_bytes(w)
    total_bytes = sum(nbytes.values())

    def bf16(a):
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)

    def host(a):
        return (bf16(a) if a.dtype == np.uint16 else torch.from_numpy(a)).pin_memory()

    # pinned host copies (for the end-to-end leg) and device-resident inputs
    h = {}
    for k in ["ln"] + [f"lnb{c}" for c in LN_BF16_COLS]:
        for t in ("x", "gamma", "beta", "dy"):
            h[f"{k}_{t}"] = host(w[k][t])
    h["sm_x"] = host(w["sm"]["x"])
    h["xe_x"] = host(w["xe"]["logits"])
    h["xe_l"] = host(w["xe"]["labels"])
    d = {k: v.to(dev) for k, v in h.items()}
    o = {"sm_y": torch.empty_like(d["sm_x"]),
         "xe_loss": torch.empty(w["xe"]["logits"].shape[0], device=dev)}
    ws = {}
    for k in ["ln"] + [f"lnb{c}" for c in LN_BF16_COLS]:
        x = d[f"{k}_x"]
        R, C = x.shape
        o[f"{k}_y"], o[f"{k}_dx"] = torch.empty_like(x), torch.empty_like(x)
        o[f"{k}_mean"] = torch.empty(R, device=dev)
        o[f"{k}_rstd"] = torch.empty(R, device=dev)
        o[f"{k}_dg"], o[f"{k}_db"] = torch.empty_like(d[f"{k}_gamma"]), torch.empty_like(
            d[f"{k}_gamma"])
        ws[k] = torch.empty(max(1, rr.rr_layernorm_bwd_workspace_size(R, C, x.dtype)),
                            dtype=torch.uint8, device=dev)

    def ln_fwd(k):
        rr.rr_layernorm_fwd(d[f"{k}_x"], d[f"{k}_gamma"], d[f"{k}_beta"], o[f"{k}_y"],
                            o[f"{k}_mean"], o[f"{k}_rstd"], eps=w[k]["eps"])

    def ln_bwd(k):
        rr.rr_layernorm_bwd(d[f"{k}_dy"], d[f"{k}_x"], o[f"{k}_mean"], o[f"{k}_rstd"],
                            d[f"{k}_gamma"], o[f"{k}_dx"], o[f"{k}_dg"], o[f"{k}_db"], ws[k])

    # the step, in order: (name, call, kernel launches); the names match nbytes
    stages = [("ln_fwd", lambda: ln_fwd("ln"), 1),
              ("softmax", lambda: rr.rr_softmax_fwd(d["sm_x"], o["sm_y"]), 1),
              ("ln_bwd", lambda: ln_bwd("ln"), 2)]
    for c in LN_BF16_COLS:
        stages.append((f"ln_bf16_c{c}_fwd", (lambda k: lambda: ln_fwd(k))(f"lnb{c}"), 1))
        stages.append((f"ln_bf16_c{c}_bwd", (lambda k: lambda: ln_bwd(k))(f"lnb{c}"), 2))
    stages.append(("xent", lambda: rr.rr_softmax_xent_fwd_bwd(d["xe_x"], d["xe_l"],
                                                               o["xe_loss"], d["xe_x"]), 1))
    assert [n for n, _, _ in stages] == list(nbytes)
    launches_per_step = sum(n for _, _, n in stages)

    def step(ev=None):
        for i, (_, fn, _) in enumerate(stages):
            if ev is not None:
                ev[i].record()
            fn()
        if ev is not None:
            ev[len(stages)].record()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    # The timed steps replay a CUDA graph of one step: the same kernels in the
    # same order, issued by one host call a step, so the host's per-call work
    # (argument checks, planning, Python) cannot leave the GPU idle between
    # kernels on a slow or busy host.  The per-stage durations come from a
    # second, eager pass with events.
    graph = torch.cuda.CUDAGraph()
    gstream = torch.cuda.Stream()
    gstream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(gstream):
        with torch.cuda.graph(graph, stream=gstream):
            step()
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        t_start.record()
        for i in range(args.steps):
            graph.replay()
        t_end.record()
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ms = t_start.elapsed_time(t_end)
    nst = len(stages)
    n_ev = min(args.steps, 200)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)] for _ in range(n_ev)]
    for i in range(n_ev):
        step(evs[i])
    torch.cuda.synchronize()
    per = {n: [e[i].elapsed_time(e[i + 1]) for e in evs] for i, (n, _, _) in enumerate(stages)}
    err = rr.rr.rr_read_device_error(torch.cuda.current_device())

    # end to end through the public API with host buffers: H2D of every input,
    # the step, D2H of the per-row loss and of dgamma / dbeta.
    e2e_steps = max(3, min(args.steps, args.e2e_steps))
    outs = ["xe_loss"] + [f"{k}_{t}" for k in ["ln"] + [f"lnb{c}" for c in LN_BF16_COLS]
                          for t in ("dg", "db")]
    oh = {k: torch.empty_like(o[k], device="cpu").pin_memory() for k in outs}
    h2d = sum(v.numel() * v.element_size() for v in h.values())
    d2h = sum(v.numel() * v.element_size() for v in oh.values())

    # Two sets of device inputs: while step i computes on the current stream,
    # a copy stream brings step i + 1's inputs into the other set (after step
    # i - 1, which used that set, is done with it); the stages look their
    # inputs up in `d` at call time, so each step points `d` at its set.
    # Every step's H2D and D2H lie inside the timed region.
    sets = [{k: d[k] for k in h}, {k: torch.empty_like(d[k]) for k in h}]
    cstream = torch.cuda.Stream()
    cur = torch.cuda.current_stream()
    copied = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]

    def e2e_copy(j):
        with torch.cuda.stream(cstream):
            cstream.wait_event(done[j % 2])
            for k, v in h.items():
                sets[j % 2][k].copy_(v, non_blocking=True)
            copied[j % 2].record(cstream)

    def e2e_run(n):
        for j in range(2):
            done[j].record(cur)
        e2e_copy(0)
        for i in range(n):
            if i + 1 < n:
                e2e_copy(i + 1)
            cur.wait_event(copied[i % 2])
            d.update(sets[i % 2])
            step()
            for k, v in oh.items():
                v.copy_(o[k], non_blocking=True)
            done[i % 2].record(cur)

    e2e_run(max(3, min(args.warmup, 10)))  # warm-up, as for the device-timed steps
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    e2e_run(e2e_steps)
    cur.wait_stream(cstream)
    b.record()
    torch.cuda.synchronize()
    e2e_ms = a.elapsed_time(b) / e2e_steps
    d.update(sets[0])

    # max over ranks
    if world > 1:
        ms, e2e_ms = max_over_ranks([ms, e2e_ms], device=dev)
    if rank != 0:
        return None

    ms_step = ms / args.steps
    peak, peak_src = hbm_peak()
    value = job_value(world, total_bytes, ms_step)
    x_ms = statistics.mean(per["xent"])
    x_gbs = nbytes["xent"] / (x_ms * 1e-3) / 1e9
    traffic = recorded_traffic("xent_bf16_16384x50304")
    kernels = {}
    for k in per:
        t = statistics.median(per[k])
        kernels[k] = {"ms_median": round(t, 5), "bytes": nbytes[k],
                      "gbs": round(nbytes[k] / (t * 1e-3) / 1e9, 1),
                      "frac_of_peak": round(nbytes[k] / (t * 1e-3) / 1e9 / peak, 4)}
    # LayerNorm fwd+bwd pairs: (bytes_fwd + bytes_bwd) / (t_fwd + t_bwd)
    for pre in ["ln"] + [f"ln_bf16_c{c}" for c in LN_BF16_COLS]:
        f, b = kernels[f"{pre}_fwd"], kernels[f"{pre}_bwd"]
        t = f["ms_median"] + b["ms_median"]
        nb = f["bytes"] + b["bytes"]
        kernels[f"{pre}_fwd+bwd"] = {"ms_median": round(t, 5), "bytes": nb,
                                     "gbs": round(nb / (t * 1e-3) / 1e9, 1),
                                     "frac_of_peak": round(nb / (t * 1e-3) / 1e9 / peak, 4)}
    out = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded numpy PCG64, recipes in row_reduction_pass_gb300/synth.py)",
        "config": {"workload": WORKLOAD, "bytes_per_step": total_bytes,
                   "xent_in_place": XENT_IN_PLACE,
                   "storage": "bf16 and f32 tensors (per workload), f32 arithmetic",
                   "l2": "inputs larger than L2: the 3.3 GB xent pass streams through the "
                         "129 MB L2 every step (the LayerNorm and softmax inputs are read "
                         "after it)", "frac_of_peak": round(value / world / peak, 4),
                   "parallelism": f"replicas x{world} (rows are independent; no collective)",
                   "launch": "timed steps replay a CUDA graph of one step (the step's kernels, "
                             "one host call a step); per-kernel times from an eager pass"},
        "kernels": kernels,
        "roofline": {"bound": "hbm", "achieved": round(x_gbs, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(x_gbs / peak, 4),
                     "traffic": traffic,
                     "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum of one "
                                       "full launch (all 16384 rows, not scaled), "
                                       "profiles/traffic.txt; null once the kernel's sources "
                                       "change",
                     "traffic_over_algorithmic": (round(traffic / nbytes["xent"], 4)
                                                  if traffic else None),
                     "kernel": "row_kernel<OpSoftmaxXent bf16 chunks, staged> (xent 16384x50304)",
                     "peak_source": peak_src},
        "clocks": clk.summary(),
        "e2e": {"value": round(job_value(world, total_bytes, e2e_ms), 1), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4), "steps": e2e_steps,
                "overlap": "step i+1's host-to-device copies on a second stream during step i "
                           "(two device input sets); every step's copies are timed"},
        "gpu_launches": launches_per_step * args.steps,
        "device_error_word": err,
    }
    if not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    return out


# ------------------------------------------------------- CPU oracle timing --

def _oracle_sample(frac):
    """Run the oracle over `frac` of every workload of the step; returns
    (algorithmic bytes of the sample, seconds)."""
    w = make_inputs(scale_rows=frac)
    nb = sum(step_bytes(w).values())
    t0 = time.perf_counter()
    oracle_step(w)
    return nb, time.perf_counter() - t0


def _oracle_part(frac, barrier, results):
    """One worker of the N-core oracle timing: draws its share of the sample,
    waits for every worker, then times the oracle over it."""
    import oracle
    oracle.build()
    w = make_inputs(scale_rows=frac)
    nb = sum(step_bytes(w).values())
    barrier.wait()
    t0 = time.perf_counter()
    oracle_step(w)
    results.put((nb, time.perf_counter() - t0))


def _oracle_ncores(frac: float, n: int):
    """The unchanged single-thread oracle in n processes (spawned: safe after
    CUDA work), each over 1/n of the sample, started together; returns
    (bytes, wall seconds of the slowest worker)."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(n)
    results = ctx.Queue()
    procs = [ctx.Process(target=_oracle_part, args=(frac / n, barrier, results)) for _ in range(n)]
    for p in procs:
        p.start()
    got = []
    deadline = time.monotonic() + 180.0
    try:
        while len(got) < n:
            try:
                got.append(results.get(timeout=1.0))
            except Exception:  # queue.Empty: check that every worker is still going
                if time.monotonic() > deadline or any(
                        not p.is_alive() and p.exitcode not in (0, None) for p in procs):
                    raise RuntimeError("an oracle worker failed or ran out of time")
    finally:
        for p in procs:
            p.join(timeout=5)
            if p.is_alive():
                p.terminate()
                p.join(timeout=5)
    return sum(g[0] for g in got), max(g[1] for g in got)


def cpu_baseline(seconds: float):
    """The float64 oracle on the host cores over a bounded sample of the step:
    one thread, and (when the host has more) the same code in one process per
    core; `value` / `cores` are the faster, the single-thread figure is kept."""
    frac = 1 / 512
    nb, t = _oracle_sample(frac)
    if t < seconds / 4:
        frac = min(1.0, frac * seconds / max(t, 1e-3) / 2)
        nb, t = _oracle_sample(frac)
    one = round(nb / t / 1e9, 4)
    out = {"value": one, "unit": "GB/s", "cores": 1, "kind": "oracle", "value_1_thread": one,
           "sample": f"float64 C oracle, single thread, on {frac:.4%} of the rows of every "
                     f"workload of the step ({nb / 1e6:.1f} MB algorithmic) in {t:.2f} s"}
    n = len(os.sched_getaffinity(0))
    if n > 1:
        try:
            nbn, tn = _oracle_ncores(frac, n)
        except Exception as e:  # noqa: BLE001 -- the 1-thread figure still stands
            out["n_core_error"] = str(e)[:200]
            return out
        if nbn / tn / 1e9 > one:
            out.update(value=round(nbn / tn / 1e9, 4), cores=n,
                       sample=f"float64 C oracle in {n} processes (one per core, spawned, "
                              f"started together), each on 1/{n} of {frac:.4%} of the rows of "
                              f"every workload of the step ({nbn / 1e6:.1f} MB algorithmic in "
                              f"all) in {tn:.2f} s; one thread: {one} GB/s")
    return out


def max_over_ranks(values, device=None):
    """Element-wise maximum of per-rank timings across the process group (every
    rank calls it; the job's time is its slowest rank's)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def job_value(world, bytes_per_step, ms_per_step):
    """Whole-job throughput in GB/s: every rank processes its own replica of the
    step's bytes (weak scaling), in the slowest rank's time."""
    return world * bytes_per_step / (ms_per_step * 1e-3) / 1e9


def run_reference(args, rank, world):
    if rank != 0:
        return None
    # per-step sample sized so warmup + steps finish within ~2 minutes
    budget = 120.0 / max(1, args.steps + args.warmup)
    frac = 1 / 2048
    nb, t = _oracle_sample(frac)
    frac = max(1 / 65536, min(1.0, frac * budget / max(t, 1e-4)))
    w = make_inputs(scale_rows=frac)
    nb = sum(step_bytes(w).values())
    for _ in range(args.warmup):
        oracle_step(w)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(w)
        times.append(time.perf_counter() - t0)
    tot = sum(times)
    value = nb * args.steps / tot / 1e9
    sample = (f"float64 C oracle, single thread, {frac:.5%} of the rows of every workload "
              f"per step ({nb / 1e6:.2f} MB algorithmic per step)")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(tot / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (same seeded generators, row sample)",
            "config": {"workload": WORKLOAD, "sample_fraction": frac},
            "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": 1,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_profile_case(args):
    """Runs one kernel of the step alone (W warm-up + K launches) on a smaller
    batch, for ncu captures of a single kernel; prints a one-line summary."""
    import torch
    import row_reduction_pass_gb300 as rr

    dev = torch.device("cuda", 0)
    rr.load_library()

    def bf16(a):
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)

    if args.profile == "xent":
        if args.profile_workload:
            xe = synth.make(args.profile_workload)
        else:
            xe = synth.make("xent_bf16_16384x50304", rows=args.profile_rows or 4096)
        lg = xe["logits"]
        x = bf16(lg) if lg.dtype == np.uint16 else torch.from_numpy(lg).to(dev)
        lab = torch.from_numpy(xe["labels"]).to(dev)
        loss = torch.empty(x.shape[0], device=dev)
        fn = lambda: rr.rr_softmax_xent_fwd_bwd(x, lab, loss, x)  # noqa: E731
    elif args.profile == "attention":
        # causal attention, 8 batches x 16 heads x 512 queries; --profile-rows
        # gives the head dimension (64 by default), --profile-seq the queries
        # (4096: 32 heads, the tensor-bound sweep shape)
        d_head = args.profile_rows or 64
        seq = args.profile_seq or 512
        heads = 128 if seq == 512 else max(1, (32 * 4096) // seq)
        q, k, v = (bf16(a) for a in synth.attn_inputs(heads, seq, d_head, 31 + d_head))
        o = torch.empty_like(q)
        lse = torch.empty((heads, seq), device=dev)
        fn = lambda: rr.rr_attention_fwd(q, k, v, o, lse, causal=True)  # noqa: E731
    elif args.profile == "softmax":
        sm = synth.make("softmax_bf16_causal_65536x512")
        x = bf16(sm["x"])
        y = torch.empty_like(x)
        fn = lambda: rr.rr_softmax_fwd(x, y)  # noqa: E731
    else:
        if args.profile_workload:
            ln = synth.make(args.profile_workload)
        else:
            ln = synth.make("ln_f32_4096x768", rows=args.profile_rows or 4096)

        def tdev(a):
            if a.dtype == np.uint16:
                return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
            return torch.from_numpy(a).to(dev)
        x, g, b, dy = (tdev(ln[k]) for k in ("x", "gamma", "beta", "dy"))
        y = torch.empty_like(x)
        mean = torch.empty(x.shape[0], device=dev)
        rstd = torch.empty(x.shape[0], device=dev)
        rr.rr_layernorm_fwd(x, g, b, y, mean, rstd, eps=ln["eps"])
        dx, dg, db = torch.empty_like(x), torch.empty_like(g), torch.empty_like(g)
        if args.profile == "ln_fwd":
            fn = lambda: rr.rr_layernorm_fwd(x, g, b, y, mean, rstd, eps=ln["eps"])  # noqa: E731
        else:
            fn = lambda: rr.rr_layernorm_bwd(dy, x, mean, rstd, g, dx, dg, db)  # noqa: E731
    for _ in range(args.warmup + args.steps):
        fn()
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": args.profile, "launches": args.warmup + args.steps}))


def run_sweep(args):
    """Times every operation of every measured workload on its own (L2 flushed
    between repetitions by writing a 256 MB buffer and reading another), against
    the HBM roofline.
    Prints one JSON line per case; not the contract line."""
    import torch
    import row_reduction_pass_gb300 as rr

    dev = torch.device("cuda", 0)
    rr.load_library()
    peak, peak_src = hbm_peak()
    # L2 flush between calls: write 256 MB (twice the L2), then read another
    # 256 MB, so the flush's own dirty lines are written back inside the flush
    # and the timed call starts with an L2 of clean lines that hold none of its data
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_rd = torch.zeros(32 << 20, dtype=torch.int64, device=dev)
    flush_sink = torch.zeros((), dtype=torch.int64, device=dev)

    def l2_flush():
        flush.zero_()
        torch.sum(flush_rd, dim=0, out=flush_sink)

    reps = max(3, args.steps)

    def tdev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(a).to(dev)

    def timed(fn):
        """Device time of one call: CUDA-graph replay of `reps` x (L2 flush, call)
        minus the replay of `reps` x (L2 flush), so host launch latency is
        excluded and every call starts with a cold L2."""
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g_both, g_flush = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g_both, stream=s):
                for _ in range(reps):
                    l2_flush()
                    fn()
            with torch.cuda.graph(g_flush, stream=s):
                for _ in range(reps):
                    l2_flush()
        torch.cuda.synchronize()

        def run(gr):
            gr.replay()
            torch.cuda.synchronize()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            gr.replay()
            b.record()
            torch.cuda.synchronize()
            return a.elapsed_time(b)

        t_both = min(run(g_both) for _ in range(3))
        t_flush = min(run(g_flush) for _ in range(3))
        return max(t_both - t_flush, 1e-6) / reps

    def report(name, op, nbytes, ms):
        gbs = nbytes / (ms * 1e-3) / 1e9
        print(json.dumps({"case": name, "op": op, "bytes": nbytes, "us": round(ms * 1e3, 2),
                          "gbs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
                          "peak": peak, "peak_source": peak_src}), flush=True)

    names = ["xent_f32_64x1000", "ln_f32_4096x768", "softmax_bf16_causal_65536x512",
             "xent_bf16_16384x50304"]
    names += [f"sweep_{k}_{dt}_c{c}" for dt in ("f32", "bf16") for c in synth.SWEEP_COLS
              for k in ("xent", "ln")]
    if args.cases:
        names = [n for n in names if any(c in n for c in args.cases.split(","))]
    for name in names:
        d = synth.make(name)
        e = 2 if d["dtype"] == "bf16" else 4
        if d["kind"] == "xent":
            x, lab = tdev(d["logits"]), tdev(d["labels"])
            R, C = x.shape
            loss = torch.empty(R, device=dev)
            y = torch.empty_like(x)
            n_ign = int((d["labels"] == synth.IGNORE_INDEX).sum())
            ms = timed(lambda: rr.rr_softmax_xent_fwd_bwd(x, lab, loss, y))
            report(name, "xent", xent_bytes(R, C, e, n_ign), ms)
            # the softmax family on the same logits: log-softmax forward, and the
            # softmax / log-softmax backward with a second, distinct input (dy)
            report(name, "log_softmax", softmax_bytes(R, C, e),
                   timed(lambda: rr.rr_log_softmax_fwd(x, y)))
            dyt = x.clone()
            report(name, "softmax_bwd", 3 * R * C * e, timed(lambda: rr.rr_softmax_bwd(x, dyt, y)))
            report(name, "log_softmax_bwd", 3 * R * C * e,
                   timed(lambda: rr.rr_log_softmax_bwd(x, dyt, y)))
            del dyt
        elif d["kind"] == "causal":
            x = tdev(d["x"])
            y = torch.empty_like(x)
            ms = timed(lambda: rr.rr_softmax_fwd(x, y))
            report(name, "softmax", softmax_bytes(*x.shape, e), ms)
        else:
            x, g, b, dy = (tdev(d[k]) for k in ("x", "gamma", "beta", "dy"))
            R, C = x.shape
            y, dx = torch.empty_like(x), torch.empty_like(x)
            mean, rstd = torch.empty(R, device=dev), torch.empty(R, device=dev)
            dg, db = torch.empty_like(g), torch.empty_like(g)
            ws = torch.empty(max(1, rr.rr_layernorm_bwd_workspace_size(R, C, x.dtype)),
                             dtype=torch.uint8, device=dev)
            fb, bb = ln_bytes(R, C, e)
            mf = timed(lambda: rr.rr_layernorm_fwd(x, g, b, y, mean, rstd, eps=d["eps"]))
            mb = timed(lambda: rr.rr_layernorm_bwd(dy, x, mean, rstd, g, dx, dg, db, ws))
            report(name, "ln_fwd", fb, mf)
            report(name, "ln_bwd", bb, mb)
            report(name, "ln_fwd+bwd", fb + bb, mf + mb)
            if rr.rr_rmsnorm_bwd_workspace_size(R, C, x.dtype) > 0:
                # RMSNorm on the same rows (rows of up to 8192 columns)
                ws_r = torch.empty(rr.rr_rmsnorm_bwd_workspace_size(R, C, x.dtype),
                                   dtype=torch.uint8, device=dev)
                rf, rb = rms_bytes(R, C, e)
                tf = timed(lambda: rr.rr_rmsnorm_fwd(x, g, y, rstd, eps=d["eps"]))
                tb = timed(lambda: rr.rr_rmsnorm_bwd(dy, x, rstd, g, dx, dg, ws_r))
                report(name, "rms_fwd", rf, tf)
                report(name, "rms_bwd", rb, tb)
                report(name, "rms_fwd+bwd", rf + rb, tf + tb)
        del d
        torch.cuda.empty_cache()
    if not args.cases or "attention" in args.cases:
        # the online softmax extended to causal attention: 8 batches x 16 heads
        # x 512 queries (the causal softmax's shape), head_dim 64 and 128, bf16
        # At these sizes the kernel's floor is set by HBM, not the tensor cores:
        # q, k, v read once and o written once (L2 is flushed before each call)
        # take longer at the measured copy bandwidth than the two products at
        # the measured bf16 rate, so the line reports both and the fraction of
        # the larger floor (the roofline time) that the kernel reaches.
        # Two more lines at 32 heads x 4096 queries, where the products
        # outweigh the tensors' traffic and the tensor-core rate is the bound.
        tpk, tsrc = bf16_peak()
        hpk, hsrc = hbm_peak()
        for bh, seq, d_head in ((128, 512, 64), (128, 512, 128), (32, 4096, 64), (32, 4096, 128)):
            q, k, v = (tdev(a) for a in synth.attn_inputs(bh, seq, d_head, 31 + d_head))
            o = torch.empty_like(q)
            lse = torch.empty((bh, seq), device=dev)
            ms = timed(lambda: rr.rr_attention_fwd(q, k, v, o, lse, causal=True))
            fl = attn_flops(bh, seq, d_head, True)
            nbytes = 4 * bh * seq * d_head * 2 + bh * seq * 4  # q, k, v, o (bf16), lse
            t_tensor, t_hbm = fl / (tpk * 1e12) * 1e6, nbytes / (hpk * 1e9) * 1e6  # us
            us = ms * 1e3
            print(json.dumps({"case": f"attention_bf16_{bh}x{seq}x{d_head}_causal", "op": "attention",
                              "flops": fl, "bytes": nbytes, "us": round(us, 2),
                              "tflops": round(fl / (ms * 1e-3) / 1e12, 1),
                              "frac_of_tensor_peak": round(fl / (ms * 1e-3) / 1e12 / tpk, 4),
                              "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
                              "frac_of_hbm_peak": round(nbytes / (ms * 1e-3) / 1e9 / hpk, 4),
                              "bound": "hbm" if t_hbm >= t_tensor else "tensor",
                              "roofline_us": round(max(t_tensor, t_hbm), 2),
                              "frac_of_roofline": round(max(t_tensor, t_hbm) / us, 4),
                              "tensor_peak": tpk, "hbm_peak": hpk,
                              "peak_source": tsrc if tsrc == hsrc else f"{tsrc}/{hsrc}"}), flush=True)
            del q, k, v, o, lse
    if not args.cases or "graph" in args.cases:
        run_graph_lines(rr, torch, dev)


def run_graph_lines(rr, torch, dev, iters=200):
    """Small shapes, where host launch overhead dominates: the per-step time of
    back-to-back eager calls against the replay of a CUDA graph of the same
    calls (LayerNorm fwd -> bwd at 4096 x 768 fp32, cross-entropy at 64 x 1000
    fp32).  L2-warm on purpose: these inputs fit in L2 whichever way they run."""
    ln = synth.make("ln_f32_4096x768")
    x, g, b, dy = (torch.from_numpy(ln[k]).to(dev) for k in ("x", "gamma", "beta", "dy"))
    R, C = x.shape
    y, dx = torch.empty_like(x), torch.empty_like(x)
    mean, rstd = torch.empty(R, device=dev), torch.empty(R, device=dev)
    dg, db = torch.empty_like(g), torch.empty_like(g)
    ws = torch.empty(rr.rr_layernorm_bwd_workspace_size(R, C, x.dtype), dtype=torch.uint8,
                     device=dev)
    xe = synth.make("xent_f32_64x1000")
    lx = torch.from_numpy(xe["logits"]).to(dev)
    lab = torch.from_numpy(xe["labels"]).to(dev)
    loss, dl = torch.empty(lx.shape[0], device=dev), torch.empty_like(lx)
    steps = {
        "ln_f32_4096x768 fwd+bwd": (lambda: (rr.rr_layernorm_fwd(x, g, b, y, mean, rstd),
                                             rr.rr_layernorm_bwd(dy, x, mean, rstd, g, dx, dg, db,
                                                                 ws)), 3),
        "xent_f32_64x1000": (lambda: rr.rr_softmax_xent_fwd_bwd(lx, lab, loss, dl), 1),
    }
    for name, (fn, nl) in steps.items():
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            for _ in range(iters):
                fn()
            e.record(s)
            torch.cuda.synchronize()
            eager = a.elapsed_time(e) / iters
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=s):
                fn()
            graph.replay()
            torch.cuda.synchronize()
            a.record(s)
            for _ in range(iters):
                graph.replay()
            e.record(s)
            torch.cuda.synchronize()
            rep = a.elapsed_time(e) / iters
        print(json.dumps({"case": name, "op": "eager_vs_graph", "kernels_per_step": nl,
                          "eager_us": round(eager * 1e3, 2), "graph_us": round(rep * 1e3, 2)}),
              flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", choices=["xent", "softmax", "ln_fwd", "ln_bwd", "attention"],
                    default=None,
                    help="run only this kernel (for ncu captures of one kernel)")
    ap.add_argument("--profile-rows", type=int, default=0)
    ap.add_argument("--profile-seq", type=int, default=0, help="queries for --profile attention")
    ap.add_argument("--profile-workload", default="", help="LayerNorm workload name for --profile")
    ap.add_argument("--sweep", action="store_true",
                    help="time every workload and sweep case separately (one JSON line each)")
    ap.add_argument("--cases", default="", help="comma-separated name filters for --sweep")
    args = ap.parse_args()
    if args.sweep:
        run_sweep(args)
        return
    if args.profile:
        run_profile_case(args)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        out = run_reference(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    out = run_ours(args, rank, world)
    if out is not None:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
