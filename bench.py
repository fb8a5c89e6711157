"""Benchmark of the attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--workload NAME] [--split heads|strong|replicate]
                    [--no-e2e] [--no-cpu-baseline] [--no-extras]

One step is one fa_fwd launch over the whole workload (default: batch 8,
32 heads, N = 8192, head dim 64, bf16, non-causal -- the headline shape of
the pages' forward-time tables).  Inputs are seeded synthetic N(0, 1) data
already resident in HBM; they are 805 MB, larger than the 129 MB L2, so
no flush is needed between steps (smaller workloads rotate through enough
input sets that no step reads inputs left in L2 by the previous ones).
The metric is the attention-forward throughput, 4*B*H*N^2*d counted FLOPs
per step (half when causal), in TFLOPS.  Prints one JSON line on rank 0.
At one GPU the line also carries ``extras``: short event-timed runs of the
rest of the forward table (the N sweep 512..8192 causal and not, the fp16
N = 512 case, the long-context d = 128 case, the e4m3 forward) and of the
backward, each with its own kernel time, fraction of peak and clock record.

Under torchrun (N > 1) the (batch, head) problems are split over the ranks
with ``fwd_shard`` (no data exchange).  ``--split heads`` (default): the
global workload has N times the batch, every rank computes its B*H share
(weak scaling); ``--split strong``: the one workload is split (strong
scaling); ``--split replicate``: every rank runs its own seeded copy.  value
is the FLOPs of all ranks over the slowest rank's time.

``--impl reference`` times the fp64 CPU oracle on the host cores instead,
on a bounded sample of the same workload per step (rank 0 only).

``--impl standard`` times the unfused "standard" attention the pages compare
against (score matrix materialised in HBM, softmax, second product; torch
and cuBLAS on the GPU, one batch element at a time to bound memory).  It is
a comparator for the pages' "标准" columns, not a check of results.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from exact_attention_39_gb300 import workloads as W  # noqa: E402

METRIC = "attn fwd TFLOPS & % of GB300 BF16 tensor peak (B8 H32 d64, N=512–8192)"
UNIT = "TFLOPS"
# NVIDIA's dense (no 2:4 sparsity) bf16 tensor figure for one GB300 GPU.
DATASHEET_TFLOPS = 2250.0
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
                  "bf16_tflops_sustained": 1700.0}
WORKLOADS = {w.name: w for w in
             [W.TINY, W.N512, W.N512_Q8, W.N2048, W.N2048_CAUSAL, W.N8192,
              W.N8192_CAUSAL, W.LONG, W.N8192_E4M3, W.N8192_E4M3_CAUSAL, W.LONG_E4M3]
             + W.sweep(False) + W.sweep(True)}
DEFAULT_WORKLOAD = W.N8192.name
# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from an
# ncu capture of the kernel, keyed by a hash of the kernel sources and the
# workload; reported only while the sources are unchanged.
MEASURED_TRAFFIC = {
    ("73f65183777beac0", "b8h32n8192d64_bf16"): 805581568.0 + 252197120.0,
}
CLOCK_FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw",
                "clocks_event_reasons.active",
                "clocks_event_reasons.hw_slowdown",
                "clocks_event_reasons.hw_thermal_slowdown",
                "clocks_event_reasons.sw_thermal_slowdown",
                "clocks_event_reasons.sw_power_cap"]


# ---------------------------------------------------------------- helpers
def kernel_source_hash():
    """Hash of the forward kernel's device code (the traffic figures below
    were captured with exactly this code).  Line comments, trailing blanks
    and empty lines are left out, so that editing a comment keeps the key."""
    csrc = os.path.join(ROOT, "exact_attention_39_gb300", "csrc")
    texts = []
    for f in ("fa_fwd_kernel.cuh", "ptx.cuh"):
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            texts.append(fh.read())
    return code_digest(texts)


def code_digest(texts):
    """16 hex digits of SHA-256 over the code lines of C++/CUDA sources:
    line comments, trailing blanks and empty lines do not count."""
    import hashlib
    import re
    h = hashlib.sha256()
    for text in texts:
        for line in text.splitlines():
            code = re.sub(r"//.*", "", line).rstrip()
            if code:
                h.update(code.encode("utf-8") + b"\n")
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(local_ms, local_units, world):
    """Max of the per-rank times and sum of the per-rank work units over
    the process group (identity for one process).  Returns (ms, units)."""
    if world == 1:
        return float(local_ms), float(local_units)
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) \
        if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=dev)
    u = torch.tensor([float(local_units)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    def __init__(self, gpu_index, period_ms=50):
        self.gpu_index = gpu_index
        self.period_ms = period_ms
        self.proc = None
        self.path = None

    def __enter__(self):
        self.path = os.path.join(tempfile.gettempdir(), "fa_clocks_%d.csv" % os.getpid())
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index),
                 "--query-gpu=" + ",".join(CLOCK_FIELDS), "--format=csv,noheader,nounits",
                 "-lms", str(self.period_ms)], stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) == len(CLOCK_FIELDS):
                    rows.append(dict(zip(CLOCK_FIELDS, parts)))
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        power = [num(r["power.draw"]) for r in rows]
        sm = [num(r["clocks.sm"]) for r in rows]
        pmax = max(p for p in power if p is not None) if any(p is not None for p in power) else None
        # "under load": samples drawing at least half of the peak power seen
        loaded = [s for s, p in zip(sm, power)
                  if s is not None and (pmax is None or (p is not None and p >= 0.5 * pmax))]
        reasons = set()
        for r in rows:
            for key in CLOCK_FIELDS[5:]:
                if r[key].lower() == "active":
                    reasons.add(key.split(".")[-1])
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": num(rows[0]["clocks.max.sm"]),
                "power_w_max": pmax,
                "samples": len(rows),
                "reasons": sorted(reasons)}


L2_BYTES = 129 * 10 ** 6
# GPU clock cycles of sleep per timed step enqueued ahead of a timed region
# (about 100 us at 2 GHz: more than the host needs to enqueue one step)
SLEEP_CYCLES_PER_STEP = 200000
SLEEP_CYCLES_MAX = 200000000                # about 0.1 s


def set_bytes(w):
    """Bytes one step reads and writes: q, k, v, O and LSE."""
    e = 1 if w.dtype == "e4m3" else 2
    return w.B * w.H * ((w.N + 2 * w.n_keys) * w.d * e + w.N * w.d * 2 + 4 * w.N)


def input_sets(w):
    """How many separate input/output sets the timed steps rotate through so
    that no step finds its inputs in the 129 MB L2: one when a set is larger
    than twice the L2, else enough sets to pass more than twice the L2's
    bytes between two uses of the same set."""
    return max(1, -(-2 * L2_BYTES // set_bytes(w)))


def l2_note(w):
    """How the timed steps stand to the 129 MB L2."""
    mb = (w.N + 2 * w.n_keys) * w.B * w.H * w.d * (1 if w.dtype == "e4m3" else 2) // 10 ** 6
    n = input_sets(w)
    if n == 1:
        return "inputs %d MB > 129 MB L2, no flush" % mb
    return ("inputs %d MB: %d input sets rotated (%d MB between reuses > 129 MB L2), "
            "no flush" % (mb, n, n * set_bytes(w) // 10 ** 6))


def time_oracle(w, budget_s, max_heads, rows_1t=256):
    """Time the fp64 oracle on whole heads of ``w`` until ``budget_s`` of
    work is done, on every host core; then on one core, ``rows_1t`` evenly
    spaced query rows of one head.  Returns (seconds, flops, heads, threads,
    one-core flop/s)."""
    import numpy as np
    import oracle
    q, k, v = W.make_inputs(w.with_(B=1, H=max_heads))
    nt = oracle.default_threads()
    flops, secs, heads = 0.0, 0.0, 0
    for h in range(max_heads):
        qh, kh, vh = (t[0, h].double().numpy() for t in (q, k, v))
        t0 = time.perf_counter()
        oracle.attention_fwd(qh, kh, vh, w.scale, w.causal, nthreads=nt)
        secs += time.perf_counter() - t0
        flops += w.with_(B=1, H=1).flops()
        heads += 1
        if secs >= budget_s:
            break
    qh, kh, vh = (t[0, 0].double().numpy() for t in (q, k, v))
    rows = min(w.N, rows_1t)
    sel = np.arange(rows, dtype=np.int64) * (w.N // rows)
    t0 = time.perf_counter()
    oracle.attention_fwd(qh, kh, vh, w.scale, w.causal, rows=sel, nthreads=1)
    one = time.perf_counter() - t0
    row_flops = 4.0 * w.n_keys * w.d / (2.0 if w.causal else 1.0)
    return secs, flops, heads, nt, row_flops * rows / one


# ---------------------------------------------------------------- timing
def time_launches(step, n_sets, warmup, steps, stream, local):
    """Run ``step(i)`` (launching on ``stream``) ``warmup`` times untimed,
    then ``steps`` times, each bracketed by CUDA events on ``stream``, while
    nvidia-smi samples the clocks.  ``i`` cycles over ``n_sets`` input sets.
    Returns (region ms, per-launch ms list, clock summary)."""
    # inputs and outputs were made on the device's current stream: the
    # launches on ``stream`` come after that work
    stream.wait_stream(torch.cuda.current_stream(stream.device))
    for i in range(warmup):
        step(i % n_sets)
    stream.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    torch.cuda.synchronize(local)
    with ClockSampler(local) as clocks:
        # a short sleep kernel holds the stream while the host enqueues every
        # timed launch, so launches run back to back and the events bracket
        # the kernels, not the host's time to enqueue the next one (which can
        # exceed a short kernel)
        sleep = getattr(torch.cuda, "_sleep", None)   # torch's clock-bounded spin kernel
        if sleep is not None:
            with torch.cuda.stream(stream):
                sleep(min(SLEEP_CYCLES_PER_STEP * steps, SLEEP_CYCLES_MAX))
        for i in range(steps):
            starts[i].record(stream)
            step((warmup + i) % n_sets)
            ends[i].record(stream)
        stream.synchronize()
    torch.cuda.synchronize(local)
    return (starts[0].elapsed_time(ends[-1]),
            [s.elapsed_time(e) for s, e in zip(starts, ends)], clocks.summary())


def fwd_step_fn(fa, w, sets, stream):
    """One forward launch on input set i (fa_fwd, or fa_fwd_fp8 for e4m3)."""
    fp8 = w.dtype == "e4m3"

    def step(i):
        q, k, v, o, lse = sets[i]
        if fp8:
            ds = W.E4M3_DESCALE
            fa.fwd_fp8(q, k, v, ds, ds, ds, causal=w.causal, scale=w.scale,
                       out=o, lse=lse, stream=stream)
        else:
            fa.fwd(q, k, v, causal=w.causal, scale=w.scale, out=o, lse=lse,
                   stream=stream)
    return step


def fwd_outputs(w, q):
    o = torch.empty(q.shape, dtype=torch.bfloat16 if w.dtype == "e4m3" else q.dtype,
                    device=q.device)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=q.device)
    return o, lse


def peak_tflops(fp8=False):
    """The measured bf16 burst peak (x 2, the nominal fp8/bf16 dense ratio,
    for e4m3 contractions) and a description of where it came from."""
    peaks, src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    desc = ("%s bf16 burst (MEASURED_PEAKS.json)" % src if src == "measured"
            else "fallback 1.9 PFLOP/s bf16")
    if fp8:
        return 2.0 * peak, desc + " x 2 (nominal fp8/bf16 ratio)"
    return peak, desc


EXTRA_FWD = (W.sweep(False) + W.sweep(True)
             + [W.N512, W.LONG, W.N8192_E4M3, W.N8192_E4M3_CAUSAL, W.LONG_E4M3])
EXTRA_BWD = [W.N2048, W.N2048_CAUSAL, W.N8192, W.N8192_CAUSAL, W.LONG]


def run_extras(args, local):
    """Short event-timed runs of the rest of the forward table and of the
    backward, one record each (kernel time, TFLOPS, fraction of the peak,
    clocks).  Inputs are drawn on the device (seeded); parity on these shapes
    is the tests' business."""
    import exact_attention_39_gb300 as fa
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)
    out = []
    for w in EXTRA_FWD:
        n = input_sets(w)
        sets = []
        for s in range(n):
            q, k, v = W.make_inputs_on(w.with_(seed=w.seed + s), dev)
            sets.append((q, k, v) + fwd_outputs(w, q))
        _, ks, clk = time_launches(fwd_step_fn(fa, w, sets, stream), n, args.extra_warmup,
                                   args.extra_steps, stream, local)
        if fa.last_device_error(stream) != 0:
            raise RuntimeError("device status set while timing %s" % w.name)
        peak, _ = peak_tflops(w.dtype == "e4m3")
        avg = sum(ks) / len(ks)
        tf = w.flops() / (avg * 1e-3) / 1e12
        out.append({"pass": "fwd", "workload": w.name, "B": w.B, "H": w.H, "N": w.N,
                    "d": w.d, "dtype": w.dtype, "causal": w.causal,
                    "kernel_ms": avg, "kernel_ms_median": sorted(ks)[len(ks) // 2],
                    "tflops": tf, "frac": tf / peak, "l2": l2_note(w), "clocks": clk})
        del sets
    for w in EXTRA_BWD:
        q, k, v = W.make_inputs_on(w, dev)
        g = torch.randn(q.shape, generator=torch.Generator(device=dev).manual_seed(w.seed + 1000),
                        device=dev).to(q.dtype)
        o, lse = fa.fwd(q, k, v, causal=w.causal, scale=w.scale)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(fa.bwd_workspace_bytes(w.B, w.H, w.N), dtype=torch.uint8, device=dev)

        def step(i):
            fa.bwd(q, k, v, o, lse, g, causal=w.causal, scale=w.scale, dq=dq, dk=dk,
                   dv=dv, workspace=ws, stream=stream)
        _, ks, clk = time_launches(step, 1, args.extra_warmup, args.extra_steps, stream, local)
        if fa.last_device_error(stream) != 0:
            raise RuntimeError("device status set while timing the backward of %s" % w.name)
        peak, _ = peak_tflops()
        avg = sum(ks) / len(ks)
        tf = 2.5 * w.flops() / (avg * 1e-3) / 1e12
        out.append({"pass": "bwd", "workload": w.name, "B": w.B, "H": w.H, "N": w.N,
                    "d": w.d, "dtype": w.dtype, "causal": w.causal,
                    "kernel_ms": avg, "kernel_ms_median": sorted(ks)[len(ks) // 2],
                    "tflops": tf, "frac": tf / peak,
                    "flops_convention": "10*B*H*N^2*d, half causal", "clocks": clk})
        del q, k, v, g, o, lse, dq, dk, dv, ws
    return out


# ---------------------------------------------------------------- arms
def run_reference(args, w, world, rank):
    """The oracle on the host cores: each step is a bounded sample of the
    workload (a block of query rows of one head)."""
    if rank != 0:
        return None
    import numpy as np
    import oracle
    rows = min(w.N, args.ref_rows)
    q, k, v = W.make_inputs(w.with_(B=1, H=1))
    qh, kh, vh = (t[0, 0].double().numpy() for t in (q, k, v))
    sel = np.arange(rows, dtype=np.int64) * (w.N // rows)
    nt = oracle.default_threads()
    row_flops = 4.0 * w.n_keys * w.d / (2.0 if w.causal else 1.0)
    for _ in range(args.warmup):
        oracle.attention_fwd(qh, kh, vh, w.scale, w.causal, rows=sel, nthreads=nt)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.attention_fwd(qh, kh, vh, w.scale, w.causal, rows=sel, nthreads=nt)
    secs = time.perf_counter() - t0
    value = row_flops * rows * args.steps / secs / 1e12
    sample = ("%d query rows (every %d-th) of one head of %s per step, fp64, "
              "%d threads" % (rows, w.N // rows, w.name, nt))
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                   "causal": w.causal, "sample": sample},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": nt,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def standard_attention(q, k, v, causal, scale, out=None):
    """Unfused attention with library calls, one batch element at a time:
    S = scale * Q K^T materialised in the input dtype, the causal mask
    (bottom-right aligned: key j visible to query i iff j <= i + Nk - Nq),
    softmax in fp32, P rounded to the input dtype, O = P V.  q [B, H, Nq, d],
    k and v [B, H, Nk, d]; returns O like q.  A query row that sees no key
    (Nq > Nk, causal) has no softmax and comes out NaN."""
    nq, nk = q.shape[2], k.shape[2]
    o = torch.empty_like(q) if out is None else out
    mask = None
    if causal:
        mask = torch.ones(nq, nk, dtype=torch.bool, device=q.device).tril(nk - nq)
    for b in range(q.shape[0]):
        s_ = torch.matmul(q[b], k[b].transpose(-1, -2)) * scale
        if mask is not None:
            s_ = s_.masked_fill(~mask, float("-inf"))
        p_ = torch.softmax(s_.float(), dim=-1).to(q.dtype)
        torch.matmul(p_, v[b], out=o[b])
    return o


def run_standard(args, w, world, rank, local):
    """The unfused comparator on the GPU (torch/cuBLAS): same FLOP count as
    fa_fwd."""
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    q, k, v = (t.to(dev) for t in W.make_inputs(w.with_(seed=w.seed + rank)))
    o = torch.empty_like(q)

    def step():
        standard_attention(q, k, v, w.causal, w.scale, out=o)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    barrier(world)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(args.steps):
        step()
    t1.record()
    torch.cuda.synchronize(dev)
    ms, flops_all = aggregate(t0.elapsed_time(t1), w.flops() * args.steps, world)
    if rank != 0:
        return None
    value = flops_all / (ms * 1e-3) / 1e12
    return {"impl": "standard", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N,
                       "d": w.d, "causal": w.causal,
                       "method": "materialised S (dtype), fp32 softmax, torch/cuBLAS"}}


def run_bwd(args, w, world, rank, local):
    """The backward (fa_bwd: row sums, dQ kernel, dK/dV kernel) per step, on
    the forward's own O and LSE.  Counted FLOPs: 2.5x the forward's
    (10*B*H*N^2*d, half when causal), the usual convention for the five
    products of the backward; the kernels execute seven (S and dP are
    computed in both the dQ and the dK/dV kernel)."""
    import exact_attention_39_gb300 as fa
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    q, k, v = (t.to(dev) for t in W.make_inputs(w.with_(seed=w.seed + rank)))
    g = W.make_upstream_grad(w).to(dev)
    o, lse = fa.fwd(q, k, v, causal=w.causal, scale=w.scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.bwd_workspace_bytes(w.B, w.H, w.N), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step(i):
        fa.bwd(q, k, v, o, lse, g, causal=w.causal, scale=w.scale, dq=dq, dk=dk,
               dv=dv, workspace=ws, stream=stream)

    barrier(world)
    region_ms, _, clk = time_launches(step, 1, args.warmup, args.steps, stream, local)
    if fa.last_device_error(stream) != 0:
        raise RuntimeError("device status set during the timed region")
    flops = 2.5 * w.flops()
    ms, flops_all = aggregate(region_ms, flops * args.steps, world)
    if rank != 0:
        return None
    peak, _ = peak_tflops()
    value = flops_all / (ms * 1e-3) / 1e12
    return {"pass": "bwd", "metric": "attn bwd TFLOPS (10*B*H*N^2*d counted FLOPs, "
            "half causal)", "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                       "causal": w.causal},
            "gpu_launches": 3 * args.steps,
            "pct_of_peak": 100.0 * value / peak,
            "clocks": clk}


def split_plan(w, world, rank, mode):
    """The problems rank ``rank`` of ``world`` computes under split ``mode``.

    Returns (global workload, h0, h1, scaling): the rank computes the
    flattened (batch, head) problems [h0, h1) of the global workload with
    ``fwd_shard``.  "heads": the global workload has ``world`` times the
    batch, so every rank's share is the B*H problems of ``w`` (weak
    scaling); "strong": ``w`` itself is split; "replicate": every rank runs
    all of ``w`` (its own seeded copy)."""
    from exact_attention_39_gb300.shard import head_range
    if mode == "replicate" or world == 1:
        return w, 0, w.B * w.H, "weak"
    if mode == "heads":
        g = w.with_(B=w.B * world)
        h0, h1 = head_range(g.B * g.H, world, rank)
        return g, h0, h1, "weak"
    if mode == "strong":
        h0, h1 = head_range(w.B * w.H, world, rank)
        return w, h0, h1, "strong"
    raise ValueError("unknown split mode %r" % mode)


def run_gpu(args, w, world, rank, local):
    import exact_attention_39_gb300 as fa

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    fp8 = w.dtype == "e4m3"
    stream = torch.cuda.Stream(device=dev)
    gw, h0, h1, scaling = split_plan(w, world, rank, args.split)
    local_flops = w.flops() * (h1 - h0) / (w.B * w.H)   # this rank's share
    sharded = world > 1 and args.split != "replicate"
    if world == 1:
        # the input recipe itself (CPU generator), as the parity tests draw it
        q_h, k_h, v_h = W.make_inputs(w)
    if sharded:
        if fp8:
            raise SystemExit("--split heads/strong shards the fp16/bf16 forward only")
        # every rank holds the same global inputs and computes its problems
        # [h0, h1) in place with fwd_shard
        q, k, v = W.make_inputs_on(gw, dev)
        n_sets = 1
        o = torch.empty((h1 - h0, w.N, w.d), dtype=q.dtype, device=dev)
        lse = torch.empty((h1 - h0, w.N), dtype=torch.float32, device=dev)

        def step(i):
            fa.fwd_shard(q, k, v, world, rank, causal=w.causal, scale=w.scale,
                         stream=stream, out=o, lse=lse)
    else:
        n_sets = input_sets(w)
        sets = []
        for s in range(n_sets):
            if world == 1 and s == 0:
                q, k, v = (t.to(dev) for t in (q_h, k_h, v_h))
            else:
                q, k, v = W.make_inputs_on(w.with_(seed=w.seed + 97 * rank + s), dev)
            sets.append((q, k, v) + fwd_outputs(w, q))
        q, k, v, o, lse = sets[0]
        step = fwd_step_fn(fa, w, sets, stream)

    barrier(world)
    region_ms, kernel_ms, clk = time_launches(step, n_sets, args.warmup, args.steps,
                                              stream, local)
    barrier(world)
    if fa.last_device_error(stream) != 0:
        raise RuntimeError("device status set during the timed region")

    ms, flops_all = aggregate(region_ms, local_flops * args.steps, world)
    value = flops_all / (ms * 1e-3) / 1e12
    ms_per_step = ms / args.steps
    kern_avg_ms = sum(kernel_ms) / len(kernel_ms)

    # ---- end to end through the public API: host buffers, copies timed
    # (sharded: this rank's problems, uploaded into their places in the
    # global device inputs)
    e2e = None
    if not args.no_e2e and not fp8:
        if sharded:
            flat = lambda t: t.reshape(gw.B * gw.H, *t.shape[2:])[h0:h1].unsqueeze(0)
            qd, kd, vd = flat(q), flat(k), flat(v)
            od, ld = o.unsqueeze(0), lse.unsqueeze(0)
        else:
            qd, kd, vd, od, ld = q, k, v, o, lse
        if world > 1:
            q_h, k_h, v_h = (t.cpu() for t in (qd, kd, vd))
        pin = [t.pin_memory() for t in (q_h, k_h, v_h)]
        o_h = torch.empty_like(pin[0]).pin_memory()
        l_h = torch.empty(tuple(ld.shape), dtype=torch.float32).pin_memory()
        e2e_steps = max(1, min(args.steps, args.e2e_steps))
        for _ in range(2):
            fa.fwd_host(*pin, qd, kd, vd, od, ld, o_h, l_h, causal=w.causal,
                        scale=w.scale, stream=stream)
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            fa.fwd_host(*pin, qd, kd, vd, od, ld, o_h, l_h, causal=w.causal,
                        scale=w.scale, stream=stream)
        e_ms = (time.perf_counter() - t0) * 1e3
        barrier(world)
        e_ms, e_flops = aggregate(e_ms, local_flops * e2e_steps, world)
        h2d = sum(t.numel() * t.element_size() for t in pin)
        d2h = o_h.numel() * o_h.element_size() + l_h.numel() * l_h.element_size()
        e2e = {"value": e_flops / (e_ms * 1e-3) / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": e2e_steps, "ms_per_step": e_ms / e2e_steps}

    extras = None
    if world == 1 and not args.no_extras:
        extras = run_extras(args, local)

    if rank != 0:
        return None
    peak, peak_desc = peak_tflops(fp8)
    achieved = local_flops / (kern_avg_ms * 1e-3) / 1e12
    kern_sorted = sorted(kernel_ms)
    kern_med = kern_sorted[len(kern_sorted) // 2]
    props = torch.cuda.get_device_properties(dev)
    sm_mhz = clk.get("sm_mhz") or 0
    # one exponential per visible score: N*Nk per head, about half when causal
    exps = (h1 - h0) * w.N * w.n_keys / (2.0 if w.causal else 1.0)
    key = (kernel_source_hash(), w.name)
    traffic = args.traffic if args.traffic is not None else MEASURED_TRAFFIC.get(key)
    if args.traffic is not None:
        traffic_src = "given on the command line"
    elif traffic is not None:
        traffic_src = "ncu capture of this kernel source (hash %s)" % key[0]
    else:
        traffic_src = ("not measured for this kernel source (hash %s): no ncu capture "
                       "since the kernel last changed" % key[0])
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_source": peak_desc,
                "traffic": traffic if world == 1 else None,
                "traffic_source": traffic_src,
                "algorithmic_bytes": w.hbm_bytes() * (h1 - h0) / (w.B * w.H),
                "kernel_ms": kern_avg_ms,
                "kernel_ms_median": kern_med, "kernel_ms_min": kern_sorted[0],
                "pct_of_datasheet": 100.0 * achieved / (DATASHEET_TFLOPS * (2 if fp8 else 1)),
                "exp_per_clk_per_sm": (exps / (kern_avg_ms * 1e-3)
                                       / (sm_mhz * 1e6 * props.multi_processor_count)
                                       if sm_mhz else None),
                "hbm_gbs_algorithmic": w.hbm_bytes() * (h1 - h0) / (w.B * w.H)
                / (kern_avg_ms * 1e-3) / 1e9}
    cpu = None
    if not args.no_cpu_baseline and world == 1:   # the CPU leg runs at N = 1 only
        secs, fl, heads, nt, one = time_oracle(w, args.cpu_budget, args.cpu_max_heads)
        cpu = {"value": fl / secs / 1e12, "unit": UNIT, "cores": nt,
               "kind": "oracle",
               "sample": "%d whole head(s) (all %d query rows) of %s, fp64, %.1f s"
                         % (heads, w.N, w.name, secs),
               "value_1_core": one / 1e12,
               "sample_1_core": "256 evenly spaced query rows of one head, 1 thread"}
    if world == 1:
        par = "1 GPU"
    elif args.split == "replicate":
        par = "a seeded copy of the workload per GPU"
    else:
        par = "(batch, head) problems split over %d GPUs (fwd_shard, no collective)" % world
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": scaling, "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                   "causal": w.causal, "global_batch": gw.B if sharded else w.B * world,
                   "seq_len": w.N, "parallelism": par, "split": args.split,
                   "l2": l2_note(w) if not sharded else "inputs > 129 MB L2, no flush"},
        "gpu_launches": args.steps,
        "pct_of_peak": 100.0 * achieved / peak,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "clocks": clk,
    }
    if extras is not None:
        line["extras"] = extras
    return line


def parse_shape(text):
    """"B,H,N,d,dtype[,causal]" -> a Workload named like the others."""
    parts = [p.strip() for p in text.split(",")]
    if len(parts) not in (5, 6) or parts[4] not in W.DTYPES:
        raise SystemExit("--shape wants B,H,N,d,dtype[,causal], dtype one of %s"
                         % ", ".join(sorted(W.DTYPES)))
    B, H, N, d = (int(x) for x in parts[:4])
    causal = len(parts) == 6 and parts[5].lower() in ("1", "causal", "true")
    name = "b%dh%dn%dd%d_%s%s" % (B, H, N, d, parts[4], "_causal" if causal else "")
    return W.Workload(name, B, H, N, d, parts[4], causal, seed=0,
                      in_mult=0.5 if d == 128 else 1.0)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["gb300", "reference", "standard"], default="gb300")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--shape", default=None,
                    help="B,H,N,d,dtype[,causal]: a workload of another shape (for "
                         "profiling small cases); overrides --workload")
    ap.add_argument("--pass", dest="pass_", choices=["fwd", "bwd"], default="fwd",
                    help="time the forward (default, the headline) or fa_bwd")
    ap.add_argument("--split", choices=["heads", "strong", "replicate"], default="heads",
                    help="how N > 1 ranks share the (batch, head) problems")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--cpu-max-heads", type=int, default=16)
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the other forward/backward shapes of the one-GPU line")
    ap.add_argument("--extra-steps", type=int, default=20)
    ap.add_argument("--extra-warmup", type=int, default=5)
    ap.add_argument("--ref-rows", type=int, default=1024,
                    help="query rows per reference step")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch from an ncu capture of this kernel")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "gb300" and args.steps > 3:
        print("note: fewer than 3 warm-up steps", file=sys.stderr)
    world, rank, local = dist_env()
    w = WORKLOADS[args.workload] if args.shape is None else parse_shape(args.shape)
    if world > 1 and args.impl in ("gb300", "standard"):
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    try:
        if args.impl == "reference":
            line = run_reference(args, w, world, rank)
        elif args.impl == "standard":
            line = run_standard(args, w, world, rank, local)
        elif args.pass_ == "bwd":
            line = run_bwd(args, w, world, rank, local)
        else:
            line = run_gpu(args, w, world, rank, local)
        if line is not None:
            print(json.dumps(line), flush=True)
    finally:
        if world > 1 and args.impl in ("gb300", "standard"):
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
