"""Benchmark of the SP-region hot path on GB300.

One step = one pass of the whole hot path over one synthetic batch of the
pages' benchmark shape (T=2, S=2048, B=2, H=768, bf16, RMSNorm, p=0.1):
  forward of every sequence shard (reduce-scatter's reduce, dropout, residual,
  RMSNorm) -> sp2hp of the norm output -> hp2sp back (on a side stream,
  concurrent with) the backward of every shard (norm, residual and dropout
  backward, dgamma).
The timed run is exactly --steps steps, replayed from CUDA graphs of (at
most 512) consecutive steps, each step on its own buffer set; the sets rotate
so that between two uses of a set every kernel's own bytes exceed twice the
L2, so HBM (not L2) serves the inputs.  The timed run is repeated until the
runs cover at least 50 ms (and at least 3 runs); the reported time is the
median run.  The JSON line also carries per-kernel launch times (back to back
and single), the end-to-end number through host buffers, the mask-free step,
the oracle's CPU rate, the clocks seen, and the same per-kernel figures for
the other workloads (GPT LayerNorm, the large-hidden stress case at p = 0.1
and p = 0, and the layout transforms) under "workloads".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Rank 0 prints one JSON line.  Under torchrun rank r plays tensor-parallel
rank r % T of data-parallel replica r // T: it runs its own sequence shard
(forward, layout, backward of shard j = r % T) of its replica's batch, with
no data-path collective (weak scaling once N >= T; one GPU alone plays the
whole tensor-parallel group and runs every shard).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = "pages_rms_bf16"
METRIC = "SP-region fwd+bwd tokens/s and achieved HBM GB/s (% of GB300 peak), 1 GPU"
LAUNCHES_PER_STEP = 5  # fwd, sp2hp, hp2sp, bwd, dgamma column sum
NOMINAL_HBM_GBS = 8000.0  # GB300's nominal HBM3e bandwidth (the measured copy peak is the roofline)
MAX_GRAPH_STEPS = 512
MIN_TIMED_MS = 50.0
# the other workloads reported beside the headline: (key, workload, p override)
EXTRA_WORKLOADS = [("gpt_ln_bf16", "gpt_ln_bf16", None),
                   ("large_rms_bf16_p0.1", "large_rms_bf16", 0.1),
                   ("large_rms_bf16_p0", "large_rms_bf16", 0.0)]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--roofline-iters", type=int, default=400)
    ap.add_argument("--e2e-steps", type=int, default=300)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    ap.add_argument("--seq", type=int, default=None,
                    help="override S (smaller captures of the same kernels for ncu)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# algorithmic bytes (what each launch must move at minimum)
# ---------------------------------------------------------------------------

def fwd_bytes(w, rows):
    e = 2 if w.dtype == "bf16" else 4
    per_elem = w.T * e + e + e + e + (1 if w.p > 0 else 0)  # partials, residual, h, y, mask
    per_row = 4 + (4 if w.norm == "ln" else 0)               # rstd (+ mean)
    return rows * (w.H * per_elem + per_row) + w.H * e * (2 if w.norm == "ln" else 1)


def bwd_bytes(w, rows):
    e = 2 if w.dtype == "bf16" else 4
    per_elem = 5 * e + (1 if w.p > 0 else 0)  # dy, dh_out, h, d_residual, d_sum (+ mask)
    per_row = 4 + (4 if w.norm == "ln" else 0)
    return rows * (w.H * per_elem + per_row) + w.H * (e + 4 * (2 if w.norm == "ln" else 1))


def layout_bytes(w, rows):
    e = 2 if w.dtype == "bf16" else 4
    return 2 * rows * w.H * e


def rotation_sets(l2: int, per_set: int, *kernel_bytes: int) -> int:
    """How many buffer sets the steps rotate over: enough that each kernel's
    own bytes over one rotation exceed twice the L2 (the layout kernel,
    touching only y and y_hp, needs the most), and at least 2."""
    touched = min(per_set, *kernel_bytes)
    return max(2, -(-2 * l2 // touched) + 1)


def graph_steps(steps: int) -> int:
    """Steps per CUDA graph for a timed run of `steps` steps: all of them up
    to MAX_GRAPH_STEPS, else the largest divisor of `steps` not above it."""
    if steps <= MAX_GRAPH_STEPS:
        return steps
    d = max(k for k in range(1, MAX_GRAPH_STEPS + 1) if steps % k == 0)
    if d < 16:
        raise ValueError(f"--steps {steps} has no divisor in [16, {MAX_GRAPH_STEPS}]; pick another count")
    return d


def graph_rotation(g: int, min_sets: int) -> tuple[int, int]:
    """(buffer sets, graph variants) for graphs of g consecutive steps that
    continue one rotation over the sets from replay to replay: at least
    min_sets sets; a multiple of g when g is smaller (variant v starts at set
    v*g), else a divisor of g (every graph starts at set 0)."""
    if g < min_sets:
        n = -(-min_sets // g) * g
        return n, n // g
    n = min(k for k in range(min_sets, g + 1) if g % k == 0)
    return n, 1


def timed_runs(run_once, min_ms: float = MIN_TIMED_MS, min_runs: int = 3, max_runs: int = 1000):
    """Repeat run_once() (which returns its own duration in ms) until the runs
    cover min_ms and there are at least min_runs; returns the durations."""
    out = []
    while len(out) < min_runs or (sum(out) < min_ms and len(out) < max_runs):
        out.append(run_once())
    return out


def tp_dp_rank(rank: int, world: int, T: int) -> tuple[int, int, int]:
    """(first shard j, shards in this rank's call, data-parallel replica) of
    a rank: one GPU alone plays the whole tensor-parallel group (all T
    shards); with N ranks, rank r is tensor-parallel rank r % T of replica
    r // T and owns sequence shard r % T."""
    if world <= 1:
        return 0, T, 0
    return rank % T, 1, rank // T


def packed_block(named, device, pin=False):
    """One flat byte buffer holding tensors shaped like the (name, tensor)
    pairs in `named`, each at a 256-byte aligned offset; returns (flat, views).
    The end-to-end pipeline moves a step's inputs and results as one such
    block each way."""
    import torch

    offs, off = [], 0
    for _, v in named:
        offs.append(off)
        off += -(-v.numel() * v.element_size() // 256) * 256
    flat = torch.empty(off, dtype=torch.uint8, device=device, pin_memory=pin)
    views = [flat[o:o + v.numel() * v.element_size()].view(v.dtype).view(v.shape)
             for o, (_, v) in zip(offs, named)]
    return flat, views


# ---------------------------------------------------------------------------
# multi-rank aggregation (one process per GPU)
# ---------------------------------------------------------------------------

def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time: the job is done when every rank is."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_tokens_per_s(tokens_per_step: int, steps: int, world: int, ms: float) -> float:
    """Whole-job throughput: every rank processed `steps` steps of its own
    `tokens_per_step` token rows in at most `ms` milliseconds."""
    return tokens_per_step * steps * world / (ms / 1e3)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index, enabled=True):
        self.proc = None
        self.idx = device_index
        if enabled:
            try:
                self.f = tempfile.NamedTemporaryFile("w+", prefix=f"spfuse_clocks{device_index}_",
                                                     suffix=".csv", delete=False)
                self.path = self.f.name
                self.proc = subprocess.Popen(
                    ["nvidia-smi", f"--id={device_index}", f"--query-gpu={self.FIELDS}",
                     "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                    stderr=subprocess.DEVNULL)
            except (OSError, FileNotFoundError):
                self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            lines = f.readlines()
        os.unlink(self.path)
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smmax=float(parts[2]),
                                 power=float(parts[3]) if parts[3] not in ("[N/A]", "N/A") else 0.0,
                                 hw=parts[5], hwt=parts[6], swt=parts[7], swp=parts[8]))
            except ValueError:
                continue
        if not rows:
            return None
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows),
                "sm_max_mhz": max(r["smmax"] for r in rows), "samples": len(rows),
                "power_w_max": max(r["power"] for r in rows), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

class Harness:
    """Buffer sets, launch wrappers and graph timing for one workload on one
    rank: shards j .. j+nshards-1 of the workload's batch."""

    def __init__(self, w, dev, j, nshards, seed_offset=0, sets_for=None):
        import torch

        from residual_sp_rs_gb300 import ops, synthetic as syn

        self.torch, self.ops, self.syn = torch, ops, syn
        self.w, self.dev = w, dev
        self.T, self.H = w.T, w.H
        self.rows = w.R * nshards
        self.row0 = w.R * j
        self.desc = ops.make_desc(w.T, j, w.S, w.B, w.H, w.dtype, w.norm, w.p, w.eps, w.seed + seed_offset,
                                  nshards=nshards)
        self.l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.seed_offset = seed_offset
        first = self.make_set(0)
        self.per_set = self.set_bytes(first)
        need = rotation_sets(self.l2, self.per_set, fwd_bytes(w, self.rows), bwd_bytes(w, self.rows),
                             layout_bytes(w, self.rows))
        # sets_for: the caller's set count for this need (e.g. to suit its graphs)
        self.n_sets = sets_for(need) if sets_for else need
        self.sets = [first] + [self.make_set(k) for k in range(1, self.n_sets)]
        self.side = torch.cuda.Stream()
        self.cap_stream = torch.cuda.Stream()

    def make_set(self, k):
        torch, syn, w = self.torch, self.syn, self.w
        seed = w.input_seed + 17 * k + 1000 * self.seed_offset
        inp = syn.fwd_inputs(w, self.dev, seed=seed)
        gr = syn.upstream_grads(w, self.dev, seed=seed)
        rows, H, r0 = self.rows, self.H, self.row0
        tdt = syn.torch_dtype(w.dtype)
        s = dict(partials=inp["partials"], residual=inp["residual"].view(-1, H)[r0:r0 + rows],
                 gamma=inp["gamma"], beta=inp["beta"], dy=gr["dy"].view(-1, H)[r0:r0 + rows],
                 dh=gr["dh_out"].view(-1, H)[r0:r0 + rows])
        s["h"] = torch.empty((rows, H), device=self.dev, dtype=tdt)
        s["y"] = torch.empty((rows, H), device=self.dev, dtype=tdt)
        s["mask"] = torch.empty((rows, H), device=self.dev, dtype=torch.uint8) if w.p > 0 else None
        s["rstd"] = torch.empty(rows, device=self.dev)
        s["mean"] = torch.empty(rows, device=self.dev) if w.norm == "ln" else None
        s["y_hp"] = torch.empty((self.T, rows, H // self.T), device=self.dev, dtype=tdt)
        s["y_sp"] = torch.empty((rows, H), device=self.dev, dtype=tdt)
        s["d_res"] = torch.empty((rows, H), device=self.dev, dtype=tdt)
        s["d_sum"] = torch.empty((rows, H), device=self.dev, dtype=tdt)
        s["dgamma"] = torch.empty(H, device=self.dev)
        s["dbeta"] = torch.empty(H, device=self.dev) if w.norm == "ln" else None
        s["ws"] = self.ops.workspace_for(self.desc, self.dev)
        return s

    def set_bytes(self, s):
        T = self.torch
        return sum(v.numel() * v.element_size() for k, v in s.items()
                   if isinstance(v, T.Tensor)) + sum(p.numel() * p.element_size() for p in s["partials"])

    # ---- launches ---------------------------------------------------------
    def fwd(self, s, mask_free=False):
        self.ops.sp_rs_dropout_residual_norm_fwd(self.desc, s["partials"], s["residual"], s["gamma"],
                                                 s["beta"], s["h"], s["y"],
                                                 None if mask_free else s["mask"], s["rstd"], s["mean"])

    def bwd(self, s, mask_free=False):
        self.ops.sp_rs_dropout_residual_norm_bwd(self.desc, s["dy"], s["dh"], s["h"], s["gamma"],
                                                 None if mask_free else s["mask"], s["rstd"], s["mean"],
                                                 s["d_res"], s["d_sum"], s["dgamma"], s["dbeta"], s["ws"])

    def sp2hp(self, s):
        self.ops.sp2hp(s["y"], s["y_hp"], self.rows, self.H, self.T, self.w.dtype)

    def hp2sp(self, s):
        self.ops.hp2sp(s["y_hp"], s["y_sp"], self.rows, self.H, self.T, self.w.dtype)

    def step(self, s, mask_free=False):
        # the layout transforms of y and the backward both depend only on the
        # forward: they run as two concurrent branches of the step
        torch = self.torch
        self.fwd(s, mask_free)
        cur = torch.cuda.current_stream()
        self.side.wait_stream(cur)
        with torch.cuda.stream(self.side):
            self.sp2hp(s)
            self.hp2sp(s)
        self.bwd(s, mask_free)

    def record_steps(self, n, start, mask_free=False):
        """n consecutive steps from set `start`; the layout branch joins the
        main stream once per rotation over the sets and at the end (no step in
        between touches the buffers it reads or writes)."""
        cur = self.torch.cuda.current_stream()
        for i in range(n):
            k = (start + i) % self.n_sets
            self.step(self.sets[k], mask_free)
            if k == self.n_sets - 1 or i == n - 1:
                cur.wait_stream(self.side)

    def capture(self, fn):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.cap_stream, capture_error_mode="relaxed"):
            fn()
        return g

    def time_launches(self, fn, reps, per_graph=None):
        """Mean duration of one launch of fn over the rotating sets, launched
        back to back from one CUDA graph (median over `reps` replays)."""
        torch = self.torch
        per_graph = per_graph or self.n_sets * max(1, -(-16 // self.n_sets))
        g = self.capture(lambda: [fn(self.sets[i % self.n_sets]) for i in range(per_graph)])
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
        evs[0].record()
        for i in range(reps):
            g.replay()
            evs[i + 1].record()
        torch.cuda.synchronize()
        return float(np.median([evs[i].elapsed_time(evs[i + 1]) for i in range(reps)])) / per_graph

    def time_single(self, fn, reps=50, warm=10):
        """One launch at a time: events around it, a synchronize after each,
        so launch latency is included (median)."""
        torch = self.torch
        out = []
        for i in range(warm + reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn(self.sets[i % self.n_sets])
            b.record()
            torch.cuda.synchronize()
            if i >= warm:
                out.append(a.elapsed_time(b))
        return float(np.median(out))


def _kernel_entry(ms, nbytes, hbm_peak, single=None):
    gbs = nbytes / (ms / 1e3) / 1e9
    d = {"launch_ms": round(ms, 5), "algorithmic_bytes": nbytes, "gbs": round(gbs, 1),
         "frac_of_measured": round(gbs / hbm_peak, 4), "frac_of_nominal_8000": round(gbs / NOMINAL_HBM_GBS, 4)}
    if single is not None:
        d["single_launch_ms"] = round(single, 5)
    return d


def measure_workload(w, dev, hbm_peak, cpu_seconds=None):
    """Per-kernel back-to-back launch times and the step time of another
    workload (all its shards in one call), on sets rotating past the L2."""
    import torch

    hn = Harness(w, dev, 0, w.T)
    rows = hn.rows
    for s in hn.sets:
        hn.step(s)
    torch.cuda.current_stream().wait_stream(hn.side)
    torch.cuda.synchronize()
    reps = 20
    per_graph = max(8, hn.n_sets)
    t_fwd = hn.time_launches(hn.fwd, reps, per_graph)
    t_bwd = hn.time_launches(hn.bwd, reps, per_graph)
    t_sp2hp = hn.time_launches(hn.sp2hp, reps, per_graph)
    g = hn.capture(lambda: hn.record_steps(per_graph, 0))
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    evs[0].record()
    for i in range(reps):
        g.replay()
        evs[i + 1].record()
    torch.cuda.synchronize()
    step_ms = float(np.median([evs[i].elapsed_time(evs[i + 1]) for i in range(reps)])) / per_graph
    out = {"config": f"T={w.T} S={w.S} B={w.B} H={w.H} {w.dtype} {w.norm} p={w.p}, all {w.T} shards "
                     f"in one call; {hn.n_sets} buffer sets",
           "tokens_per_step": rows, "step_ms": round(step_ms, 5),
           "tokens_per_s": round(rows / (step_ms / 1e3), 1),
           "per_kernel": {"fwd": _kernel_entry(t_fwd, fwd_bytes(w, rows), hbm_peak),
                          "bwd": _kernel_entry(t_bwd, bwd_bytes(w, rows), hbm_peak),
                          "sp2hp": _kernel_entry(t_sp2hp, layout_bytes(w, rows), hbm_peak)}}
    del hn, g
    torch.cuda.empty_cache()
    # the same bytes moved by a pure copy in one launch, for scale
    for k in ("fwd", "bwd"):
        e = out["per_kernel"][k]
        cf = measure_copy_floor(dev, e["algorithmic_bytes"], w.H, hbm_peak)
        e["copy_at_same_bytes_gbs"] = cf["gbs"]
        e["frac_of_copy_at_same_bytes"] = round(e["gbs"] / cf["gbs"], 4)
    if cpu_seconds:
        out["cpu_baseline"] = cpu_baseline(w, cpu_seconds)
    return out


def measure_copy_floor(dev, nbytes, H, hbm_peak):
    """sp2hp, a pure copy (each byte read once and written once), of about
    `nbytes` read plus written bytes in rows of H bf16 elements, back to back
    over sets rotating past the L2: what moving that many bytes in one launch
    costs on this GPU, launch and ramp included."""
    import torch

    from residual_sp_rs_gb300 import ops

    T = 2
    N = max(T, int(nbytes // (4 * H)) // T * T)
    byt = 4 * N * H
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    n_sets = max(2, -(-2 * l2 // byt) + 1)
    gen = torch.Generator(device=dev).manual_seed(4242)
    xs = [torch.randn((N, H), device=dev, generator=gen).to(torch.bfloat16) for _ in range(n_sets)]
    ys = [torch.empty((T, N, H // T), device=dev, dtype=torch.bfloat16) for _ in xs]
    cap = torch.cuda.Stream()
    for k in range(n_sets):
        ops.sp2hp(xs[k], ys[k], N, H, T, 1)
    per_graph = max(16, n_sets)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap, capture_error_mode="relaxed"):
        for i in range(per_graph):
            ops.sp2hp(xs[i % n_sets], ys[i % n_sets], N, H, T, 1)
    g.replay()
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(21)]
    evs[0].record()
    for i in range(20):
        g.replay()
        evs[i + 1].record()
    torch.cuda.synchronize()
    ms = float(np.median([evs[i].elapsed_time(evs[i + 1]) for i in range(20)])) / per_graph
    del xs, ys, g
    torch.cuda.empty_cache()
    d = _kernel_entry(ms, byt, hbm_peak)
    d["note"] = (f"sp_layout_kernel (sp2hp, a pure copy) of {byt} read+written bytes, N={N} H={H}, "
                 f"{n_sets} buffer sets, back to back: the cost of moving that many bytes in one launch")
    return d


def measure_layout(dev, hbm_peak):
    """sp2hp and hp2sp alone on the layout workload (T=4, N=16384 tokens,
    H=4096, bf16), back to back over sets rotating past the L2."""
    import torch

    from residual_sp_rs_gb300 import ops, synthetic as syn

    lw = syn.LAYOUT
    nbytes = 2 * lw.N * lw.H * 2
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    n_sets = max(2, -(-2 * l2 // nbytes) + 1)
    xs = [syn.layout_input(lw, dev, seed=lw.input_seed + k) for k in range(n_sets)]
    hps = [torch.empty((lw.T, lw.N, lw.H // lw.T), device=dev, dtype=torch.bfloat16) for _ in xs]
    backs = [torch.empty_like(x) for x in xs]
    cap = torch.cuda.Stream()
    res = {}
    for name, fn in (("sp2hp", lambda k: ops.sp2hp(xs[k], hps[k], lw.N, lw.H, lw.T, lw.dtype)),
                     ("hp2sp", lambda k: ops.hp2sp(hps[k], backs[k], lw.N, lw.H, lw.T, lw.dtype))):
        for k in range(n_sets):
            fn(k)
        per_graph = max(8, n_sets)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap, capture_error_mode="relaxed"):
            for i in range(per_graph):
                fn(i % n_sets)
        g.replay()
        torch.cuda.synchronize()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(21)]
        evs[0].record()
        for i in range(20):
            g.replay()
            evs[i + 1].record()
        torch.cuda.synchronize()
        ms = float(np.median([evs[i].elapsed_time(evs[i + 1]) for i in range(20)])) / per_graph
        res[name] = _kernel_entry(ms, nbytes, hbm_peak)
    torch.cuda.synchronize()
    ok = torch.equal(backs[0], xs[0])
    del xs, hps, backs
    torch.cuda.empty_cache()
    return {"config": f"T={lw.T} N={lw.N} H={lw.H} {lw.dtype}; {n_sets} buffer sets",
            "roundtrip_identity": ok, "per_kernel": res}


def run_ours(args):
    import torch
    import torch.distributed as dist

    from residual_sp_rs_gb300 import build as spbuild
    from residual_sp_rs_gb300 import ops, synthetic as syn

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        spbuild.build()
    if world > 1:
        dist.barrier()
    ops.lib()

    w = syn.WORKLOADS[args.workload]
    if args.seq:
        w = w.with_(S=args.seq)
    T, H = w.T, w.H
    j, nshards, dp = tp_dp_rank(rank, world, T)
    K = args.steps
    G = graph_steps(K)
    # as many sets as the rotation needs, arranged so that graphs of G steps
    # continue the rotation from replay to replay
    hn = Harness(w, dev, j, nshards, seed_offset=dp, sets_for=lambda need: graph_rotation(G, need)[0])
    n_sets = hn.n_sets
    variants = n_sets // G if G < n_sets else 1
    rows = hn.rows

    for s in hn.sets:
        hn.step(s)
    torch.cuda.current_stream().wait_stream(hn.side)
    torch.cuda.synchronize()
    graphs = [hn.capture(lambda v=v: hn.record_steps(G, (v * G) % n_sets)) for v in range(variants)]
    torch.cuda.synchronize()
    state = {"v": 0}

    def run_steps(k):
        # k a multiple of G: consecutive variants continue the rotation
        for _ in range(k // G):
            graphs[state["v"]].replay()
            state["v"] = (state["v"] + 1) % variants

    run_steps(max(args.warmup, 3) // G * G or G)
    torch.cuda.synchronize()

    # ---- timed region: runs of exactly K steps, repeated to >= 50 ms -------------
    clocks = ClockSampler(local, enabled=not args.no_clocks)
    time.sleep(0.2)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()

    def one_run():
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        run_steps(K)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    runs = timed_runs(one_run)
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    ms = max_over_ranks(float(np.median(runs)), world, dev)
    ms_per_step = ms / K
    value = weak_scaling_tokens_per_s(rows, K, world, ms)
    step_bytes = fwd_bytes(w, rows) + bwd_bytes(w, rows) + 2 * layout_bytes(w, rows)
    step_gbs = step_bytes / (ms_per_step / 1e3) / 1e9

    # ---- the mask-free mode (not the headline): the forward stores no mask and
    # the backward draws the keep bits again -- 2 bytes per element less
    # traffic, Philox twice
    mask_free = None
    if w.p > 0:
        gmf = [hn.capture(lambda v=v: hn.record_steps(G, (v * G) % n_sets, mask_free=True))
               for v in range(variants)]
        for g in gmf:
            g.replay()
        torch.cuda.synchronize()
        mf = {"v": 0}

        def one_mf():
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(K // G):
                gmf[mf["v"]].replay()
                mf["v"] = (mf["v"] + 1) % variants
            e1.record()
            torch.cuda.synchronize()
            return e0.elapsed_time(e1)

        ms_mf = max_over_ranks(float(np.median(timed_runs(one_mf))), world, dev) / K
        mask_free = {"ms_per_step": round(ms_mf, 6),
                     "value": round(weak_scaling_tokens_per_s(rows, 1, world, ms_mf), 1),
                     "unit": "tokens/s",
                     "note": "same step with the mask pointers NULL: the forward keeps no mask, the "
                             "backward regenerates the keep bits from the seed"}
        del gmf

    # ---- per-launch durations of the main kernels: each kernel alone, launched
    # back to back from one CUDA graph over the rotating sets, CUDA events
    # around the replays on the launching stream
    per_graph = n_sets * max(1, -(-64 // n_sets))
    reps = max(50, args.roofline_iters // per_graph)
    t_fwd = hn.time_launches(hn.fwd, reps, per_graph)
    t_bwd = hn.time_launches(hn.bwd, reps, per_graph)
    t_sp2hp = hn.time_launches(hn.sp2hp, reps, per_graph)
    single = {"fwd": hn.time_single(hn.fwd), "bwd": hn.time_single(hn.bwd), "sp2hp": hn.time_single(hn.sp2hp)}
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except OSError:
        pass
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"
    kern = {"fwd": (t_fwd, fwd_bytes(w, rows), "sp_fwd_tma_kernel"),
            "bwd": (t_bwd, bwd_bytes(w, rows), "sp_bwd_tma_kernel+sp_colsum_kernel"),
            "sp2hp": (t_sp2hp, layout_bytes(w, rows), "sp_layout_kernel")}
    dom = max(("fwd", "bwd"), key=lambda k: kern[k][0])
    d_ms, d_bytes, d_name = kern[dom]
    achieved = d_bytes / (d_ms / 1e3) / 1e9
    traffic = None
    try:
        tr = json.load(open(os.path.join(ROOT, "profiles", f"{dom}_{args.workload}_traffic.json")))
        if tr.get("source_sha256") == spbuild.source_hash() and world == 1 and not args.seq:
            traffic = tr.get("bytes_per_launch")
    except (OSError, ValueError):
        pass
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(achieved / hbm_peak, 4), "traffic": traffic, "kernel": d_name,
                "frac_of_nominal_8000": round(achieved / NOMINAL_HBM_GBS, 4),
                "peak_source": peak_src, "algorithmic_bytes_per_launch": d_bytes,
                "launch_ms": round(d_ms, 5),
                "launch_timing": "launch_ms: median over CUDA graph replays of back-to-back "
                                 "launches over the rotating buffer sets; single_launch_ms: median "
                                 "of 50 launches each alone between events and a synchronize "
                                 "(includes launch latency)",
                "per_kernel": {k: _kernel_entry(v[0], v[1], hbm_peak, single[k]) for k, v in kern.items()}}
    if world == 1 and not args.seq:
        cf = measure_copy_floor(dev, d_bytes, H, hbm_peak)
        roofline["copy_at_same_bytes"] = cf
        roofline["frac_of_copy_at_same_bytes"] = round(achieved / cf["gbs"], 4)

    # ---- end to end: pinned host inputs in, results out, every step -------------
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, w, hn, world)
    del graphs, hn
    torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(w, args.cpu_seconds)

    # ---- the other workloads (one GPU only: per-kernel figures) -----------------
    extra = None
    if world == 1 and not args.no_extra and not args.seq:
        extra = {}
        cpu_s = None if args.no_cpu else 4.0
        for key, name, p in EXTRA_WORKLOADS:
            wx = syn.WORKLOADS[name] if p is None else syn.WORKLOADS[name].with_(p=p)
            extra[key] = measure_workload(wx, dev, hbm_peak, cpu_s)
        extra["layout_bf16"] = measure_layout(dev, hbm_peak)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16"
            if w.dtype == "bf16" else "f32", "data": "synthetic (seeded torch.Generator)",
            "config": {"workload": f"{w.name}: SP region fwd+sp2hp+hp2sp+bwd, T={T} S={w.S} B={w.B} "
                                   f"H={H} {w.dtype} {w.norm} p={w.p}",
                       "T": T, "S": w.S, "B": w.B, "H": H, "norm": w.norm, "p": w.p,
                       "tokens_per_step_per_gpu": rows,
                       "parallelism": ("one GPU plays the whole tensor-parallel group (all shards)"
                                       if world == 1 else
                                       f"rank r runs sequence shard r % {T} of data-parallel replica "
                                       f"r // {T} ({world} ranks)"),
                       "l2": f"inputs rotate over {n_sets} buffer sets, {n_sets * hn_set_mb(w, rows):.0f} MB; "
                             "between two uses of a set each kernel's own bytes exceed 2x L2",
                       "launch": f"timed run = exactly {K} steps from CUDA graphs of {G} steps "
                                 f"({variants} graph variant(s) continuing the rotation), programmatic "
                                 "dependent launch between the kernels of a graph; the layout branch is "
                                 "concurrent with the backward; median of "
                                 f"{len(runs)} timed runs ({sum(runs):.1f} ms in all)"},
            "step_algorithmic_gbs": round(step_gbs, 1),
            "step_algorithmic_gbs_note": "algorithmic bytes of the step's five launches / step time; "
                                         "the backward's reads of h and mask and the layout's read of y "
                                         "are served from L2 right after the forward wrote them, so this "
                                         "is not a DRAM rate",
            "roofline": roofline,
            "gpu_launches": LAUNCHES_PER_STEP * K * len(runs),
            "gpu_launches_note": f"{LAUNCHES_PER_STEP} launches per step x {K} steps x {len(runs)} timed runs",
            "clocks": clk, "e2e": e2e, "cpu_baseline": cpu, "mask_free": mask_free,
            "workloads": extra,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def hn_set_mb(w, rows):
    """Approximate bytes of one buffer set (MB), for the config note."""
    e = 2 if w.dtype == "bf16" else 4
    full = w.S * w.B * w.H * e
    per_rows = rows * w.H * e
    return (w.T * full + 2 * full + per_rows * 8 + rows * w.H) / 1e6


def run_e2e(args, w, hn, world):
    """Through the public API with HOST buffers: every step copies its inputs
    from pinned host memory, runs the step and copies its results back.  The
    steps run as a three-stage pipeline on two device buffer sets (inputs in
    on one stream, the step on a second, results out on a third), so one
    step's copies overlap the neighbouring steps' compute and copies, as in a
    training loop that prefetches its next batch."""
    import torch

    from residual_sp_rs_gb300 import ops

    T, H, rows, row0 = w.T, w.H, hn.rows, hn.row0
    desc, dev, sets = hn.desc, hn.dev, hn.sets
    s0 = sets[0]
    rowb = H * (2 if w.dtype == "bf16" else 4)

    # a step's inputs travel as one block and its results as another: one
    # copy each way per step; only this rank's rows of each partial travel
    in_named = [(f"P{t}", p.view(-1, H)[row0:row0 + rows]) for t, p in enumerate(s0["partials"])]
    in_named += [(k, s0[k]) for k in ("residual", "dy", "dh", "gamma", "beta") if s0[k] is not None]
    out_named = [(k, s0[k]) for k in ("y", "d_res", "d_sum", "dgamma", "dbeta") if s0[k] is not None]
    host_in, hv = packed_block(in_named, "cpu", pin=True)
    for (_, v), h in zip(in_named, hv):
        h.copy_(v.cpu())
    host_out, _ = packed_block(out_named, "cpu", pin=True)
    dsets, dev_in, dev_out = [], [], []
    for k in range(2):
        fi, vi = packed_block(in_named, dev)
        fo, vo = packed_block(out_named, dev)
        d = dict(sets[k])
        # the call addresses partial t by global row (shard j's rows start at
        # row j*R), so it gets the address row0 rows before the resident rows
        d["partials"] = [v.data_ptr() - row0 * rowb for v in vi[:T]]
        d.update({name: v for (name, _), v in zip(in_named[T:], vi[T:])})
        d.update({name: v for (name, _), v in zip(out_named, vo)})
        dsets.append(d)
        dev_in.append(fi)
        dev_out.append(fo)
    bi = host_in.numel()
    bo = host_out.numel()
    st_in, st_cmp, st_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in dsets]
    ev_cmp = [torch.cuda.Event() for _ in dsets]
    ev_out = [torch.cuda.Event() for _ in dsets]

    def one_step(i):
        k = i % len(dsets)
        s = dsets[k]
        st_in.wait_event(ev_cmp[k])  # the set's inputs are free once its last step ran
        with torch.cuda.stream(st_in):
            dev_in[k].copy_(host_in, non_blocking=True)
            ev_in[k].record(st_in)
        st_cmp.wait_event(ev_in[k])
        st_cmp.wait_event(ev_out[k])  # the set's outputs are free once copied out
        with torch.cuda.stream(st_cmp):
            ops.sp_rs_dropout_residual_norm_fwd(desc, s["partials"], s["residual"], s["gamma"], s["beta"],
                                                s["h"], s["y"], s["mask"], s["rstd"], s["mean"])
            ops.sp2hp(s["y"], s["y_hp"], rows, H, T, w.dtype)
            ops.hp2sp(s["y_hp"], s["y_sp"], rows, H, T, w.dtype)
            ops.sp_rs_dropout_residual_norm_bwd(desc, s["dy"], s["dh"], s["h"], s["gamma"], s["mask"],
                                                s["rstd"], s["mean"], s["d_res"], s["d_sum"],
                                                s["dgamma"], s["dbeta"], s["ws"])
            ev_cmp[k].record(st_cmp)
        st_out.wait_event(ev_cmp[k])
        with torch.cuda.stream(st_out):
            host_out.copy_(dev_out[k], non_blocking=True)
            ev_out[k].record(st_out)

    for i in range(6):
        one_step(i)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(st_in)
    for i in range(args.e2e_steps):
        one_step(i)
    b.record(st_out)  # after the last step's results are on the host
    torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b), world, dev)
    return {"value": round(rows * args.e2e_steps * world / (ms / 1e3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "steps": args.e2e_steps,
            "ms_per_step": round(ms / args.e2e_steps, 5),
            "pipeline": "copy-in / step / copy-out on three streams over two device buffer sets; "
                        "each step's inputs and results each one packed pinned block (one copy each way)"}


# ---------------------------------------------------------------------------
# CPU oracle: the cpu_baseline leg and the reference arm
# ---------------------------------------------------------------------------

def _oracle_setup(w):
    import oracle
    from residual_sp_rs_gb300 import synthetic as syn

    oracle.build()
    inp = syn.fwd_inputs(w, "cpu")
    gr = syn.upstream_grads(w, "cpu")
    H, rows = w.H, w.S * w.B
    st = dict(parts=[syn.to_storage(p).reshape(rows, H) for p in inp["partials"]],
              res=syn.to_storage(inp["residual"]).reshape(rows, H),
              gamma=syn.to_storage(inp["gamma"]),
              beta=None if inp["beta"] is None else syn.to_storage(inp["beta"]),
              dy=syn.to_storage(gr["dy"]).reshape(rows, H),
              dh=syn.to_storage(gr["dh_out"]).reshape(rows, H))
    return oracle, st


def _oracle_step(oracle, w, st, row0, n):
    """The oracle's pass over token rows [row0, row0+n) (n a multiple of T):
    forward, sp2hp/hp2sp of the norm output, backward."""
    pr = oracle.problem(w.T, 0, w.S, w.B, w.H, w.dtype, w.norm, float(np.float32(w.p)),
                        float(np.float32(w.eps)), w.seed)
    grows = np.arange(row0, row0 + n)
    f = oracle.fwd_rows(pr, grows, [p[row0:row0 + n] for p in st["parts"]], st["res"][row0:row0 + n],
                        st["gamma"], st["beta"], w.dtype)
    hp = oracle.sp2hp(f["y"], w.T)
    oracle.hp2sp(hp)
    oracle.bwd_rows(pr, st["dy"][row0:row0 + n], st["dh"][row0:row0 + n], f["h"], st["gamma"],
                    f["mask"], w.dtype)


def _cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.processor() or platform.machine()


class _PinnedThread:
    """Pins the calling thread to one core (the last one it may use) for the
    oracle's timing, and restores its affinity afterwards."""

    def __enter__(self):
        self.saved = os.sched_getaffinity(0)
        self.core = max(self.saved)
        os.sched_setaffinity(0, {self.core})
        return self

    def __exit__(self, *exc):
        os.sched_setaffinity(0, self.saved)
        return False


def _host_note(core):
    return f"single thread pinned to core {core}; host: {os.cpu_count()} cores, {_cpu_model()}"


def cpu_baseline(w, seconds):
    with _PinnedThread() as pin:
        return _cpu_baseline(w, seconds, pin.core)


def _cpu_baseline(w, seconds, core):
    # the oracle's cost per token row does not depend on S: draw the inputs
    # for a short sequence of the same shape and cycle over its rows
    w = w.with_(S=min(w.S, w.T * max(1, 128 // w.B)))
    oracle, st = _oracle_setup(w)
    rows = w.S * w.B
    n = max(w.T, (64 // w.T) * w.T)
    done, t0 = 0, time.perf_counter()
    row0 = 0
    while time.perf_counter() - t0 < seconds:
        _oracle_step(oracle, w, st, row0, n)
        done += n
        row0 = (row0 + n) % (rows - n + 1)
    dt = time.perf_counter() - t0
    return {"value": round(done / dt, 2), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{done} token rows of the workload's shape (T={w.T}, H={w.H}, {w.dtype}, "
                      f"{w.norm}, p={w.p}; inputs drawn for S={w.S}, rows cycled) through the fp64 "
                      f"oracle (fwd, sp2hp, hp2sp, bwd), {dt:.1f} s, " + _host_note(core)}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from residual_sp_rs_gb300 import synthetic as syn

    w = syn.WORKLOADS[args.workload]
    with _PinnedThread() as pin:
        _run_reference(args, world, w, pin.core)


def _run_reference(args, world, w, core):
    oracle, st = _oracle_setup(w)
    rows = w.S * w.B
    # size each step's sample so the whole run ends within about two minutes
    t0 = time.perf_counter()
    _oracle_step(oracle, w, st, 0, w.T * 4)
    per_row = (time.perf_counter() - t0) / (w.T * 4)
    budget = 100.0 / max(1, args.steps + args.warmup)
    n = int(budget / per_row) // w.T * w.T
    n = max(w.T, min(n, rows))
    for i in range(args.warmup):
        _oracle_step(oracle, w, st, (i * n) % (rows - n + 1), n)
    t0 = time.perf_counter()
    for i in range(args.steps):
        _oracle_step(oracle, w, st, (i * n) % (rows - n + 1), n)
    dt = time.perf_counter() - t0
    value = n * args.steps / dt
    sample = (f"{n} of {rows} token rows per step through the fp64 oracle "
              f"(fwd, sp2hp, hp2sp, bwd), " + _host_note(core))
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{w.name}: SP region fwd+sp2hp+hp2sp+bwd, T={w.T} S={w.S} "
                                   f"B={w.B} H={w.H} {w.dtype} {w.norm} p={w.p}",
                       "tokens_per_step_sampled": n},
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": 1,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
