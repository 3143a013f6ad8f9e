"""Benchmark of the SP-region hot path on GB300.

One step = one pass of the whole hot path over one synthetic batch of the
pages' benchmark shape (T=2, S=2048, B=2, H=768, bf16, RMSNorm, p=0.1):
  forward of every sequence shard (reduce-scatter's reduce, dropout, residual,
  RMSNorm) -> sp2hp of the norm output -> hp2sp back -> backward of every
  shard (norm, residual and dropout backward, dgamma).
Steps run from CUDA graphs of about 64 steps (whole rotations over the
buffer sets, each step of a rotation on its own set); there are enough sets
that every kernel's own bytes over a rotation exceed twice the L2 size, so
HBM (not L2) serves the inputs.  The JSON line also carries per-kernel
launch times (back to back and single), the end-to-end number through host
buffers, the mask-free step, the oracle's CPU rate and the clocks seen.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Rank 0 prints one JSON line.  Under torchrun every rank runs the same
workload on its own GPU (weak scaling; no data-path collective).
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = "pages_rms_bf16"
METRIC = "SP-region fwd+bwd tokens/s and achieved HBM GB/s (% of GB300 peak), 1 GPU"
LAUNCHES_PER_STEP = 5  # fwd, sp2hp, hp2sp, bwd, dgamma column sum
NOMINAL_HBM_GBS = 8000.0  # GB300's nominal HBM3e bandwidth (the measured copy peak is the roofline)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--roofline-iters", type=int, default=400)
    ap.add_argument("--e2e-steps", type=int, default=300)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
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
# multi-rank aggregation (one process per GPU, the same workload on each)
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
    batch in at most `ms` milliseconds."""
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
        self.path = os.path.join(ROOT, "gpurun_out", f"clocks_rank{device_index}.csv")
        if enabled:
            try:
                os.makedirs(os.path.dirname(self.path), exist_ok=True)
                self.f = open(self.path, "w")
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
        for line in open(self.path):
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
    rows = w.S * w.B
    tdt = syn.torch_dtype(w.dtype)
    desc = ops.make_desc(T, 0, w.S, w.B, H, w.dtype, w.norm, w.p, w.eps, w.seed, nshards=T)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size

    def make_set(k):
        inp = syn.fwd_inputs(w, dev, seed=w.input_seed + 17 * k)
        gr = syn.upstream_grads(w, dev, seed=w.input_seed + 17 * k)
        s = dict(partials=inp["partials"], residual=inp["residual"].view(rows, H),
                 gamma=inp["gamma"], beta=inp["beta"], dy=gr["dy"].view(rows, H),
                 dh=gr["dh_out"].view(rows, H))
        s["h"] = torch.empty((rows, H), device=dev, dtype=tdt)
        s["y"] = torch.empty((rows, H), device=dev, dtype=tdt)
        s["mask"] = torch.empty((rows, H), device=dev, dtype=torch.uint8) if w.p > 0 else None
        s["rstd"] = torch.empty(rows, device=dev)
        s["mean"] = torch.empty(rows, device=dev) if w.norm == "ln" else None
        s["y_hp"] = torch.empty((T, rows, H // T), device=dev, dtype=tdt)
        s["y_sp"] = torch.empty((rows, H), device=dev, dtype=tdt)
        s["d_res"] = torch.empty((rows, H), device=dev, dtype=tdt)
        s["d_sum"] = torch.empty((rows, H), device=dev, dtype=tdt)
        s["dgamma"] = torch.empty(H, device=dev)
        s["dbeta"] = torch.empty(H, device=dev) if w.norm == "ln" else None
        s["ws"] = ops.workspace_for(desc, dev)
        return s

    def set_bytes(s):
        return sum(v.numel() * v.element_size() for k, v in s.items()
                   if isinstance(v, torch.Tensor)) + sum(p.numel() * p.element_size()
                                                         for p in s["partials"])

    first = make_set(0)
    per_set = set_bytes(first)
    n_sets = rotation_sets(l2, per_set, fwd_bytes(w, rows), bwd_bytes(w, rows), layout_bytes(w, rows))
    sets = [first] + [make_set(k) for k in range(1, n_sets)]

    def fwd(s, stream=None, mask_free=False):
        ops.sp_rs_dropout_residual_norm_fwd(desc, s["partials"], s["residual"], s["gamma"], s["beta"],
                                            s["h"], s["y"], None if mask_free else s["mask"], s["rstd"],
                                            s["mean"], stream)

    def bwd(s, stream=None, mask_free=False):
        ops.sp_rs_dropout_residual_norm_bwd(desc, s["dy"], s["dh"], s["h"], s["gamma"],
                                            None if mask_free else s["mask"],
                                            s["rstd"], s["mean"], s["d_res"], s["d_sum"], s["dgamma"],
                                            s["dbeta"], s["ws"], stream=stream)

    side = torch.cuda.Stream()

    def step(s, join=True, mask_free=False):
        # the layout transforms of y and the backward both depend only on the
        # forward: they run as two concurrent branches of the step
        fwd(s, mask_free=mask_free)
        cur = torch.cuda.current_stream()
        side.wait_stream(cur)
        with torch.cuda.stream(side):
            ops.sp2hp(s["y"], s["y_hp"], rows, H, T, w.dtype)
            ops.hp2sp(s["y_hp"], s["y_sp"], rows, H, T, w.dtype)
        bwd(s, mask_free=mask_free)
        if join:
            cur.wait_stream(side)

    # a graph replay boundary costs a few microseconds (the next replay starts
    # only when the previous one has finished, with no programmatic dependent
    # launch across them): one graph holds enough rotations for about 64 steps
    n_rot = max(1, -(-64 // n_sets))
    steps_per_graph = n_rot * n_sets

    def rotations(mask_free=False):
        # n_rot times n_sets consecutive steps, step k on buffer set k % n_sets;
        # the layout branch of a step joins the main stream at the end of its
        # rotation (no step in between touches its buffers)
        for _ in range(n_rot):
            for s in sets:
                step(s, join=False, mask_free=mask_free)
            torch.cuda.current_stream().wait_stream(side)

    for s in sets:
        step(s)
    torch.cuda.synchronize()
    # one CUDA graph for a whole rotation (programmatic dependent launch then
    # also links one step's last kernel to the next step's first), and one
    # single-step graph per set for a remainder of steps
    cap_stream = torch.cuda.Stream()
    g_rot = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_rot, stream=cap_stream, capture_error_mode="relaxed"):
        rotations()
    graphs = []
    for s in sets:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap_stream, capture_error_mode="relaxed"):
            step(s)
        graphs.append(g)
    torch.cuda.synchronize()

    def run_steps(k):
        for _ in range(k // steps_per_graph):
            g_rot.replay()
        for i in range(k % steps_per_graph):
            graphs[i % n_sets].replay()

    run_steps(args.warmup)
    torch.cuda.synchronize()

    # ---- timed region ----------------------------------------------------------
    clocks = ClockSampler(local, enabled=not args.no_clocks)
    time.sleep(0.2)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    run_steps(args.steps)
    ev1.record()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    ms = max_over_ranks(ev0.elapsed_time(ev1), world, dev)
    ms_per_step = ms / args.steps
    value = weak_scaling_tokens_per_s(rows, args.steps, world, ms)
    step_bytes = fwd_bytes(w, rows) + bwd_bytes(w, rows) + 2 * layout_bytes(w, rows)
    step_gbs = step_bytes / (ms_per_step / 1e3) / 1e9

    # ---- the mask-free mode (not the headline): the forward stores no mask and
    # the backward draws the keep bits again -- 2 bytes per element less
    # traffic, Philox twice
    mask_free = None
    if w.p > 0:
        g_mf = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_mf, stream=cap_stream, capture_error_mode="relaxed"):
            rotations(mask_free=True)
        for _ in range(3):
            g_mf.replay()
        torch.cuda.synchronize()
        reps_mf = max(5, min(args.steps, 20000) // steps_per_graph)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps_mf):
            g_mf.replay()
        e1.record()
        torch.cuda.synchronize()
        ms_mf = max_over_ranks(e0.elapsed_time(e1), world, dev) / (reps_mf * steps_per_graph)
        mask_free = {"ms_per_step": round(ms_mf, 6),
                     "value": round(weak_scaling_tokens_per_s(rows, 1, world, ms_mf), 1),
                     "unit": "tokens/s", "steps": reps_mf * steps_per_graph,
                     "note": "same step with the mask pointers NULL: the forward keeps no mask, the "
                             "backward regenerates the keep bits from the seed"}

    # ---- per-launch durations of the main kernels: each kernel alone, launched
    # back to back from one CUDA graph over the rotating sets, CUDA events
    # around the replays on the launching stream
    def time_launches(fn, reps):
        per_graph = steps_per_graph
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap_stream, capture_error_mode="relaxed"):
            for i in range(per_graph):
                fn(sets[i % n_sets])
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
        evs[0].record()
        for i in range(reps):
            g.replay()
            evs[i + 1].record()
        torch.cuda.synchronize()
        # median over replays of the mean launch duration within a replay
        return float(np.median([evs[i].elapsed_time(evs[i + 1]) for i in range(reps)])) / per_graph

    def time_single(fn, reps=50, warm=10):
        """One launch at a time: events around it, a synchronize after each,
        so launch latency is included (median)."""
        out = []
        for i in range(warm + reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn(sets[i % n_sets])
            b.record()
            torch.cuda.synchronize()
            if i >= warm:
                out.append(a.elapsed_time(b))
        return float(np.median(out))

    reps = max(50, args.roofline_iters // steps_per_graph)
    t_fwd = time_launches(fwd, reps)
    t_bwd = time_launches(bwd, reps)
    t_sp2hp = time_launches(lambda s: ops.sp2hp(s["y"], s["y_hp"], rows, H, T, w.dtype), reps)
    single = {"fwd": time_single(fwd), "bwd": time_single(bwd),
              "sp2hp": time_single(lambda s: ops.sp2hp(s["y"], s["y_hp"], rows, H, T, w.dtype))}
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except OSError:
        pass
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"
    kern = {"fwd": (t_fwd, fwd_bytes(w, rows), "sp_fwd_kernel"),
            "bwd": (t_bwd, bwd_bytes(w, rows), "sp_bwd_kernel+sp_colsum_kernel"),
            "sp2hp": (t_sp2hp, layout_bytes(w, rows), "sp_layout_kernel")}
    dom = max(("fwd", "bwd"), key=lambda k: kern[k][0])
    d_ms, d_bytes, d_name = kern[dom]
    achieved = d_bytes / (d_ms / 1e3) / 1e9
    traffic = None
    try:
        tr = json.load(open(os.path.join(ROOT, "profiles", f"{dom}_{args.workload}_traffic.json")))
        from residual_sp_rs_gb300.build import _deps
        import hashlib
        h = hashlib.sha256()
        for p in sorted(_deps()):
            h.update(open(p, "rb").read())
        if tr.get("source_sha256") == h.hexdigest():
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
                "per_kernel": {k: {"launch_ms": round(v[0], 5), "single_launch_ms": round(single[k], 5),
                                   "algorithmic_bytes": v[1],
                                   "gbs": round(v[1] / (v[0] / 1e3) / 1e9, 1),
                                   "frac_of_measured": round(v[1] / (v[0] / 1e3) / 1e9 / hbm_peak, 4),
                                   "frac_of_nominal_8000": round(v[1] / (v[0] / 1e3) / 1e9 / NOMINAL_HBM_GBS,
                                                                 4)}
                               for k, v in kern.items()}}

    # ---- end to end: pinned host inputs in, results out, every step -------------
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, w, desc, dev, sets, rows, world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(w, args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16"
            if w.dtype == "bf16" else "f32", "data": "synthetic (seeded torch.Generator)",
            "config": {"workload": f"{w.name}: SP region fwd+sp2hp+hp2sp+bwd, T={T} S={w.S} B={w.B} "
                                   f"H={H} {w.dtype} {w.norm} p={w.p}",
                       "T": T, "S": w.S, "B": w.B, "H": H, "norm": w.norm, "p": w.p,
                       "tokens_per_step": rows, "parallelism": f"replica x{world}",
                       "l2": f"inputs rotate over {n_sets} buffer sets, {n_sets * per_set / 1e6:.0f} MB; "
                             f"each kernel's own bytes over a rotation > 2x L2 ({l2 / 1e6:.0f} MB)",
                       "launch": f"one CUDA graph replay per {steps_per_graph} steps ({n_rot} rotations "
                                 f"over the {n_sets} buffer sets; layout branch concurrent with the "
                                 "backward, joined once per rotation), programmatic dependent launch "
                                 "between the kernels of a replay; single-step graphs for a remainder"},
            "hbm_gbs_step": round(step_gbs, 1),
            "hbm_frac_step": round(step_gbs / hbm_peak, 4),
            "hbm_frac_step_of_nominal_8000": round(step_gbs / NOMINAL_HBM_GBS, 4),
            "roofline": roofline,
            "gpu_launches": LAUNCHES_PER_STEP * args.steps,
            "clocks": clk, "e2e": e2e, "cpu_baseline": cpu, "mask_free": mask_free,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_e2e(args, w, desc, dev, sets, rows, world):
    """Through the public API with HOST buffers: every step copies its inputs
    from pinned host memory, runs the step and copies its results back.  The
    steps run as a three-stage pipeline on two device buffer sets (inputs in
    on one stream, the step on a second, results out on a third), so one
    step's copies overlap the neighbouring steps' compute and copies, as in a
    training loop that prefetches its next batch."""
    import torch

    from residual_sp_rs_gb300 import ops

    T, H = w.T, w.H
    s0 = sets[0]

    # a step's inputs travel as one block and its results as another: one
    # copy each way per step
    in_named = [(f"P{t}", p.view(rows, H)) for t, p in enumerate(s0["partials"])]
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
        d["partials"] = vi[:T]
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
    ms = a.elapsed_time(b)
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
            "sample": f"{done} token rows ({done / rows:.2f} of one step's {rows}) of the same "
                      f"workload through the fp64 oracle (fwd, sp2hp, hp2sp, bwd), {dt:.1f} s, "
                      + _host_note(core)}


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
