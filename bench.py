"""Benchmark of the DiLoCo outer synchronisation step on GB300.

Workload (default, ``decoder_10b``): the 10B decoder-shaped fp32 tensor set
(381 tensors, 42 layers, d=4096, FFN 14336, 32 q / 8 kv heads, vocab 128256)
cut by the LPT planner into P=24 fragments; the median fragment (18 tensors,
415,260,672 elements) is resident in HBM with its K=14 learner replicas. One
step = one outer synchronisation of that fragment through dl_outer_sync:
stats -> quantise -> merge + Nesterov, theta_g and momentum carried from step
to step. A second timed pass makes the same steps as separate C-ABI calls with
CUDA events around each call: the per-call GB/s and the roofline of the
dominant call come from it. ``quorum_10b`` is the same fragment with K=16 and
a random present subset and token weights per step; ``ragged_heavy`` is the
2000-tensor heavy-tail batch (K=8) synced as one fragment.

``decoder_1b`` keeps the whole 1.1B model (K=4, all 24 fragments) resident and
syncs every fragment per step, consecutive fragments overlapped on two
streams; ``learner_1b`` / ``learner_10b`` time the learner-side quantiser.
Inputs are synthetic (seeded generator); every call streams far more than the
129 MB L2, so no L2 flush is needed between calls.

Metric: outer-step params/s (whole job) and achieved HBM GB/s of each call,
against the measured copy bandwidth in MEASURED_PEAKS.json.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]

N > 1 runs under torchrun as N independent replicas of the workload (one per
GPU; the path has no data exchange), timed with a barrier and the max over
ranks. The reference arm (--impl reference) times the CPU oracle on the host
cores on a bounded sample of the same workload.
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

import synthetic  # noqa: E402

METRIC = "outer-step params/s & achieved HBM GB/s (quantise+merge+Nesterov, K learners)"
UNIT = "params/s"
LEARNER_METRIC = "learner-side quantiser params/s (stats + quantise, K=1, whole model)"


def algo_bytes(K):
    """Algorithmic HBM bytes per fragment element of each call (minimum traffic:
    Delta never stored, codes written once and read once)."""
    return {"stats": 4 * (K + 1), "quantize": 4 * (K + 1) + K, "merge": K + 16}


def max_over_ranks(value, world, device):
    """The largest value over all ranks (timings: the job is as slow as its
    slowest rank); the value itself on one rank."""
    if world <= 1:
        return value
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def env_rank():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_uuid):
        self.uuid = device_uuid
        self.proc = None
        self.lines = []

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# workload data


def fragment_tensors(wl, frag_of):
    return [[t for t in range(wl.n_tensors) if frag_of[t] == f] for f in range(wl.n_frags)]


def generate_host(wl, frags, pin):
    """theta_g and K replicas of every fragment as (pinned) host tensors."""
    import torch

    out = []
    for tensors in frags:
        n = sum(wl.numels[t] for t in tensors)
        g = torch.empty(n, dtype=torch.float32, pin_memory=pin)
        reps = [torch.empty(n, dtype=torch.float32, pin_memory=pin) for _ in range(wl.K)]
        gn, rn = g.numpy(), [r.numpy() for r in reps]
        o = 0
        for t in tensors:
            m = wl.numels[t]
            wl.theta_global(t, out=gn[o:o + m])
            for k in range(wl.K):
                wl.replica(k, t, gn[o:o + m], out=rn[k][o:o + m])
            o += m
        out.append((g, reps))
    return out


class DeviceRun:
    """Device-resident state of every fragment plus shared scratch buffers."""

    def __init__(self, wl, frags, host, dev):
        import torch

        import pseudo_grad_sync_gb300 as dl

        self.dl, self.wl, self.frags = dl, wl, frags
        K = wl.K
        self.F = [dl.Fragment([wl.numels[t] for t in ts], dev) for ts in frags]
        self.g = [h[0].to(dev, non_blocking=True) for h in host]
        self.m = [torch.zeros_like(x) for x in self.g]
        self.reps = [[r.to(dev, non_blocking=True) for r in h[1]] for h in host]
        max_n = max(f.n for f in self.F)
        max_t = max(f.T for f in self.F)
        self.codes = [torch.empty(max_n, dtype=torch.uint8, device=dev) for _ in range(K)]
        self.codebook = torch.empty((K, max_t, 256), dtype=torch.float32, device=dev)
        self.stats = dl.new_stats(K, max_t, dev)
        self.ws_s = dl.new_workspace(max(dl.stats_workspace_bytes(f, K) for f in self.F), dev)
        self.ws_q = dl.new_workspace(max(dl.quantize_workspace_bytes(f, K) for f in self.F), dev)
        self.msync = dl.ModelSync(self.F, K, dev)
        torch.cuda.synchronize()

    def sync_step(self, stream=None):
        """The whole outer step in one dl_outer_sync call (fragments pipelined)."""
        self.dl.plan_fragments(self.wl.numels, self.wl.n_frags)
        self.msync.step(self.g, self.m, self.reps, stream=stream)

    def step(self, reps=None, events=None, stream=None):
        dl, K = self.dl, self.wl.K
        dl.plan_fragments(self.wl.numels, self.wl.n_frags)
        for f, F in enumerate(self.F):
            # stats / codebook buffers are used as flat [K*T] / [K*T*256] arrays
            r = self.reps[f] if reps is None else reps[f]
            if events is not None:
                events[f][0].record(stream)
            dl.pseudograd_stats(self.g[f], r, F, 6.0, self.stats, self.ws_s, stream)
            if events is not None:
                events[f][1].record(stream)
            dl.quantize(self.g[f], r, F, self.stats, self.codes, self.codebook, None, self.ws_q,
                        stream)
            if events is not None:
                events[f][2].record(stream)
            dl.merge_outer_step(self.g[f], self.m[f], F, self.codes, self.codebook, K=K,
                                lr=0.7, mu=0.9, stream=stream)
            if events is not None:
                events[f][3].record(stream)


LAUNCHES_PER_FRAGMENT = {"stats": 1, "quantize": 3, "merge": 1}


def traffic_record(name):
    """Per-element DRAM traffic of a kernel from a committed ncu summary, valid
    only while the kernel's source is unchanged (hash recorded with it)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        rec = json.load(fh).get(name)
    if not rec:
        return None
    h = hashlib.sha256()
    for src in rec["sources"]:
        with open(os.path.join(ROOT, src), "rb") as fh:
            h.update(fh.read())
    return rec if h.hexdigest() == rec["sha256"] else None


def learner_device_data(wl, dev, gen_seed=0):
    """theta_g and the learner's replica of the whole model, filled on the
    device with the workload's distributions (theta_g ~ N(0, theta_std),
    Delta ~ N(0, sigma_t) per tensor)."""
    import torch

    gen = torch.Generator(device=dev)
    gen.manual_seed(gen_seed)
    n = wl.n_elems
    g = torch.empty(n, dtype=torch.float32, device=dev).normal_(0.0, wl.theta_std, generator=gen)
    r = torch.empty_like(g)
    o = 0
    for t, m in enumerate(wl.numels):
        d = torch.empty(m, dtype=torch.float32, device=dev).normal_(0.0, wl.tensor_scale(t),
                                                                   generator=gen)
        torch.sub(g[o:o + m], d, out=r[o:o + m])
        o += m
    return g, r


def run_learner(args, rank, world, local):
    """Learner-side quantiser: one learner's whole model, every tensor in one
    ragged batch, dl_pseudograd_stats + dl_quantize with K=1 per step (codes
    and codebooks are what the learner would send)."""
    import torch

    import pseudo_grad_sync_gb300 as dl

    dev = f"cuda:{local}"
    torch.cuda.set_device(local)
    wl = synthetic.WORKLOADS[args.workload]()
    F = dl.Fragment(wl.numels, dev)
    g, r = learner_device_data(wl, dev, gen_seed=rank)
    stats = dl.new_stats(1, F.T, dev)
    codes = [torch.empty(F.n, dtype=torch.uint8, device=dev)]
    cb = torch.empty((1, F.T, 256), dtype=torch.float32, device=dev)
    ws_s = dl.new_workspace(dl.stats_workspace_bytes(F, 1), dev)
    ws_q = dl.new_workspace(dl.quantize_workspace_bytes(F, 1), dev)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        dl.pseudograd_stats(g, [r], F, 6.0, stats, ws_s, stream)
        if ev is not None:
            ev[1].record(stream)
        dl.quantize(g, [r], F, stats, codes, cb, None, ws_q, stream)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:
        uuid = None
    clocks = ClockSampler(uuid)
    clocks.start()
    time.sleep(0.3)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for s in range(args.steps):
        step(ev[s])
    end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = start.elapsed_time(end)
    if world > 1:
        ms = max_over_ranks(ms, world, dev)
    ms_per_step = ms / args.steps
    peak, peak_kind = load_peaks()
    ab = {"stats": 8, "quantize": 9}
    calls = {}
    for i, name in enumerate(("stats", "quantize")):
        tot = sum(e[i].elapsed_time(e[i + 1]) for e in ev)
        avg_s = tot / args.steps / 1e3
        gbs = ab[name] * wl.n_elems / avg_s / 1e9
        calls[name] = {"ms_per_step": tot / args.steps, "algo_bytes_per_elem": ab[name],
                       "achieved_gbs": gbs, "frac": gbs / peak}
    dominant = max(calls, key=lambda c: calls[c]["ms_per_step"])
    full_gbs = 17 * wl.n_elems / (ms_per_step / 1e3) / 1e9
    out = {
        "metric": LEARNER_METRIC,
        "value": world * wl.n_elems / (ms_per_step / 1e3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (device-filled)",
        "config": {"workload": wl.name + ": " + wl.description, "K": 1, "params": wl.n_elems,
                   "l2": "no flush: every call streams >= 8.8 GB, inputs larger than L2"},
        "full_step_gbs": full_gbs, "full_step_frac": full_gbs / peak, "calls": calls,
        "roofline": {"bound": "hbm", "achieved": round(calls[dominant]["achieved_gbs"], 1),
                     "peak": peak, "unit": "GB/s", "frac": round(calls[dominant]["frac"], 4),
                     "traffic": None, "kernel": {"stats": "k_stats",
                                                 "quantize": "k_quantize"}[dominant],
                     "note": f"peak = {peak_kind} copy bandwidth"},
        "clocks": clk, "gpu_launches": args.steps * (1 + LAUNCHES_PER_FRAGMENT["quantize"]), "e2e": None,
    }
    if rank == 0:
        print(json.dumps(out), flush=True)


def ring_algo_bytes(S):
    """Algorithmic bytes per element of one ring step over S learners: hop 0
    reads theta_g and a replica and writes P (12), accumulating P's
    statistics as it goes; each later hop quantises P (4 + 1) and then reads
    the codes, theta_g and a replica and writes P (13), the last one instead
    reading momentum and writing theta and momentum (21)."""
    if S == 1:
        return 24
    return 12 + 5 * (S - 1) + 13 * (S - 2) + 21


def ring_launches(S):
    """Kernels of one ring step per fragment: hop 0, then per later hop the
    statistics finalisation, the quantiser's kernels and the hop."""
    if S == 1:
        return 1
    return 1 + (2 + LAUNCHES_PER_FRAGMENT["quantize"]) * (S - 1)


def run_ring(args, rank, world, local):
    """Ring accumulation with re-quantisation at every hop (dl_ring_outer_step)
    over every fragment of the workload, one call per fragment."""
    import torch

    import pseudo_grad_sync_gb300 as dl

    dev = f"cuda:{local}"
    torch.cuda.set_device(local)
    wl = synthetic.WORKLOADS[args.workload]()
    frag_of, load = dl.plan_fragments(wl.numels, wl.n_frags)
    frags = fragment_tensors(wl, frag_of)
    host = generate_host(wl, frags, pin=False)
    run = DeviceRun(wl, frags, host, dev)
    del host
    ws = dl.new_workspace(max(dl.ring_workspace_bytes(F) for F in run.F), dev)
    stream = torch.cuda.current_stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in run.F]

    def step(timed=False):
        for f, F in enumerate(run.F):
            if timed:
                ev[f][0].record(stream)
            dl.ring_outer_step(run.g[f], run.m[f], F, run.reps[f], workspace=ws, stream=stream)
            if timed:
                ev[f][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(None)
    clocks.start()
    time.sleep(0.3)
    tot_call = 0.0
    for _ in range(args.steps):
        step(timed=True)
        torch.cuda.synchronize()
        tot_call += sum(e[0].elapsed_time(e[1]) for e in ev)
    clk = clocks.stop()
    ms_per_step = tot_call / args.steps  # the calls run back to back within a step
    peak, peak_kind = load_peaks()
    ab = ring_algo_bytes(wl.K)
    gbs = ab * wl.n_elems / (tot_call / args.steps / 1e3) / 1e9
    out = {
        "metric": "ring outer-step params/s (re-quantised at every hop, K learners)",
        "value": world * wl.n_elems / (ms_per_step / 1e3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": wl.name + ": " + wl.description, "K": wl.K,
                   "fragments": wl.n_frags, "params": wl.n_elems, "mode": "ring"},
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(gbs / peak, 4), "traffic": None,
                     "note": f"{ab} algorithmic B/elem per ring step; calls timed with CUDA "
                             f"events; peak = {peak_kind} copy bandwidth"},
        "clocks": clk, "gpu_launches": args.steps * len(frags) * ring_launches(wl.K),
        "e2e": None,
    }
    if rank == 0:
        print(json.dumps(out), flush=True)


def run_rda(args, rank, world, local):
    """The outer step with the Radial-Directional Averaging merge: per fragment
    dl_pseudograd_stats, dl_quantize (with bucket counts) and
    dl_rda_merge_outer_step. The headline is one dl_outer_sync call with
    DL_SYNC_RDA (fragments pipelined); the same sequence as separate calls is
    timed after it and reported beside."""
    import torch

    import pseudo_grad_sync_gb300 as dl

    dev = f"cuda:{local}"
    torch.cuda.set_device(local)
    wl = synthetic.WORKLOADS[args.workload]()
    K = wl.K
    frag_of, load = dl.plan_fragments(wl.numels, wl.n_frags)
    frags = fragment_tensors(wl, frag_of)
    host = generate_host(wl, frags, pin=False)
    run = DeviceRun(wl, frags, host, dev)
    del host
    max_t = max(F.T for F in run.F)
    counts = torch.empty((K, max_t, 256), dtype=torch.int32, device=dev)
    ws_r = dl.new_workspace(max(dl.rda_workspace_bytes(F, K) for F in run.F), dev)
    stream = torch.cuda.current_stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in run.F]

    msync = dl.ModelSync(run.F, K, dev, mode=dl.DL_SYNC_RDA)
    ev_sync = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def step(timed=False):
        for f, F in enumerate(run.F):
            if timed:
                ev[f][0].record(stream)
            dl.pseudograd_stats(run.g[f], run.reps[f], F, 6.0, run.stats, run.ws_s, stream)
            dl.quantize(run.g[f], run.reps[f], F, run.stats, run.codes, run.codebook, counts,
                        run.ws_q, stream)
            dl.rda_merge_outer_step(run.g[f], run.m[f], F, run.codes, run.codebook, counts,
                                    workspace=ws_r, stream=stream, K=K)
            if timed:
                ev[f][1].record(stream)

    def sync_step(timed=False):
        if timed:
            ev_sync[0].record(stream)
        msync.step(run.g, run.m, run.reps, stream=stream)
        if timed:
            ev_sync[1].record(stream)

    for _ in range(args.warmup):
        step()
        sync_step()
    torch.cuda.synchronize()
    clocks = ClockSampler(None)
    clocks.start()
    time.sleep(0.3)
    tot = tot_calls = 0.0
    for _ in range(args.steps):
        sync_step(timed=True)
        torch.cuda.synchronize()
        tot += ev_sync[0].elapsed_time(ev_sync[1])
        step(timed=True)
        torch.cuda.synchronize()
        tot_calls += sum(e[0].elapsed_time(e[1]) for e in ev)
    clk = clocks.stop()
    ms_per_step = tot / args.steps  # the whole step through dl_outer_sync (DL_SYNC_RDA)
    peak, peak_kind = load_peaks()
    ab = 11 * K + 24  # stats 4(K+1), quantise 4(K+1)+K, ||u|| pass K, merge K+16
    gbs = ab * wl.n_elems / (ms_per_step / 1e3) / 1e9
    out = {
        "metric": "RDA outer-step params/s (stats + quantise + RDA merge + Nesterov)",
        "value": world * wl.n_elems / (ms_per_step / 1e3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": wl.name + ": " + wl.description, "K": K,
                   "fragments": wl.n_frags, "params": wl.n_elems, "mode": "rda"},
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(gbs / peak, 4), "traffic": None,
                     "note": f"{ab} algorithmic B/elem per step; peak = {peak_kind} copy "
                             "bandwidth"},
        "per_call_ms_per_step": tot_calls / args.steps,
        "clocks": clk, "gpu_launches": args.steps * len(frags) * (5 + LAUNCHES_PER_FRAGMENT["quantize"]),
        "e2e": None,
        "gpu_launches_note": "kernels in the headline dl_outer_sync (DL_SYNC_RDA) region; the "
                             "per-call sequence, timed after it, launches as many again",
    }
    if rank == 0:
        print(json.dumps(out), flush=True)


# ---------------------------------------------------------------------------
# one fragment resident: the 10B decoder's median fragment (K=14, or K=16 with
# a random quorum) and the ragged heavy-tail batch, one dl_outer_sync call per
# step


FRAGMENT_WORKLOADS = ("decoder_10b", "quorum_10b", "ragged_heavy")


def bench_fragment(wl, plan, which="median"):
    """Tensors of the fragment a step syncs: for a model cut into P fragments
    the median one by load (ties broken by fragment index), or the largest
    one (the lowest index among equal loads); for a one-batch workload every
    tensor. Returns (tensors, fragment index)."""
    if wl.n_frags == 1:
        return list(range(wl.n_tensors)), 0
    frag_of, load = plan(wl.numels, wl.n_frags)
    if which == "largest":
        f = int(np.argmax(load))
    else:
        f = int(np.argsort(load, kind="stable")[len(load) // 2])
    return [t for t in range(wl.n_tensors) if frag_of[t] == f], f


def quorum_schedule(wl, step):
    """Present mask and weights of bench step `step`: with a random quorum the
    steps walk through every (fragment, outer step) draw of the workload in
    turn (fragment = step mod P, outer step = step div P mod steps), so the
    mix of quorum sizes is the workload's; otherwise all present, weight 1."""
    f, s = step % wl.n_frags, (step // wl.n_frags) % wl.steps
    return wl.present(f, s), wl.weights(f, s)


def fragment_device_fill(wl, ts, dev, seed=0):
    """theta_g and the K replicas (rows padded to 64 elements) filled on the
    device from a seeded generator with the workload's distributions
    (theta_g ~ N(0, theta_std), Delta = scale * N(0, 1) or scale *
    Student-t(3))."""
    import torch

    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    n = sum(wl.numels[t] for t in ts)
    g = torch.empty(n, dtype=torch.float32, device=dev).normal_(0.0, wl.theta_std, generator=gen)
    # rows padded to 64 elements: every replica starts 256-byte aligned
    reps = torch.empty((wl.K, -(-n // 64) * 64), dtype=torch.float32, device=dev)[:, :n]
    chunk = 1 << 26
    for k in range(wl.K):
        o = 0
        for t in ts:
            m = wl.numels[t]
            for a in range(0, m, chunk):
                b = min(m, a + chunk)
                x = torch.randn(b - a, device=dev, generator=gen)
                if wl.delta_dist == 1:  # Student-t(3) = Z / sqrt(chi2_3 / 3)
                    c = torch.randn(3, b - a, device=dev, generator=gen).square_().sum(0)
                    x.div_(c.div_(3.0).sqrt_())
                torch.sub(g[o + a:o + b], x.mul_(wl.tensor_scale(t)), out=reps[k, o + a:o + b])
            o += m
    return g, reps


def oracle_fragment_pass(g, reps, off, present, weights):
    """One outer step of the oracle over one fragment with the present
    learners (what the GPU step computes); returns the seconds it took."""
    import oracle

    idx = [k for k in range(len(reps)) if present[k]]
    t0 = time.perf_counter()
    o = oracle.outer_step(g, np.zeros_like(g), [reps[k] for k in idx], offsets=off,
                          weights=np.asarray(weights, np.float32)[idx])
    dt = time.perf_counter() - t0
    assert o["status"] == 0
    return dt


def fragment_cpu_sample(wl, ts, limit, generate=True):
    """Host arrays (theta_g, replicas, offsets, elements, tensors) of the
    oracle's bounded sample: the fragment's tensors in order up to `limit`
    elements (at least one tensor; a first tensor longer than `limit` is cut
    to its first `limit` values), generated on the host (generate=False: the
    selection only)."""
    sel, sizes, tot = [], [], 0
    for t in ts:
        if sel and tot + wl.numels[t] > limit:
            continue
        sel.append(t)
        sizes.append(min(wl.numels[t], limit))
        tot += sizes[-1]
    if not generate:
        return None, None, None, tot, sel
    off = synthetic.offsets_of(sizes)
    g = np.empty(tot, dtype=np.float32)
    reps = [np.empty(tot, dtype=np.float32) for _ in range(wl.K)]
    for i, t in enumerate(sel):
        a, b = int(off[i]), int(off[i + 1])
        wl.theta_global(t, out=g[a:b], n=b - a)
        for k in range(wl.K):
            wl.replica(k, t, g[a:b], out=reps[k][a:b])
    return g, reps, off, tot, sel


def fragment_cpu_baseline(wl, ts, budget_s):
    """The oracle on the host cores over (a bounded sample of) the bench
    fragment, with step 0's quorum; the single-thread figure on its first
    tensor beside it."""
    import oracle

    oracle.lib()
    present, weights = quorum_schedule(wl, 0)
    g, reps, off, tot, sel = fragment_cpu_sample(wl, ts, 1 << 26)
    total, passes = 0.0, 0
    while passes == 0 or total < budget_s:
        total += oracle_fragment_pass(g, reps, off, present, weights)
        passes += 1
    cores = oracle.threads()
    # one thread on one tensor of the sample: the smallest with >= 2^20 elements
    size = [int(off[i + 1] - off[i]) for i in range(len(sel))]
    big = [i for i in range(len(sel)) if size[i] >= 1 << 20]
    i1 = min(big, key=lambda i: size[i]) if big else 0
    a1, n1 = int(off[i1]), size[i1]
    oracle.set_threads(1)
    try:
        t1 = oracle_fragment_pass(g[a1:a1 + n1], [r[a1:a1 + n1] for r in reps],
                                  np.array([0, n1], np.int64), present, weights)
    finally:
        oracle.set_threads(cores)
    np_ = int(np.count_nonzero(present))
    if tot < sum(wl.numels[t] for t in sel):
        whole = f"the first {tot} values of its {len(ts)}-tensor fragment"
    elif len(sel) == len(ts):
        whole = "the whole fragment"
    else:
        whole = f"{len(sel)} of its {len(ts)} tensors"
    return {"value": tot * passes / total, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{whole} ({tot} elements x {np_} present learners), full outer step "
                      f"(stats+quantise+merge+Nesterov), {passes} pass(es) in {total:.1f} s",
            "single_thread": {"value": n1 / t1, "unit": UNIT, "cores": 1,
                              "sample": f"one tensor of it ({n1} elements x {np_} learners), "
                                        f"one pass in {t1:.1f} s"}}


class RegisteredHost:
    """A page-aligned host array of `nfloats` fp32 values registered with
    cudaHostRegister: pinned memory the copy engines read directly. `tensor`
    views it; release() unregisters it."""

    def __init__(self, nfloats):
        import torch

        nbytes = nfloats * 4
        self._raw = np.empty(nbytes + 4096, dtype=np.uint8)
        off = (-self._raw.ctypes.data) % 4096
        self._arr = self._raw[off:off + nbytes].view(np.float32)
        self._rt = torch.cuda.cudart()
        rc = self._rt.cudaHostRegister(self._arr.ctypes.data, nbytes, 0)
        if int(rc if not isinstance(rc, tuple) else rc[0]) != 0:
            raise RuntimeError(f"cudaHostRegister of {nbytes / 1e9:.1f} GB failed: {rc}")
        self.tensor = torch.from_numpy(self._arr)

    def release(self):
        if self._arr is not None:
            self._rt.cudaHostUnregister(self._arr.ctypes.data)
            self._arr = self.tensor = None


def fragment_e2e(wl, F, g, m, reps_d, host, sync, args, world, dev):
    """The same step through the public API with host buffers: every step
    uploads the present learners' replicas of the fragment from pinned host
    memory (torch's pinned allocator; one copy of the whole block when every
    learner is present, else one per learner) on an upload stream into one of
    two device buffers, runs dl_outer_sync as soon as they have landed, and
    downloads the updated theta_g on a download stream. Uploads of step s+1 run while step s
    computes and downloads; the step after waits for the download before it
    updates theta_g again."""
    import torch

    K, n = wl.K, F.n
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    stride = reps_d.stride(0)
    # the padded [K, stride] blocks behind the [K, n] views: with every learner
    # present a step uploads its replicas as one contiguous copy
    full_d = [reps_d.as_strided((K, stride), (stride, 1)),
              torch.empty(K, stride, dtype=torch.float32, device=dev)]
    bufs = [full_d[0][:, :n], full_d[1][:, :n]]
    g_out = torch.empty(n, dtype=torch.float32, pin_memory=True)
    h_reps = host[1]
    h_full = h_reps.as_strided((K, stride), (stride, 1))

    def run(steps):
        ready = [torch.cuda.Event() for _ in range(steps)]
        done = [torch.cuda.Event() for _ in range(steps)]
        fetched = [torch.cuda.Event() for _ in range(steps)]
        bi = 0
        for s in range(steps):
            present, weights = quorum_schedule(wl, s)
            buf = bufs[s % 2]
            with torch.cuda.stream(up):
                if s >= 2:
                    up.wait_event(done[s - 2])
                if present.all():
                    full_d[s % 2].copy_(h_full, non_blocking=True)
                    bi += K * stride * 4
                else:
                    for k in range(K):
                        if present[k]:
                            buf[k].copy_(h_reps[k], non_blocking=True)
                            bi += n * 4
                ready[s].record(up)
            comp.wait_event(ready[s])
            if s >= 1:
                comp.wait_event(fetched[s - 1])
            sync.step([g], [m], [[buf[k] for k in range(K)]], weights=[weights],
                      present=[present], stream=comp)
            done[s].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(done[s])
                g_out.copy_(g, non_blocking=True)
                fetched[s].record(down)
        comp.wait_stream(up)
        comp.wait_stream(down)
        return bi

    steps = max(3, min(args.steps, 6))
    run(2)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    bi = run(steps)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    if world > 1:
        dt = max_over_ranks(dt, world, dev)
    # the host link alone, CUDA events: the same replica block copied by
    # itself from the staging buffer, and one replica copied from a
    # page-aligned host buffer registered with cudaHostRegister
    def copy_gbs(dst, src, reps=2):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(comp)
        for _ in range(reps):
            dst.copy_(src, non_blocking=True)
        b.record(comp)
        torch.cuda.synchronize()
        return reps * src.numel() * 4 / (a.elapsed_time(b) / 1e3) / 1e9

    plain = copy_gbs(full_d[1], h_full)
    registered = None
    try:
        rh = RegisteredHost(n)
        try:
            rh.tensor.copy_(h_reps[0])
            registered = copy_gbs(full_d[1][0, :n], rh.tensor)
        finally:
            rh.release()
    except (RuntimeError, MemoryError):
        registered = None
    return {"value": world * n * steps / dt, "unit": UNIT, "h2d_bytes_per_step": bi // steps,
            "d2h_bytes_per_step": n * 4, "steps": steps, "ms_per_step": dt / steps * 1e3,
            "h2d_gbs": bi / dt / 1e9, "h2d_plain_copy_gbs": plain,
            "h2d_registered_copy_gbs": registered,
            "note": "present replicas H2D from pinned memory on an upload stream (one copy of "
                    "the whole [K, n] block when every learner is present; two device buffers, "
                    "step s+1 uploads while step s computes), dl_outer_sync per step, updated "
                    "theta_g D2H on a download stream; momentum and theta_g stay on the device. "
                    "h2d_plain_copy_gbs: the same block copied alone from torch's pinned "
                    "memory; h2d_registered_copy_gbs: one replica from a cudaHostRegister'ed "
                    "buffer"}


def run_fragment(args, rank, world, local):
    """One fragment resident in HBM with its K replicas; a step is one outer
    synchronisation of that fragment through dl_outer_sync (stats -> quantise
    -> merge + Nesterov), momentum and theta_g carried from step to step. A
    second timed pass makes the same steps as separate C-ABI calls with CUDA
    events around each call."""
    import torch

    import pseudo_grad_sync_gb300 as dl

    dev = f"cuda:{local}"
    torch.cuda.set_device(local)
    wl = synthetic.WORKLOADS[args.workload]()
    K = wl.K
    ts, fid = bench_fragment(wl, dl.plan_fragments, args.fragment)
    if args.sample_elems:
        # a smaller case of the same kernels (profiling): the fragment's
        # tensors in order up to that many elements
        ts = fragment_cpu_sample(wl, ts, args.sample_elems, generate=False)[4]
    numels = [wl.numels[t] for t in ts]
    F = dl.Fragment(numels, dev)
    n = F.n
    # inputs filled on the device from a seeded generator (seconds, where the
    # host generator would take minutes for every rank of a multi-GPU run);
    # the e2e pass uploads a pinned host copy of the same values
    t0 = time.time()
    g, reps = fragment_device_fill(wl, ts, dev, seed=rank)
    host, e2e_error = None, None
    if not args.no_e2e and wl.name != "ragged_heavy":
        try:
            h_reps = torch.empty(K, reps.stride(0), dtype=torch.float32, pin_memory=True)[:, :n]
            h_reps.copy_(reps)
            host = (None, h_reps)
        except (RuntimeError, MemoryError) as exc:  # host memory exhausted (many ranks per node)
            e2e_error = f"pinned host buffer of {K * reps.stride(0) * 4 / 1e9:.1f} GB: {exc}"[:300]
    gen_s = time.time() - t0
    m = torch.zeros_like(g)
    rep_list = [reps[k] for k in range(K)]
    sync = dl.ModelSync([F], K, dev)
    stats = dl.new_stats(K, F.T, dev)
    ws_s = dl.new_workspace(dl.stats_workspace_bytes(F, K), dev)
    ws_q = dl.new_workspace(dl.quantize_workspace_bytes(F, K), dev)
    codebook = torch.empty((K, F.T, 256), dtype=torch.float32, device=dev)
    codes = [torch.empty(n, dtype=torch.uint8, device=dev) for _ in range(K)]
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()

    def sync_step(s):
        present, weights = quorum_schedule(wl, s)
        sync.step([g], [m], [rep_list], weights=[weights], present=[present], stream=stream)

    def call_step(s, ev=None):
        present, weights = quorum_schedule(wl, s)
        idx = [k for k in range(K) if present[k]]
        kp = len(idx)
        rp = [rep_list[k] for k in idx]
        w = np.asarray(weights, dtype=np.float32)[idx]
        if ev is not None:
            ev[0].record(stream)
        dl.pseudograd_stats(g, rp, F, 6.0, stats[:kp], ws_s, stream)
        if ev is not None:
            ev[1].record(stream)
        dl.quantize(g, rp, F, stats[:kp], codes[:kp], codebook[:kp], None, ws_q, stream)
        if ev is not None:
            ev[2].record(stream)
        dl.merge_outer_step(g, m, F, codes[:kp], codebook[:kp], weights=w, lr=0.7, mu=0.9,
                            stream=stream)
        if ev is not None:
            ev[3].record(stream)
        return kp

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    for s in range(args.warmup):
        sync_step(s)
        call_step(s)
    barrier()
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:
        uuid = None
    clocks = ClockSampler(uuid)
    clocks.start()
    time.sleep(0.3)

    def timed(body):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        start.record(stream)
        for s in range(args.steps):
            body(s)
        end.record(stream)
        barrier()
        return max_over_ranks(start.elapsed_time(end), world, dev) / args.steps

    ms_per_step = timed(sync_step)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    kps = []
    ms_calls = timed(lambda s: kps.append(call_step(s, ev[s])))
    clk = clocks.stop()

    peak, peak_kind = load_peaks()
    calls = {}
    for i, name in enumerate(("stats", "quantize", "merge")):
        tot_ms = sum(e[i].elapsed_time(e[i + 1]) for e in ev)
        tot_bytes = sum(algo_bytes(kp)[name] * n for kp in kps)
        gbs = tot_bytes / (tot_ms / 1e3) / 1e9
        calls[name] = {"ms_per_step": tot_ms / args.steps, "achieved_gbs": gbs,
                       "frac": gbs / peak,
                       "algo_bytes_per_elem": sum(algo_bytes(kp)[name] for kp in kps) / len(kps)}
    step_bytes = sum((10 * kp + 24) * n for kp in kps) / len(kps)
    full_gbs = step_bytes / (ms_per_step / 1e3) / 1e9
    dominant = max(calls, key=lambda c: calls[c]["ms_per_step"])
    mean_np = sum(kps) / len(kps)
    kernel_of = {"stats": "k_stats", "quantize": "k_quantize",
                 "merge": "k_merge_tma"}
    tr = traffic_record(kernel_of[dominant])
    traffic = None if tr is None else tr["dram_bytes_per_elem"] * n
    roofline = {"bound": "hbm", "achieved": round(calls[dominant]["achieved_gbs"], 1),
                "peak": peak, "unit": "GB/s", "frac": round(calls[dominant]["frac"], 4),
                "traffic": traffic, "kernel": kernel_of[dominant],
                "note": (f"call '{dominant}' timed with CUDA events around its C-ABI call in "
                         "the per-call pass; algorithmic bytes per launch = "
                         f"{calls[dominant]['algo_bytes_per_elem']:.2f} B/elem x {n} elements; "
                         f"peak = {peak_kind} copy bandwidth from MEASURED_PEAKS.json; traffic "
                         "= ncu DRAM bytes per launch (null unless captured for this source)")}
    e2e = None
    if host is not None:
        e2e = fragment_e2e(wl, F, g, m, reps, host, sync, args, world, dev)
    elif e2e_error is not None:
        e2e = {"value": None, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0,
               "error": e2e_error}
    desc = {"decoder_10b": f"10B decoder set cut into P=24 by the LPT planner; the {args.fragment} "
                           f"fragment (#{fid}, {len(ts)} tensors) synced per step with K={K} "
                           "replicas resident, momentum carried across steps",
            "quorum_10b": f"10B shapes, the {args.fragment} fragment "
                          f"(#{fid}, {len(ts)} tensors), K={K} learners with a random present "
                          "subset of 1..16 and weights U[0.5,1.5] per step (the workload's "
                          "(fragment, outer step) draws in turn), momentum carried",
            "ragged_heavy": f"{len(ts)} ragged tensors 64..16Mi as one batch, K={K}, "
                            "Delta = 1e-3 Student-t(3)"}[wl.name]
    out = {
        "metric": METRIC, "value": world * n / (ms_per_step / 1e3), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (device-filled, seeded)",
        "config": {"workload": wl.name + ": " + desc, "K": K, "fragment_elems": n,
                   "fragment_tensors": len(ts), "mean_present_learners": mean_np,
                   "sample_elems": args.sample_elems or None,
                   "l2": "no flush: every call streams >= 12 GB, inputs far larger than L2",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "full_step_gbs": full_gbs, "full_step_frac": full_gbs / peak,
        "full_step_algo_bytes_per_elem": step_bytes / n,
        "ms_per_step_serial_calls": ms_calls, "calls": calls, "roofline": roofline,
        "clocks": clk, "gpu_launches": args.steps * sum(LAUNCHES_PER_FRAGMENT.values()),
        "gpu_launches_note": "kernels in the headline dl_outer_sync region; the per-call pass "
                             "launches the same number again",
        "e2e": e2e, "setup_generate_s": gen_s,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = fragment_cpu_baseline(wl, ts, args.cpu_budget)
    if rank == 0:
        print(json.dumps(out), flush=True)


def run_ours(args, rank, world, local):
    import torch

    import pseudo_grad_sync_gb300 as dl

    dev = f"cuda:{local}"
    torch.cuda.set_device(local)
    wl = synthetic.WORKLOADS[args.workload]()
    frag_of, load = dl.plan_fragments(wl.numels, wl.n_frags)
    frags = fragment_tensors(wl, frag_of)
    K = wl.K
    n_total = wl.n_elems
    t0 = time.time()
    host = generate_host(wl, frags, pin=not args.no_e2e)
    gen_s = time.time() - t0
    run = DeviceRun(wl, frags, host, dev)
    stream = torch.cuda.current_stream()

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        run.sync_step(stream)
        run.step(stream=stream)
    barrier()

    ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in frags]
          for _ in range(args.steps)]
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:
        uuid = None
    clocks = ClockSampler(uuid)
    clocks.start()
    time.sleep(0.3)

    def timed(body):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        start.record(stream)
        for s in range(args.steps):
            body(s)
        end.record(stream)
        barrier()
        ms = max_over_ranks(start.elapsed_time(end), world, dev)
        return ms / args.steps

    # headline: the whole step through dl_outer_sync (consecutive fragments
    # overlapped on two streams)
    ms_per_step = timed(lambda s: run.sync_step(stream))
    # per-call breakdown: the same step as separate C-ABI calls on one stream,
    # each bracketed by CUDA events
    ms_per_step_calls = timed(lambda s: run.step(events=ev[s], stream=stream))
    clk = clocks.stop()

    # per-call device time (CUDA events inside the timed region)
    per_call = {"stats": 0.0, "quantize": 0.0, "merge": 0.0}
    for s in range(args.steps):
        for f in range(len(frags)):
            e = ev[s][f]
            per_call["stats"] += e[0].elapsed_time(e[1])
            per_call["quantize"] += e[1].elapsed_time(e[2])
            per_call["merge"] += e[2].elapsed_time(e[3])
    peak, peak_kind = load_peaks()
    ab = algo_bytes(K)
    calls = {}
    for name, tot_ms in per_call.items():
        launches = args.steps * len(frags)
        avg_s = tot_ms / launches / 1e3
        bytes_per_launch = ab[name] * n_total / len(frags)
        gbs = bytes_per_launch / avg_s / 1e9
        calls[name] = {"ms_per_step": tot_ms / args.steps, "avg_launch_us": avg_s * 1e6,
                       "algo_bytes_per_elem": ab[name], "achieved_gbs": gbs,
                       "frac": gbs / peak}
    full_gbs = (sum(ab.values()) * n_total) / (ms_per_step / 1e3) / 1e9
    dominant = max(calls, key=lambda c: calls[c]["ms_per_step"])
    kernel_of = {"stats": "k_stats", "quantize": "k_quantize",
                 "merge": "k_merge_tma"}
    tr = traffic_record(kernel_of[dominant])
    traffic = None
    if tr is not None:
        traffic = tr["dram_bytes_per_elem"] * n_total / len(frags)
    roofline = {"bound": "hbm", "achieved": round(calls[dominant]["achieved_gbs"], 1),
                "peak": peak, "unit": "GB/s",
                "frac": round(calls[dominant]["frac"], 4), "traffic": traffic,
                "kernel": kernel_of[dominant],
                "note": (f"call '{dominant}' timed with CUDA events around its C-ABI call "
                         "in the per-call pass (includes its small setup/finalise kernels); "
                         f"peak = {peak_kind} copy bandwidth from MEASURED_PEAKS.json; "
                         "traffic = ncu DRAM bytes per launch (null if not captured for "
                         "this source)")}

    # end to end: replicas arrive from pinned host memory, theta_g goes back
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(run, host, args, world, dev)

    value = world * n_total / (ms_per_step / 1e3)
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl.name + ": " + wl.description, "K": K,
                   "fragments": wl.n_frags, "params": n_total,
                   "fragment_elems_min_max": [int(load.min()), int(load.max())],
                   "l2": "no flush: every call streams >= 0.9 GB, inputs larger than L2",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "full_step_gbs": full_gbs, "full_step_frac": full_gbs / peak,
        "ms_per_step_serial_calls": ms_per_step_calls,
        "calls": calls, "roofline": roofline, "clocks": clk,
        "gpu_launches": args.steps * len(frags) * sum(LAUNCHES_PER_FRAGMENT.values()),
        "gpu_launches_note": "kernels in the headline dl_outer_sync region; the per-call "
                             "pass launches the same number again",
        "e2e": e2e, "setup_generate_s": gen_s,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(wl, frags, host, budget_s=args.cpu_budget)
    if rank == 0:
        print(json.dumps(out), flush=True)


def run_e2e(run, host, args, world, dev):
    """Same step through the public API with host buffers: each fragment's K
    replicas are copied from pinned host memory on an upload stream (double-
    buffered), the fragment is synced with dl_outer_sync as soon as they land,
    and the updated theta_g goes back on a download stream, all inside the
    timed region. Uploads never wait for downloads, so the upload link stays
    busy for the whole step."""
    import torch

    K = run.wl.K
    max_n = max(f.n for f in run.F)
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    stage = [[torch.empty(max_n, dtype=torch.float32, device=dev) for _ in range(K)]
             for _ in range(2)]
    g_out = [torch.empty_like(h[0], pin_memory=True) for h in host]
    nF = len(run.F)
    bi = sum(K * f.n * 4 for f in run.F)
    bo = sum(f.n * 4 for f in run.F)
    ws = run.msync.workspace  # sized for the largest fragment

    def one_step():
        ready = [torch.cuda.Event() for _ in range(nF)]
        done = [torch.cuda.Event() for _ in range(nF)]
        for f in range(nF):
            buf = stage[f % 2]
            n = run.F[f].n
            with torch.cuda.stream(up):
                if f >= 2:
                    up.wait_event(done[f - 2])
                for k in range(K):
                    buf[k][:n].copy_(host[f][1][k], non_blocking=True)
                ready[f].record(up)
            comp.wait_event(ready[f])
            run.dl.outer_sync([run.F[f]], [run.g[f]], [run.m[f]], [[b[:n] for b in buf]], K,
                              workspace=ws, stream=comp)
            done[f].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(done[f])
                g_out[f].copy_(run.g[f], non_blocking=True)
        comp.wait_stream(up)
        comp.wait_stream(down)

    steps = max(2, min(args.steps, 5))
    for _ in range(2):
        one_step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for _ in range(steps):
        one_step()
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    if world > 1:
        dt = max_over_ranks(dt, world, dev)
    return {"value": world * run.wl.n_elems * steps / dt, "unit": UNIT,
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "steps": steps,
            "ms_per_step": dt / steps * 1e3, "h2d_gbs": bi * steps / dt / 1e9,
            "note": "replicas H2D from pinned memory on an upload stream (double-buffered), "
                    "dl_outer_sync per fragment as it lands, updated theta_g D2H on a "
                    "download stream; momentum and theta_g state stay on the device; "
                    "bound by the host-to-device link"}


# ---------------------------------------------------------------------------
# CPU oracle timings


def oracle_pass(wl, host, offsets):
    """One whole-model step of the oracle, fragment by fragment, on the host
    copy of the workload (the outer step; for a learner workload, stats and
    quantisation only); returns the seconds it took."""
    import oracle

    t0 = time.perf_counter()
    for (g, reps), off in zip(host, offsets):
        gn = g.numpy()
        rn = [r.numpy() for r in reps]
        if wl.role == "learner":
            oracle.quantize(gn, rn, oracle.stats(gn, rn, off), off)
            continue
        o = oracle.outer_step(gn, np.zeros_like(gn), rn, offsets=off)
        assert o["status"] == 0
    return time.perf_counter() - t0


def fragment_offsets(wl, frags):
    out = []
    for ts in frags:
        off = np.zeros(len(ts) + 1, dtype=np.int64)
        np.cumsum([wl.numels[t] for t in ts], out=off[1:])
        out.append(off)
    return out


def cpu_baseline(wl, frags, host, budget_s=10.0):
    """The oracle on the host cores over the same workload (the same host
    arrays the GPU run uploads): whole-model passes until budget_s elapsed."""
    import oracle

    offsets = fragment_offsets(wl, frags)
    oracle.lib()  # build and load it outside the timed passes
    total, passes = 0.0, 0
    while passes == 0 or total < budget_s:
        total += oracle_pass(wl, host, offsets)
        passes += 1
    # one thread, on the first fragment (a whole pass would take minutes)
    cores = oracle.threads()
    n0 = int(offsets[0][-1])
    oracle.set_threads(1)
    try:
        t1 = oracle_pass(wl, host[:1], offsets[:1])
    finally:
        oracle.set_threads(cores)
    return {"value": wl.n_elems * passes / total, "unit": UNIT, "cores": cores,
            "kind": "oracle",
            "sample": f"the whole workload ({wl.n_elems} elements x K={wl.K}, "
                      f"{len(frags)} fragments), full outer step (stats+quantise+merge+"
                      f"Nesterov) per fragment, {passes} pass(es) in {total:.1f} s",
            "single_thread": {"value": n0 / t1, "unit": UNIT, "cores": 1,
                              "sample": f"fragment 0 ({n0} elements x K={wl.K}), one pass "
                                        f"in {t1:.1f} s"}}


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step is one outer step of the
    workload on the host cores (for a fragment workload, of a bounded sample
    of the bench fragment: its tensors in order up to 2^25 elements)."""
    import oracle

    if rank != 0:
        return
    wl = synthetic.WORKLOADS[args.workload]()
    oracle.lib()
    if wl.name in FRAGMENT_WORKLOADS:
        ts, fid = bench_fragment(wl, oracle.plan_fragments, args.fragment)
        g, reps, off, tot, sel = fragment_cpu_sample(wl, ts, 1 << 25)
        for s in range(args.warmup):
            oracle_fragment_pass(g, reps, off, *quorum_schedule(wl, s))
        dt = sum(oracle_fragment_pass(g, reps, off, *quorum_schedule(wl, s))
                 for s in range(args.steps))
        n_step = tot
        part = (f"{len(sel)} of the {len(ts)} tensors of the bench fragment"
                if tot == sum(wl.numels[t] for t in sel)
                else f"the first {tot} values of the {len(ts)}-tensor bench fragment")
        sample = (f"each step: {part} ({tot} elements), full outer step with that step's "
                  "present learners")
        config = {"workload": wl.name, "K": wl.K, "fragment_elems": sum(wl.numels[t] for t in ts),
                  "fragment_tensors": len(ts)}
    else:
        frag_of, _ = oracle.plan_fragments(wl.numels, wl.n_frags)
        frags = fragment_tensors(wl, frag_of)
        host = generate_host(wl, frags, pin=False)
        offsets = fragment_offsets(wl, frags)
        for _ in range(args.warmup):
            oracle_pass(wl, host, offsets)
        dt = sum(oracle_pass(wl, host, offsets) for _ in range(args.steps))
        n_step = wl.n_elems
        sample = (f"each step: the whole workload ({wl.n_elems} elements x K={wl.K}), full "
                  "outer step on the host")
        config = {"workload": wl.name + ": " + wl.description, "K": wl.K,
                  "fragments": wl.n_frags, "params": wl.n_elems}
    value = n_step * args.steps / dt
    metric = LEARNER_METRIC if wl.role == "learner" else METRIC
    out = {"impl": "reference", "metric": metric, "value": value, "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
           "data": "synthetic", "config": config,
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.threads(),
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(synthetic.WORKLOADS), default="decoder_10b")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--sample-elems", type=int, default=0,
                    help="fragment workloads: sync only the bench fragment's tensors in "
                         "order up to this many elements (a small case for profiling)")
    ap.add_argument("--fragment", choices=["median", "largest"], default="median",
                    help="decoder_10b, quorum_10b: the fragment a step syncs (the median "
                         "one by load, or the largest: the embedding's)")
    ap.add_argument("--mode", choices=["outer", "ring", "rda"], default="outer",
                    help="ring: accumulate along a ring, re-quantising at every hop; "
                         "rda: Radial-Directional Averaging merge")
    args = ap.parse_args()
    rank, world, local = env_rank()
    if world > 1:
        import torch.distributed as dist

        if args.impl == "ours":
            import torch

            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
        else:
            dist.init_process_group("gloo")
    wl = synthetic.WORKLOADS[args.workload]()
    learner = wl.role == "learner"
    fragment = wl.name in FRAGMENT_WORKLOADS
    # whole-model workloads keep every fragment and replica resident (and, for
    # the syncer, a host copy of the inputs): refuse before allocating those
    # that do not fit; fragment workloads hold one fragment at a time
    dev_gb = (2 * 4 + 1 if learner else (wl.K + 2) * 4 + wl.K) * wl.n_elems / 1e9
    host_gb = 0.0 if learner else (wl.K + 2) * 4 * wl.n_elems / 1e9
    if not fragment and (dev_gb > 200 or host_gb > 64):
        if rank == 0:
            print(json.dumps({"error": f"workload {wl.name} needs ~{dev_gb:.0f} GB on the device "
                                       f"and ~{host_gb:.0f} GB on the host as one resident "
                                       "model"}))
        sys.exit(2)
    if fragment and args.mode != "outer" and rank == 0:
        print(json.dumps({"error": "--mode ring/rda run whole-model workloads"}))
        sys.exit(2)
    if args.impl == "reference":
        run_reference(args, rank, world)
    elif learner:
        run_learner(args, rank, world, local)
    elif fragment:
        run_fragment(args, rank, world, local)
    elif args.mode == "ring":
        run_ring(args, rank, world, local)
    elif args.mode == "rda":
        run_rda(args, rank, world, local)
    else:
        run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
