#!/usr/bin/env python
"""Benchmark of the MoE verify layer on GB300 (one JSON line on stdout).

Workload (default ``k2_layer``): DFlash K=2 verify through one MoE layer --
hidden 2048, 256 routed experts, top-8, expert intermediate 512, a shared
expert of intermediate 512, NVFP4 expert weights, bf16 router, 2 bf16 rows.
A step is one layer call -- one persistent kernel: router logits -> top-k ->
dedup -> gate/up+SwiGLU -> down -> combine -- on one batch of K rows.  Steps cycle over a ring of distinct
seeded layers whose touched bytes exceed L2 several times, so every step
streams its experts from HBM.  The timed steps run as CUDA-graph replays.

value     = algorithmic bytes / time (GB/s): router weights + the distinct
            experts' NVFP4 bytes (codes + E4M3 scales + FP32 tensor scale,
            each distinct expert once) + activations in/out.
e2e       = the same metric through the C ABI from pinned host buffers, one
            eager call per step that takes the host buffers themselves (the
            kernel reads x and writes y across the host link), or, where the
            device cannot map them, copies of x in and y out around the call.
roofline  = the experts kernel's algorithmic bytes per launch over its mean
            CUDA-event duration (a graph-captured profiling pass with events
            around each launch), against the measured HBM copy bandwidth.
stack_sweep = 40-layer verify steps at K = 1, 2, 4, 8, 16 (and the Zipf-biased
            K = 16 stack): verified tokens/s = K / step time.
laguna_router_layer = the k2_layer call with the Laguna router tail (sigmoid
            scores, selection-only bias, routed scale 2.5), GB/s as the headline.
full_step.laguna_schedule = the full step with the Laguna layer schedule
            (dense layer 0; sliding-window and full-attention layers with
            their head counts and rotary embeddings) over the same caches.
cpu_baseline = the CPU oracle on a bounded sample of the same workload.

``--impl reference`` times the CPU oracle alone on the same workload (the
reference arm).  ``--gpus N`` under torchrun runs N independent replicas
(the layer does not shard); value sums the ranks' bytes over the slowest
rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE verify-layer HBM GB/s (% of peak) and verified tokens/s at K=1..16"
FALLBACK_HBM_GBS = 6800.0
RING = 24


def parse(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=48000)
    p.add_argument("--warmup", type=int, default=48)
    p.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    p.add_argument("--workload", default="k2_layer")
    p.add_argument("--ring", type=int, default=RING)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--no-sweep", action="store_true", help="skip the 40-layer stack sweep")
    p.add_argument("--sweep-steps", type=int, default=200)
    p.add_argument("--no-full-step", action="store_true", help="skip the full verify step (attention + MoE)")
    p.add_argument("--only-full-step", action="store_true",
                   help="run only the full verify step and print its JSON object (for profiling its launches)")
    p.add_argument("--only-laguna", action="store_true",
                   help="run only the Laguna-schedule step at the full-step shape and print its JSON object "
                        "(for profiling its launches)")
    p.add_argument("--kernel-case", choices=["attention", "lm_head"], default=None,
                   help="run only one attention block (K=4, H=2048, 32/8 heads, 16,384 cached positions) or one "
                        "lm_head argmax (151,936 x 2048) a few times and print its time (a small case for ncu)")
    p.add_argument("--case-iters", type=int, default=20)
    p.add_argument("--case-heads", type=int, default=32,
                   help="q heads of the attention kernel case (64: the Laguna sliding-window layers' projections)")
    p.add_argument("--oracle-sample", type=float, default=None,
                   help="(internal) time the CPU oracle for this many seconds and print bytes/s as JSON")
    return p.parse_args(argv)


# --------------------------------------------------------------------------- helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def pctl(ms_list):
    """median, p10 and p90 of per-replay times (ms)."""
    a = np.asarray(ms_list, np.float64)
    return {"median": float(np.median(a)), "p10": float(np.percentile(a, 10)), "p90": float(np.percentile(a, 90)),
            "n": int(a.size)}


def timed_replays(torch, stream, g, n):
    """Replays graph g n times back to back on `stream`, an event pair around
    each replay; returns the per-replay times (ms) and the total (ms)."""
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    with torch.cuda.stream(stream):
        evs[0].record(stream)
        for i in range(n):
            g.replay()
            evs[i + 1].record(stream)
    stream.synchronize()
    per = [evs[i].elapsed_time(evs[i + 1]) for i in range(n)]
    return per, evs[0].elapsed_time(evs[n])


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def oracle_single_thread(workload, seconds):
    """The oracle on one host thread (OpenMP limited to 1 in a child
    process): bytes/s, or None if the child failed."""
    env = dict(os.environ, OMP_NUM_THREADS="1")
    try:
        out = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-sample", str(seconds),
                              "--workload", workload], capture_output=True, text=True, env=env,
                             timeout=max(120.0, 10 * seconds))
        d = json.loads(out.stdout.strip().splitlines()[-1])
        return d
    except Exception:
        return None


def nvfp4_bytes(rows, cols):
    return rows * cols // 2 + rows * cols // 16 + 4


def kernel_bytes(w, n_u, residual=False, K=None):
    """Algorithmic bytes of one layer call (one kernel): the router weights
    (and bias), each distinct expert once (gate, up, down, plus the shared
    expert), x, the residual, and y."""
    K = w.K if K is None else K
    act = K * w.H * 2
    slots = n_u + (1 if w.Is else 0)
    router = w.E * w.H * 2 + (w.E * 4 if w.zipf_s else 0)
    experts = router + slots * (2 * nvfp4_bytes(w.I, w.H) + nvfp4_bytes(w.H, w.I)) + act * (3 if residual else 2)
    return dict(experts=experts, layer=experts)


class Clocks:
    """Samples SM clocks and throttle reasons with nvidia-smi during a region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = tempfile.mktemp(prefix="clk", suffix=".csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        os.unlink(self.path)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dominant_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes from the committed ncu summary, if the kernel
    sources are unchanged since it was taken (else None)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.txt")
    if not os.path.exists(path):
        return None
    kv = {}
    for line in open(path):
        if ":" in line and not line.startswith(" "):
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    if (kv.get("source_sha256", "").split() or [""])[0] != source_hash(kernel):
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# the sources each profiled kernel is compiled from (None: all kernel sources)
KERNEL_SOURCES = {"experts": ["experts.cu", "internal.h", "ptx.cuh", "../../include/moe_verify.h"]}


def source_hash(kernel=None):
    """Hash of the sources a kernel is built from, to tell whether a stored
    ncu summary still describes it."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "moe_nvfp4_block_gb300", "csrc")
    files = KERNEL_SOURCES.get(kernel) if kernel else None
    if files is None:
        files = [fn for fn in sorted(os.listdir(d)) if fn.endswith((".cu", ".cuh", ".h"))]
    for fn in files:
        h.update(open(os.path.join(d, fn), "rb").read())
    return h.hexdigest()[:16]


# --------------------------------------------------------------------------- CPU oracle timing

def oracle_sample(w, seconds, first_layer=0):
    """Times the CPU oracle on whole layers of the workload until ~seconds of
    oracle time is spent; returns (bytes/s, layers, seconds, threads)."""
    import oracle
    import synthgen
    oracle.build()
    t_total, b_total, n = 0.0, 0, 0
    while t_total < seconds or n == 0:
        l = first_layer + n
        full = synthgen.make_layer(w, l, experts=[])  # router + shared only
        x = synthgen.make_x(w, l)
        ol0 = oracle.OracleLayer.from_workload(w, full)
        idx, _ = oracle.topk(oracle.router_logits_f32(ol0, x), w.top_k)
        L = synthgen.make_layer(w, l, experts=sorted(set(idx.ravel().tolist())))
        ol = oracle.OracleLayer.from_workload(w, L)
        t0 = time.perf_counter()
        r = oracle.moe_layer(ol, x)
        t_total += time.perf_counter() - t0
        b_total += kernel_bytes(w, int(r["group"][0]))["layer"]
        n += 1
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return b_total / t_total, n, t_total, threads


# --------------------------------------------------------------------------- replicas

def combine_ranks(dist, torch, world, ms, total_bytes, device):
    """Whole-job figures of N independent replicas: the slowest rank's time and
    the bytes all ranks moved (every rank calls this; an all-gather, no
    reduction order to depend on)."""
    t = torch.tensor([ms, total_bytes], dtype=torch.float64, device=device)
    tl = [torch.zeros_like(t) for _ in range(world)]
    dist.all_gather(tl, t)
    return max(float(x[0]) for x in tl), sum(float(x[1]) for x in tl)


# --------------------------------------------------------------------------- GPU arm

def run_gpu(args):
    import torch
    import synthgen
    import __graft_entry__
    __graft_entry__.build()
    import moe_nvfp4_block_gb300 as M

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if args.kernel_case:
        print(json.dumps(kernel_case(M, torch, dev, args.kernel_case, args.case_iters, args.case_heads)), flush=True)
        return
    if args.only_full_step or args.only_laguna:
        hbm, _ = peaks()
        stream = torch.cuda.Stream(device=dev)
        res = full_step(M, torch, synthgen, dev, stream, hbm, max(3, args.sweep_steps), args.only_laguna)
        print(json.dumps({"full_step": res}), flush=True)
        return
    w = synthgen.WORKLOADS[args.workload]
    R = args.ring
    t_gen = time.perf_counter()
    layers, xs, ys = [], [], []
    for l in range(R):
        L = synthgen.make_layer(w, l)
        t = lambda p: (p.codes, p.scales, p.tscale)
        sh = None if L.sh_gate is None else (t(L.sh_gate), t(L.sh_up), t(L.sh_down))
        bias = L.router_b if w.zipf_s else None
        layers.append(M.layer_from_arrays(L.router_w, bias, t(L.gate), t(L.up), t(L.down), sh, top_k=w.top_k,
                                          routed_scale=w.routed_scale, device=dev))
        xs.append(torch.from_numpy(synthgen.make_x(w, 1000 + l)).view(torch.bfloat16).to(dev))
        ys.append(torch.empty_like(xs[-1]))
        del L
    t_gen = time.perf_counter() - t_gen
    cl = [lay.c() for lay in layers]
    ws = M.workspace(layers[0], w.K, device=dev)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()

    # routing of each ring layer (deterministic) -> distinct experts -> bytes
    n_u = []
    with torch.cuda.stream(stream):
        grp = torch.empty(M.moe_group_ints(w.K, w.E, w.top_k), dtype=torch.int32, device=dev)
        for i in range(R):
            M.moe_verify_layer(layers[i], xs[i], None, ys[i], ws, group_out=grp, stream=stream, c_layer=cl[i])
            stream.synchronize()
            n_u.append(int(grp[0].item()))
    kb = [kernel_bytes(w, n) for n in n_u]

    def call(i):
        j = i % R
        M.moe_verify_layer(layers[j], xs[j], None, ys[j], ws, stream=stream, c_layer=cl[j])

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            call(i)
    stream.synchronize()
    assert M.moe_workspace_error(ws, stream) == 0

    # graphs: full passes over the ring + a remainder
    steps = args.steps
    full, rem = divmod(steps, R)
    g_full = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_full, stream=stream):
        for i in range(R):
            call(i)
    g_rem = None
    if rem:
        g_rem = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_rem, stream=stream):
            for i in range(rem):
                call(i)
    with torch.cuda.stream(stream):
        g_full.replay()
    stream.synchronize()

    clocks = Clocks(local)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # one event after every replay of the ring graph (R steps), for the
    # per-replay distribution; the events sit between graph launches and do
    # not split the programmatic overlap inside a replay
    evr = [torch.cuda.Event(enable_timing=True) for _ in range(full)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for i in range(full):
            g_full.replay()
            evr[i].record(stream)
        if g_rem is not None:
            g_rem.replay()
        ev1.record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    clk = clocks.stop()
    if dist:
        dist.barrier()
    ms = ev0.elapsed_time(ev1)
    per_replay = [(ev0 if i == 0 else evr[i - 1]).elapsed_time(evr[i]) / R for i in range(full)]
    if len(per_replay) < 200:  # too few timed replays for a distribution: 200 more, outside the timed region
        per_replay = [t / R for t in timed_replays(torch, stream, g_full, 200)[0]]
    assert M.moe_workspace_error(ws, stream) == 0
    total_bytes = sum(kb[i % R]["layer"] for i in range(steps))
    if dist:
        ms, total_bytes = combine_ranks(dist, torch, world, ms, total_bytes, dev)
    gbs = total_bytes / (ms * 1e-3) / 1e9
    hbm, peak_src = peaks()

    # kernel duration: the profiling variant (events around the launch, no
    # overlap with the next call) captured in a graph, so host gaps do not count
    n_prof = 4 * R
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_prof)]
    for e4 in evs:
        for e in e4:
            e.record(stream)
    stream.synchronize()
    g_prof = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_prof, stream=stream):
        for i in range(n_prof):
            j = i % R
            M.moe_verify_layer_profiled(layers[j], xs[j], None, ys[j], ws, events=evs[i], stream=stream,
                                        c_layer=cl[j])
    with torch.cuda.stream(stream):
        g_prof.replay()
    stream.synchronize()
    dur = {"experts": []}
    for e in evs:
        dur["experts"].append(e[1].elapsed_time(e[2]))
    mean_ms = {k: float(np.mean(v)) for k, v in dur.items()}
    dom = max(mean_ms, key=mean_ms.get)
    dom_bytes = float(np.mean([kb[i % R][dom] for i in range(n_prof)]))
    achieved = dom_bytes / (mean_ms[dom] * 1e-3) / 1e9
    traffic = dominant_traffic(dom, args.workload)

    # end to end from pinned host buffers: the call takes the host buffers
    # themselves (the kernel reads x and writes y across the host link); if
    # the device cannot map them, a copy in and out around each call
    n_e2e = min(steps, 20 * R)
    hx = [torch.empty(xs[0].shape, dtype=torch.bfloat16, pin_memory=True) for _ in range(R)]
    hy = [torch.empty(xs[0].shape, dtype=torch.bfloat16, pin_memory=True) for _ in range(R)]
    for i in range(R):
        hx[i].copy_(xs[i].cpu())
    try:
        M.host_pointer(hx[0])
        e2e_mode = "host buffers passed to the call"
    except Exception:
        e2e_mode = "copies around the call"
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    stream.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        t_enq = time.perf_counter()
        for i in range(n_e2e):
            j = i % R
            if e2e_mode == "host buffers passed to the call":
                M.moe_verify_layer(layers[j], hx[j], None, hy[j], ws, stream=stream, c_layer=cl[j])
            else:
                xs[j].copy_(hx[j], non_blocking=True)
                M.moe_verify_layer(layers[j], xs[j], None, ys[j], ws, stream=stream, c_layer=cl[j])
                hy[j].copy_(ys[j], non_blocking=True)
        t_enq = time.perf_counter() - t_enq
        e1.record(stream)
    stream.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    e2e_gbs = sum(kb[i % R]["layer"] for i in range(n_e2e)) / (e2e_ms * 1e-3) / 1e9
    act = w.K * w.H * 2

    out = {
        "metric": METRIC, "value": round(gbs, 1), "unit": "GB/s", "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": ms / steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp4(e2m1)*fp16 mma -> f32", "data": "synthetic",
        "config": {"workload": f"{args.workload}: DFlash K={w.K} verify, {w.layers} MoE layer (H={w.H}, E={w.E}, "
                               f"top-{w.top_k}, I={w.I}, shared I={w.Is}, NVFP4 experts, bf16 router)",
                   "K": w.K, "ring_layers": R,
                   "l2": f"inputs larger than L2: steps cycle over {R} distinct layers "
                         f"({R * 257 * 3 * nvfp4_bytes(w.I, w.H) / 1e9:.1f} GB resident)",
                   "launch": "CUDA graph replay; per call one persistent kernel (router, experts, combine), "
                             "programmatic dependent launch between calls",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "pct_of_peak": round(100 * gbs / hbm, 1),
        "ms_per_step_dist": dict({k: (round(v, 5) if isinstance(v, float) else v) for k, v in pctl(per_replay).items()},
                                 replay=f"one graph replay = {R} steps (one pass over the layer ring)"),
        "row_layers_per_s": round(w.K * steps / (ms * 1e-3) * world, 1),
        "layers_per_s": round(steps / (ms * 1e-3) * world, 1),
        "distinct_experts_mean": float(np.mean(n_u)),
        "clocks": clk,
        "e2e": {"value": round(e2e_gbs, 1), "unit": "GB/s", "h2d_bytes_per_step": act, "d2h_bytes_per_step": act,
                "steps": n_e2e, "mode": e2e_mode, "host_enqueue_us_per_step": round(t_enq * 1e6 / n_e2e, 2)},
        "gpu_launches": steps,
        "kernel_ms": {k: round(v, 5) for k, v in mean_ms.items()},
        "kernel_ms_dist": {k: {kk: (round(vv, 5) if isinstance(vv, float) else vv) for kk, vv in pctl(v).items()}
                           for k, v in dur.items()},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": hbm,
                     "peak_source": peak_src, "unit": "GB/s", "frac": round(achieved / hbm, 3),
                     "traffic": traffic, "algorithmic_bytes_per_launch": dom_bytes,
                     "timing": "achieved: the kernel launched alone (no programmatic overlap), CUDA events "
                               "around each launch in a graph; achieved_in_step_mode: the same bytes over the "
                               "headline's per-step time (one launch per step, overlapped with its neighbours)",
                     "achieved_in_step_mode": round(gbs / world, 1),
                     "frac_in_step_mode": round(gbs / world / hbm, 3)},
        "setup_s": round(t_gen, 1),
    }
    if not args.no_sweep:
        out["laguna_router_layer"] = laguna_router_layer(M, torch, synthgen, dev, stream, hbm, args.steps)
        out["stack_sweep"] = stack_sweep(M, torch, synthgen, dev, stream, hbm, args.sweep_steps)
    if not args.no_full_step:
        out["full_step"] = full_step(M, torch, synthgen, dev, stream, hbm, max(10, args.sweep_steps))
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        bps, n, secs, threads = oracle_sample(w, args.cpu_seconds)
        st = oracle_single_thread(args.workload, min(10.0, args.cpu_seconds))
        out["cpu_baseline"] = {"value": round(bps / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                               "sample": f"{n} whole {args.workload} layers (K={w.K}) of the same workload, "
                                         f"{secs:.1f} s of oracle time",
                               "nproc": os.cpu_count(), "cpu_model": cpu_model(),
                               "single_thread": None if st is None else
                               {"value": round(st["bytes_per_s"] / 1e9, 4), "unit": "GB/s", "cores": 1,
                                "sample": f"{st['layers']} whole layers, {st['seconds']:.1f} s of oracle time",
                                "ms_per_layer": round(st["seconds"] / st["layers"] * 1e3, 2)},
                               "ms_per_layer": round(secs / n * 1e3, 2)}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist:
        dist.destroy_process_group()


# --------------------------------------------------------------------------- 40-layer stacks

def stack_sweep(M, torch, synthgen, dev, stream, hbm, steps):
    """Verify steps through 40-layer MoE stacks (x <- x + MoE_l(rmsnorm(x))):
    K = 1, 2, 4, 8, 16 on the k8_stack40 weights and K = 16 on the Zipf-biased
    k16_zipf_stack40 weights.  A step is one pass of all 40 layers; verified
    tokens/s = K / step time; GB/s = algorithmic bytes of the step / time."""
    res = []
    for wname, Ks in (("k8_stack40", (1, 2, 4, 8, 16)), ("k16_zipf_stack40", (16,))):
        w = synthgen.WORKLOADS[wname]
        t = lambda p: (p.codes, p.scales, p.tscale)
        layers = []
        for l in range(w.layers):
            L = synthgen.make_layer(w, l)
            sh = (t(L.sh_gate), t(L.sh_up), t(L.sh_down))
            layers.append(M.layer_from_arrays(L.router_w, L.router_b if w.zipf_s else None, t(L.gate), t(L.up),
                                              t(L.down), sh, top_k=w.top_k, device=dev))
            del L
        carr = M.layer_array(layers)
        for K in Ks:
            x0 = torch.from_numpy(synthgen.make_x(w, 900 + K, K=K)).view(torch.bfloat16).to(dev)
            x = x0.clone()
            ws = M.stack_workspace(carr, K, device=dev)
            # distinct experts per layer along the stack (routing is deterministic)
            wl = M.workspace(layers[0], K, device=dev)
            xn = torch.empty_like(x)
            grp = torch.empty(M.moe_group_ints(K, w.E, w.top_k), dtype=torch.int32, device=dev)
            n_u = []
            with torch.cuda.stream(stream):
                for l in range(w.layers):
                    M.moe_rmsnorm(x, xn, stream=stream)
                    M.moe_verify_layer(layers[l], xn, x, x, wl, group_out=grp, stream=stream)
                    stream.synchronize()
                    n_u.append(int(grp[0].item()))
            step_bytes = sum(kernel_bytes(w, n, residual=True, K=K)["layer"] for n in n_u)  # (RMSNorm inside)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                x.copy_(x0)
                M.moe_verify_stack(carr, x, ws, stream=stream)
            with torch.cuda.stream(stream):
                for _ in range(3):
                    g.replay()
            stream.synchronize()
            per, tot = timed_replays(torch, stream, g, steps)
            assert M.moe_workspace_error(ws, stream) == 0
            ms = tot / steps
            gbs = step_bytes / (ms * 1e-3) / 1e9
            dist_ = pctl(per)
            res.append({"workload": wname, "K": K, "layers": w.layers, "ms_per_step": round(ms, 4),
                        "verified_tokens_per_s": round(K / (ms * 1e-3), 1), "GBps": round(gbs, 1),
                        "pct_of_peak": round(100 * gbs / hbm, 1),
                        "distinct_experts_mean": round(float(np.mean(n_u)), 2), "steps": steps,
                        "ms_median": round(dist_["median"], 4), "ms_p10": round(dist_["p10"], 4),
                        "ms_p90": round(dist_["p90"], 4), "gpu_launches_per_step": w.layers})
        del layers, carr
        torch.cuda.empty_cache()
    return res


def full_step(M, torch, synthgen, dev, stream, hbm, steps, only_laguna=False):
    """The k4_full_step workload: 40 x (GQA attention over a 16,384-position
    bf16 cache + MoE block), lm_head argmax over 151,936 rows, accepted
    prefix; one native moe_verify_step per step, replayed from a CUDA graph.
    only_laguna: build the same layers but time only the Laguna schedule."""
    w = synthgen.WORKLOADS["k4_full_step"]
    t = lambda p: (p.codes, p.scales, p.tscale)
    d = lambda a: torch.from_numpy(a).view(torch.bfloat16).to(dev)
    layers = []
    for l in range(w.layers):
        A = synthgen.make_attention(w, l)
        L = synthgen.make_layer(w, l)
        sh = (t(L.sh_gate), t(L.sh_up), t(L.sh_down))
        moe = M.layer_from_arrays(L.router_w, None, t(L.gate), t(L.up), t(L.down), sh, top_k=w.top_k, device=dev)
        layers.append(M.DecoderLayer(d(A["Wq"]), d(A["Wk"]), d(A["Wv"]), d(A["Wo"]), d(A["kc"]), d(A["vc"]), moe))
        del A, L
    model = M.VerifyModel(layers, d(synthgen.make_lm_head(w)), w.n_q_heads, w.n_kv_heads)
    if only_laguna:
        res = {"laguna_schedule": laguna_step(M, torch, synthgen, dev, stream, hbm, steps, layers, model.lm_head, w)}
        del layers, model
        torch.cuda.empty_cache()
        return res
    K = w.K
    x0 = d(synthgen.make_x(w, 11))
    x = x0.clone()
    ws = model.workspace(K, device=dev)
    tgt = torch.empty(K, dtype=torch.int32, device=dev)
    n = torch.empty(1, dtype=torch.int32, device=dev)
    draft = torch.zeros(K, dtype=torch.int32, device=dev)
    with torch.cuda.stream(stream):  # one eager step: targets -> drafts with a known accepted length
        M.moe_verify_step(model, x, draft, tgt, n, ws, stream=stream)
    stream.synchronize()
    dr, j = synthgen.make_drafts(w, tgt.cpu().numpy())
    draft.copy_(torch.from_numpy(dr))
    # distinct experts per layer (one teacher pass with the MoE routing outputs)
    wl = M.workspace(layers[0].moe, K, device=dev)
    aws = M.attention_workspace(K, w.H, w.n_q_heads, w.n_kv_heads, device=dev)
    xn = torch.empty_like(x)
    grp = torch.empty(M.moe_group_ints(K, w.E, w.top_k), dtype=torch.int32, device=dev)
    x.copy_(x0)
    n_u = []
    with torch.cuda.stream(stream):
        for l in range(w.layers):
            dl = layers[l]
            M.moe_attention_block(x, dl.Wq, dl.Wk, dl.Wv, dl.Wo, dl.kcache, dl.vcache, x, aws, w.n_q_heads,
                                  w.n_kv_heads, stream=stream)
            M.moe_rmsnorm(x, xn, stream=stream)
            M.moe_verify_layer(dl.moe, xn, x, x, wl, group_out=grp, stream=stream)
            stream.synchronize()
            n_u.append(int(grp[0].item()))
    act = K * w.H * 2
    att_bytes = 2 * (w.n_q_heads + 2 * w.n_kv_heads) * 128 * w.H + 2 * w.H * w.n_q_heads * 128 + \
        2 * 2 * w.n_kv_heads * w.ctx * 128 + 2 * act
    step_bytes = sum(att_bytes + kernel_bytes(w, nu, residual=True, K=K)["layer"] for nu in n_u) + \
        w.vocab * w.H * 2 + 2 * act
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        x.copy_(x0)
        M.moe_verify_step(model, x, draft, tgt, n, ws, stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
    stream.synchronize()
    per, tot = timed_replays(torch, stream, g, steps)
    assert M.moe_workspace_error(ws, stream) == 0
    ms = tot / steps
    dist_ = pctl(per)
    acc = int(n.item())
    gbs = step_bytes / (ms * 1e-3) / 1e9
    loop = verify_loop(M, torch, synthgen, dev, stream, model, w, steps)
    laguna = laguna_step(M, torch, synthgen, dev, stream, hbm, steps, layers, model.lm_head, w)
    res = {"workload": "k4_full_step", "K": K, "layers": w.layers, "ctx": w.ctx, "vocab": w.vocab,
           "ms_per_step": round(ms, 4), "verified_tokens_per_s": round(K / (ms * 1e-3), 1),
           "accepted": acc, "accepted_expected": j,
           "emitted_tokens_per_s": round((acc + 1 if acc < K else K) / (ms * 1e-3), 1),
           "GBps": round(gbs, 1), "pct_of_peak": round(100 * gbs / hbm, 1),
           "step_bytes": step_bytes, "distinct_experts_mean": round(float(np.mean(n_u)), 2), "steps": steps,
           "ms_median": round(dist_["median"], 4), "ms_p10": round(dist_["p10"], 4), "ms_p90": round(dist_["p90"], 4),
           "verify_loop": loop, "laguna_schedule": laguna}
    del layers, model
    torch.cuda.empty_cache()
    return res


def laguna_router_layer(M, torch, synthgen, dev, stream, hbm, steps, R=4):
    """The k2_layer shape with the Laguna router tail: sigmoid scores, a
    selection-only bias of 0.05 N(0, 1) per expert (the size of a trained
    correction bias next to scores in (0, 1)), routed scale 2.5.  A ring of R
    layers replayed from a CUDA graph, algorithmic GB/s as in the headline
    (plus the bias's E * 4 bytes)."""
    w = synthgen.WORKLOADS["k2_layer"]
    t = lambda p: (p.codes, p.scales, p.tscale)
    layers, xs, ys = [], [], []
    for l in range(R):
        L = synthgen.make_layer(w, 40 + l)
        bias = (synthgen.bf16_to_f32(synthgen.normal_bf16(31 + l, 0, synthgen.T_ROUTER_B, 0, w.E)) * 0.05)
        sh = (t(L.sh_gate), t(L.sh_up), t(L.sh_down))
        layers.append(M.layer_from_arrays(L.router_w, bias.astype(np.float32), t(L.gate), t(L.up), t(L.down), sh,
                                          top_k=w.top_k, routed_scale=2.5, device=dev,
                                          scoring=M.MOE_SCORE_SIGMOID))
        xs.append(torch.from_numpy(synthgen.make_x(w, 1100 + l)).view(torch.bfloat16).to(dev))
        ys.append(torch.empty_like(xs[-1]))
        del L
    cl = [lay.c() for lay in layers]
    ws = M.workspace(layers[0], w.K, device=dev)
    grp = torch.empty(M.moe_group_ints(w.K, w.E, w.top_k), dtype=torch.int32, device=dev)
    n_u = []
    with torch.cuda.stream(stream):
        for i in range(R):
            M.moe_verify_layer(layers[i], xs[i], None, ys[i], ws, group_out=grp, stream=stream, c_layer=cl[i])
            stream.synchronize()
            n_u.append(int(grp[0].item()))
    nbytes = [kernel_bytes(w, n)["layer"] + w.E * 4 for n in n_u]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(R):
            M.moe_verify_layer(layers[i], xs[i], None, ys[i], ws, stream=stream, c_layer=cl[i])
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
    stream.synchronize()
    n_rep = max(200, steps // R)
    per, tot = timed_replays(torch, stream, g, n_rep)
    assert M.moe_workspace_error(ws, stream) == 0
    ms = tot / (n_rep * R)
    gbs = sum(nbytes) / R / (ms * 1e-3) / 1e9
    dist_ = pctl([p / R for p in per])
    res = {"workload": "k2_layer with the Laguna router tail (sigmoid scores, selection bias, routed scale 2.5)",
           "K": w.K, "ms_per_call": round(ms, 5), "GBps": round(gbs, 1), "pct_of_peak": round(100 * gbs / hbm, 1),
           "distinct_experts_mean": round(float(np.mean(n_u)), 2), "calls": n_rep * R,
           "ms_median": round(dist_["median"], 5), "ms_p10": round(dist_["p10"], 5), "ms_p90": round(dist_["p90"], 5)}
    del layers
    torch.cuda.empty_cache()
    return res


def laguna_step(M, torch, synthgen, dev, stream, hbm, steps, base, lm_head, w):
    """The Laguna layer schedule at the full-step shape (K=4, 40 layers over
    16,384 cached positions, lm_head over 151,936 rows): layer 0 a dense
    SwiGLU MLP (intermediate 8,192), layers 1..39 the full step's MoE layers;
    per four layers three sliding-window ones (512 positions, 64 q heads,
    RoPE on all 128 dims) then a full-attention one (48 q heads, YaRN x4 over
    a 4,096 original context on 64 of the 128 dims); 8 KV heads (the full
    step's caches).  The new q/o projections and the MLP are bf16
    N(0, 0.02) drawn on the GPU.  One moe_verify_step per step, replayed from
    a CUDA graph; bytes from a teacher pass (distinct experts per layer)."""
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    r = lambda *sz: (torch.randn(*sz, device=dev, generator=g) * 0.02).to(torch.bfloat16)
    H, K, nkv = w.H, w.K, w.n_kv_heads
    layers, cfgs = [], []
    for l, b in enumerate(base):
        cfg = synthgen.laguna_layer_kind(l)
        nq = cfg["n_q_heads"]
        pos = M.attn_pos(cfg["window"], cfg["rotary_dim"], cfg["rope_theta"], cfg["yarn_factor"], cfg["yarn_orig"])
        mlp = None
        if cfg["dense"]:
            inter = synthgen.LAGUNA_DENSE_INTER
            mlp = (r(inter, H), r(inter, H), r(H, inter))
        layers.append(M.DecoderLayer(r(nq * 128, H), b.Wk, b.Wv, r(H, nq * 128), b.kcache, b.vcache,
                                     None if cfg["dense"] else b.moe, nq, pos, mlp))
        cfgs.append(cfg)
    model = M.VerifyModel(layers, lm_head, synthgen.LAGUNA_SLIDING_HEADS, nkv)
    x0 = torch.from_numpy(synthgen.make_x(w, 17)).view(torch.bfloat16).to(dev)
    x = x0.clone()
    ws = model.workspace(K, device=dev)
    tgt = torch.empty(K, dtype=torch.int32, device=dev)
    n = torch.empty(1, dtype=torch.int32, device=dev)
    draft = torch.zeros(K, dtype=torch.int32, device=dev)
    with torch.cuda.stream(stream):
        M.moe_verify_step(model, x, draft, tgt, n, ws, stream=stream)
    stream.synchronize()
    dr, j = synthgen.make_drafts(w, tgt.cpu().numpy())
    draft.copy_(torch.from_numpy(dr))
    # teacher pass: each layer's block by itself, the MoE routing recorded
    x.copy_(x0)
    xn = torch.empty_like(x)
    wl = M.workspace(layers[1].moe, K, device=dev)
    grp = torch.empty(M.moe_group_ints(K, w.E, w.top_k), dtype=torch.int32, device=dev)
    mws = M.dense_mlp_workspace(K, H, synthgen.LAGUNA_DENSE_INTER, device=dev)
    n_u, step_bytes = [], 0
    act = K * H * 2
    with torch.cuda.stream(stream):
        for l, (dl, cfg) in enumerate(zip(layers, cfgs)):
            nq = cfg["n_q_heads"]
            aws = M.attention_workspace(K, H, nq, nkv, device=dev)
            M.moe_attention_block(x, dl.Wq, dl.Wk, dl.Wv, dl.Wo, dl.kcache, dl.vcache, x, aws, nq, nkv,
                                  stream=stream, pos=dl.pos)
            seen = min(w.ctx, cfg["window"]) if cfg["window"] else w.ctx
            step_bytes += 2 * (nq + 2 * nkv) * 128 * H + 2 * H * nq * 128 + 2 * 2 * nkv * seen * 128 + 2 * act
            if cfg["dense"]:
                M.moe_dense_mlp_block(x, dl.mlp[0], dl.mlp[1], dl.mlp[2], x, mws, stream=stream)
                step_bytes += 3 * 2 * dl.mlp[0].shape[0] * H + 3 * act
            else:
                M.moe_rmsnorm(x, xn, stream=stream)
                M.moe_verify_layer(dl.moe, xn, x, x, wl, group_out=grp, stream=stream)
                stream.synchronize()
                n_u.append(int(grp[0].item()))
                step_bytes += kernel_bytes(w, n_u[-1], residual=True, K=K)["layer"]
            stream.synchronize()
    step_bytes += w.vocab * H * 2 + 2 * act
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=stream):
        x.copy_(x0)
        M.moe_verify_step(model, x, draft, tgt, n, ws, stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            gr.replay()
    stream.synchronize()
    per, tot = timed_replays(torch, stream, gr, steps)
    assert M.moe_workspace_error(ws, stream) == 0
    ms = tot / steps
    dist_ = pctl(per)
    acc = int(n.item())
    gbs = step_bytes / (ms * 1e-3) / 1e9
    res = {"workload": "Laguna schedule at the k4_full_step shape (dense layer 0, 3 sliding : 1 full attention, "
                       "64 / 48 q heads, RoPE / YaRN)",
           "K": K, "layers": len(layers), "ctx": w.ctx, "vocab": w.vocab, "ms_per_step": round(ms, 4),
           "verified_tokens_per_s": round(K / (ms * 1e-3), 1), "accepted": acc, "accepted_expected": j,
           "GBps": round(gbs, 1), "pct_of_peak": round(100 * gbs / hbm, 1), "step_bytes": step_bytes,
           "distinct_experts_mean": round(float(np.mean(n_u)), 2), "steps": steps,
           "ms_median": round(dist_["median"], 4), "ms_p10": round(dist_["p10"], 4), "ms_p90": round(dist_["p90"], 4)}
    del layers, model
    torch.cuda.empty_cache()
    return res


def kernel_case(M, torch, dev, which, iters, nq=32):
    """One attention block of the full-step shape (nq q heads) or one lm_head argmax,
    launched `iters` times back to back on one stream (no graph), random bf16
    operands; µs per call and algorithmic GB/s.  Sized for an ncu capture
    (about 0.1 / 0.6 GB on the device)."""
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    r = lambda *s, sd=0.02: (torch.randn(*s, device=dev, generator=g) * sd).to(torch.bfloat16)
    K, H, nkv, C, V = 4, 2048, 8, 16384, 151936
    st = torch.cuda.Stream(device=dev)
    if which == "attention":
        Wq, Wk, Wv, Wo = r(nq * 128, H), r(nkv * 128, H), r(nkv * 128, H), r(H, nq * 128)
        kc, vc = r(nkv, C, 128, sd=1.0), r(nkv, C, 128, sd=1.0)
        x = r(K, H, sd=1.0)
        ws = M.attention_workspace(K, H, nq, nkv, device=dev)
        call = lambda: M.moe_attention_block(x, Wq, Wk, Wv, Wo, kc, vc, x, ws, nq, nkv, stream=st)
        nbytes = 2 * ((nq + 2 * nkv) * 128 * H + H * nq * 128 + 2 * nkv * C * 128 + 2 * K * H)
    else:
        lm = r(V, H)
        xn = r(K, H, sd=1.0)
        tok = torch.empty(K, dtype=torch.int32, device=dev)
        ws = M.lm_head_workspace(K, device=dev)
        call = lambda: M.moe_lm_head_argmax(xn, lm, tok, ws, stream=st)
        nbytes = 2 * (V * H + K * H)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    with torch.cuda.stream(st):
        for _ in range(3):
            call()
        ev[0].record(st)
        for _ in range(iters):
            call()
        ev[1].record(st)
    st.synchronize()
    us = ev[0].elapsed_time(ev[1]) * 1e3 / iters
    assert M.moe_workspace_error(ws, st) == 0
    return {"kernel_case": which, "q_heads": nq, "us_per_call": round(us, 2), "GBps": round(nbytes / (us * 1e-6) / 1e9, 1),
            "bytes": nbytes, "iters": iters}


def verify_loop(M, torch, synthgen, dev, stream, model, w, steps, rounds=16, accept_pct=75):
    """The multi-round verify loop on the full-step model: each layer's
    16,384 cached positions copied into caches with room for the rounds, a
    device-side length, and `rounds` rounds per replay (forward with in-place
    KV append, greedy tokens, synthetic drafts accepted with probability
    accept_pct % per row, accepted prefix, commit) -- one call, no host
    involvement between rounds.  Committed tokens/s counts min(n + 1, K) per
    round."""
    out = []
    for K in (2, 4):
        cap = ((w.ctx + rounds * K + 15) // 16) * 16
        layers = []
        for d in model.layers:
            kc = torch.zeros(d.kcache.shape[0], cap, d.kcache.shape[2], dtype=d.kcache.dtype, device=dev)
            vc = torch.zeros_like(kc)
            kc[:, :w.ctx].copy_(d.kcache)
            vc[:, :w.ctx].copy_(d.vcache)
            layers.append(M.DecoderLayer(d.Wq, d.Wk, d.Wv, d.Wo, kc, vc, d.moe))
        kv_len = torch.tensor([w.ctx], dtype=torch.int32, device=dev)
        kv0 = kv_len.clone()
        lm = M.VerifyModel(layers, model.lm_head, w.n_q_heads, w.n_kv_heads, kv_len=kv_len)
        import dataclasses
        wk = dataclasses.replace(w, K=K)
        xr = torch.from_numpy(np.stack([synthgen.make_x(wk, 700 + t) for t in range(rounds)])).view(torch.bfloat16).to(dev)
        coin, alt = synthgen.make_coins(wk, rounds, accept_pct)
        coin_d, alt_d = torch.from_numpy(coin).to(dev), torch.from_numpy(alt).to(dev)
        xw = torch.empty(K, w.H, dtype=torch.bfloat16, device=dev)
        tg = torch.empty(rounds, K, dtype=torch.int32, device=dev)
        df = torch.empty_like(tg)
        na = torch.empty(rounds, dtype=torch.int32, device=dev)
        ws = lm.workspace(K, device=dev)
        with torch.cuda.stream(stream):
            kv_len.copy_(kv0)
            M.moe_verify_rounds(lm, xr, coin_d, alt_d, xw, tg, df, na, ws, stream=stream)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            kv_len.copy_(kv0)
            M.moe_verify_rounds(lm, xr, coin_d, alt_d, xw, tg, df, na, ws, stream=stream)
        with torch.cuda.stream(stream):
            for _ in range(2):
                g.replay()
        stream.synchronize()
        n_rep = max(3, steps // rounds)
        per, tot = timed_replays(torch, stream, g, n_rep)
        assert M.moe_workspace_error(ws, stream) == 0
        n = na.cpu().numpy()
        committed = int(np.minimum(n + 1, K).sum())
        ms_round = tot / n_rep / rounds
        out.append({"K": K, "rounds": rounds, "accept_pct": accept_pct, "ms_per_round": round(ms_round, 4),
                    "ms_per_round_median": round(float(np.median(per)) / rounds, 4),
                    "rounds_accepting": int((n > 0).sum()), "mean_accepted": round(float(n.mean()), 3),
                    "kv_len_final": int(kv_len.item()), "committed_tokens_per_round": round(committed / rounds, 3),
                    "committed_tokens_per_s": round(committed / (tot / n_rep * 1e-3), 1), "replays": n_rep})
        del layers, lm
        torch.cuda.empty_cache()
    return out


# --------------------------------------------------------------------------- reference arm (CPU oracle)

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import synthgen
    w = synthgen.WORKLOADS[args.workload]
    # warm-up, then timed oracle steps; a step is one whole layer of the
    # workload; the number of timed steps is capped to keep the run short
    budget_s = 90.0
    bps_w, _, t_w, _ = oracle_sample(w, 0.0, first_layer=0) if args.warmup > 0 else (0, 0, 0, 0)
    per_step = max(t_w, 1e-3)
    n = max(1, min(args.steps, int(budget_s / per_step)))
    t0 = time.perf_counter()
    bytes_total, secs_total = 0.0, 0.0
    for i in range(n):
        bps, _, secs, threads = oracle_sample(w, 0.0, first_layer=1 + i)
        bytes_total += bps * secs
        secs_total += secs
    wall = time.perf_counter() - t0
    gbs = bytes_total / secs_total / 1e9
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    sample = (f"{n} of the requested {args.steps} steps (each one whole {args.workload} layer, K={w.K}); "
              f"{secs_total:.1f} s oracle time, {wall:.1f} s wall incl. input generation")
    out = {"impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": args.gpus,
           "steps": n, "warmup": args.warmup, "ms_per_step": secs_total / n * 1e3, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": f"{args.workload}: DFlash K={w.K} verify, {w.layers} MoE layer (H={w.H}, E={w.E}, "
                                  f"top-{w.top_k}, I={w.I}, shared I={w.Is})", "K": w.K},
           "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


if __name__ == "__main__":
    a = parse()
    if a.oracle_sample is not None:
        import synthgen
        bps, n, secs, threads = oracle_sample(synthgen.WORKLOADS[a.workload], a.oracle_sample)
        print(json.dumps({"bytes_per_s": bps, "layers": n, "seconds": secs, "threads": threads}))
    elif a.impl == "reference":
        run_reference(a)
    else:
        run_gpu(a)
