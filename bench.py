"""Benchmark of the FFA hot path on GB300: one step = ffa_plan + ffa_fwd + ffa_bwd
over one synthetic batch of the 1M-token varlen-causal GQA workload.

Metric (MagiAttention blog, "Training and Benchmark settings"): TFLOPs/s with
FLOPs(fwd) = 4 * MaskArea * Hq * d and FLOPs(bwd) = 2.5 * FLOPs(fwd); the
step's value is (fwd + bwd FLOPs) / step time.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Under torchrun (N > 1) every rank runs the same workload on its own GPU as an
independent replica (heads and batches are independent; no collective on the
data path), the timed region is bracketed by barriers, the time is the max
over ranks, and rank 0 prints one JSON line.  ``--impl reference`` times the
fp64 CPU oracle on a bounded sample of the workload instead.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "FFA fwd/bwd TFLOPs/s on mask-area FLOPs; % of GB300 dense BF16 peak"
# The nominal dense bf16 figure the scope table asks the percentages to be quoted against as well.
NOMINAL_BF16_TFLOPS = 2500.0
# The configurations measured beside the headline one (a few steps each; the 1M workload is the headline).
SIDE_CONFIGS = ("tiny_mixed", "varlen_causal_64k", "video_block_causal_128k", "sink_window_256k")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {"bf16_tflops": pk["bf16_tflops"], "bf16_tflops_sustained": pk["bf16_tflops_sustained"],
                "hbm_gbs": pk["hbm_gbs"], "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


def dist_setup(n_gpus):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [l.strip().split(", ") for l in self.file.read().splitlines() if l.strip()]
        os.unlink(self.file.name)
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                pw.append(float(r[3]))
            except (ValueError, IndexError):
                continue
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        load = [s for s, p in zip(sm, pw) if p >= 0.5 * max(pw)] or sm
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(pw)}


# ----------------------------------------------------------------------------
# CPU (oracle) leg
# ----------------------------------------------------------------------------

def oracle_sample(w):
    """A bounded piece of the workload for the fp64 CPU oracle: the first
    document of at most 16384 tokens, the first kv-head group, forward +
    backward over all its rows and keys."""
    docs = sorted({(s.q_start, s.q_end) for s in w.slices})
    a, b = next(((x, y) for x, y in docs if y - x <= 16384), docs[0])
    G = w.hq // w.hkv
    return a, b, G


def run_oracle_sample(w, tensors=None):
    import numpy as np
    import oracle
    import workloads as W
    a, b, G = oracle_sample(w)
    L = b - a
    t = W.make_tensors(L, G, 1, w.d, w.seed + 12345) if tensors is None else tensors
    sl = [(0, L, 0, L, 1)]
    t0 = time.perf_counter()
    oracle.attention_forward(t["q"], t["k"], t["v"], sl, w.scale)
    oracle.attention_backward(t["q"], t["k"], t["v"], t["dout"], sl, w.scale)
    dt = time.perf_counter() - t0
    area = oracle.slices_area(sl)
    flops = 3.5 * oracle.fwd_flops(area, G, w.d)
    desc = (f"fwd+bwd of one {L}-token causal document of {w.name} (kv group 0: {G} q heads, d={w.d}), "
            f"all rows and keys; FLOPs on its mask area")
    return flops, dt, desc


# The files that define ffa_bwd_main_kernel: its translation unit and every header it includes.
BWD_KERNEL_SOURCES = ("bwd.cu", "ffa_internal.h", "ptx.cuh", "tma.h")


def _code_only(text: str) -> str:
    """C/C++ source without its comments, blank lines and trailing spaces: edits to comments leave
    a kernel unchanged."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def source_sha256() -> str:
    """SHA-256 over the sources of the backward main kernel, the kernel the DRAM-traffic records
    under profiles/ describe, with comments removed: each file's name, then its code, the csrc
    files in sorted order, then include/ffa.h."""
    import hashlib
    root = os.path.dirname(os.path.abspath(__file__))
    csrc = os.path.join(root, "flexible_mask_flashattention_gb300", "csrc")
    files = [os.path.join(csrc, f) for f in sorted(BWD_KERNEL_SOURCES)]
    files.append(os.path.join(root, "include", "ffa.h"))
    h = hashlib.sha256()
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()


def recorded_traffic(workload: str):
    """DRAM bytes per launch of ffa_bwd_main_kernel from the ncu record under profiles/, or None when
    there is none for this workload or the kernel sources changed since it was taken."""
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "profiles",
                        f"ffa_bwd_main_kernel_{workload}_dram.txt")
    if not os.path.exists(path):
        return None
    rec = {}
    with open(path) as fh:
        for line in fh:
            if ":" in line:
                k, v = line.split(":", 1)
                rec[k.strip()] = v.strip()
    if rec.get("source_sha256") != source_sha256() or "traffic_bytes_per_launch" not in rec:
        return None
    return int(rec["traffic_bytes_per_launch"])


def reference_arm(args, rank, world):
    if rank != 0:
        return 0
    import workloads as W
    w = W.workload(args.workload)
    _, _, G = oracle_sample(w)
    a, b, _ = oracle_sample(w)
    t = W.make_tensors(b - a, G, 1, w.d, w.seed + 12345)
    for _ in range(args.warmup):
        run_oracle_sample(w, t)
    flops, secs = 0.0, 0.0
    desc = ""
    for _ in range(args.steps):
        f, dt, desc = run_oracle_sample(w, t)
        flops += f
        secs += dt
    value = flops / secs / 1e12
    cores = os.cpu_count()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "seqlen": w.seqlen, "hq": w.hq, "hkv": w.hkv, "d": w.d,
                       "sample": desc},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def secondary_bounds(info, hq, d):
    """Executed MMA work against the mask-area work, from the plan's block counts.

    Forward, per non-empty 128 x 128 block and q head: S = Q K^T and O += P V, 2 * bm * bn * d FLOPs
    each, plus a second P V on Partial blocks (P carried as hi + lo bf16 halves).  Backward, per k2q
    block and q head: S^T, dP^T, dV, dK at 2 * bm * bn * d each and dQ^T at 2 * bm * bn * max(d, 128)
    (a 64-dim head keeps the 128-row MMA over a zero panel).  One exponential per executed block
    element in each direction."""
    area = info["mask_area"]
    fbm, fbn, bbm, bbn = info["fwd_bm"], info["fwd_bn"], info["bwd_bm"], info["bwd_bn"]
    fwd_area_f = 4.0 * area * hq * d
    fwd_exec = 2.0 * fbm * fbn * d * hq * (2 * info["q2k_full"] + 3 * info["q2k_mask"])
    bwd_area_f = 2.5 * fwd_area_f
    bwd_exec = 2.0 * bbm * bbn * hq * (4 * d + max(d, 128)) * (info["k2q_full"] + info["k2q_mask"])
    fwd_elems = fbm * fbn * (info["q2k_full"] + info["q2k_mask"])
    bwd_elems = bbm * bbn * (info["k2q_full"] + info["k2q_mask"])
    out = {"fwd_executed_over_mask_flops": fwd_exec / fwd_area_f if area else None,
           "bwd_executed_over_mask_flops": bwd_exec / bwd_area_f if area else None,
           "fwd_exp_per_mask_element": fwd_elems / area if area else None,
           "bwd_exp_per_mask_element": bwd_elems / area if area else None,
           "partial_block_frac_fwd": info["q2k_mask"] / max(info["q2k_full"] + info["q2k_mask"], 1)}
    out["wasted_mma_frac"] = {"fwd": 1.0 - fwd_area_f / fwd_exec if fwd_exec else None,
                              "bwd": 1.0 - bwd_area_f / bwd_exec if bwd_exec else None}
    return out


def cta_balance(trace):
    """How evenly one persistent launch loaded its CTAs, from per-CTA [start ns, end ns, units, blocks]:
    busy = end - start per CTA; the span = latest end - earliest start; idle_frac = the share of
    CTA-time in the span that no unit used (1 - sum busy / (CTAs * span))."""
    import numpy as np
    if trace is None or len(trace) == 0:
        return None
    t = trace.astype(np.float64)
    busy = t[:, 1] - t[:, 0]
    span = t[:, 1].max() - t[:, 0].min()
    return {"ctas": int(len(t)), "span_ms": span / 1e6, "busy_max_ms": busy.max() / 1e6,
            "busy_mean_ms": busy.mean() / 1e6, "busy_min_ms": busy.min() / 1e6,
            "busy_max_over_mean": float(busy.max() / busy.mean()) if busy.mean() > 0 else None,
            "idle_frac": float(1.0 - busy.sum() / (len(t) * span)) if span > 0 else None,
            "units_min_max": [int(t[:, 2].min()), int(t[:, 2].max())],
            "blocks_max_over_mean": float(t[:, 3].max() / t[:, 3].mean()) if t[:, 3].mean() > 0 else None}


def planner_throughput(info, plan_ms, hbm_gbs):
    """The plan's metadata bytes over its time (the planner is integer, memory-bound work)."""
    b = info["plan_bytes"]
    gbs = b / (plan_ms / 1e3) / 1e9 if plan_ms > 0 else None
    return {"ms": plan_ms, "bytes": b, "gbs": gbs, "frac_of_hbm": gbs / hbm_gbs if gbs else None,
            "launches": info["plan_launches"]}


def pipeline_order(steps):
    """Enqueue order of the end-to-end pipeline over two device buffer sets: the inputs of step
    i + 1 are copied in before step i computes, and step i's results are copied out right after
    it, so that copies in both directions overlap the neighbouring steps' compute.  Step i uses
    buffer set i % 2; the bench adds the cross-stream waits that keep a set's copies and compute
    in order (inputs of i + 2 after compute i, compute i + 2 after the copy-out of i)."""
    order = [("h2d", 0)] if steps > 0 else []
    for i in range(steps):
        if i + 1 < steps:
            order.append(("h2d", i + 1))
        order.append(("compute", i))
        order.append(("d2h", i))
    return order


# ----------------------------------------------------------------------------
# GPU leg
# ----------------------------------------------------------------------------

def measure_side_config(ffa, W, name, stream, dev, peaks, steps=5, warmup=2):
    """fwd / bwd TFLOP/s of one more configuration (median over steps of per-kernel CUDA-event times),
    plan wall time, secondary bounds and the CTA balance of one traced launch.  L2 is flushed
    (a 256 MiB write) before every step."""
    import torch
    w = W.workload(name)
    S = w.seqlen
    with torch.cuda.stream(stream):
        t = W.make_tensors(S, w.hq, w.hkv, w.d, w.seed, device=str(dev), with_dout=w.backward)
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    fwd_ms, bwd_ms, plan_ms = [], [], []
    info = None
    for i in range(warmup + steps):
        with torch.cuda.stream(stream):
            flush.zero_()
        stream.synchronize()
        t0 = time.perf_counter()
        plan = ffa.Plan(w.slices, S, S, stream=stream)
        t1 = time.perf_counter()
        plan.enable_timing(True)
        out, lse = ffa.fwd(t["q"], t["k"], t["v"], plan, w.scale, stream=stream)
        if w.backward:
            ffa.bwd(t["q"], t["k"], t["v"], out, lse, t["dout"], plan, w.scale, stream=stream)
        plan.check_status(stream)
        tm = plan.read_timing()
        info = plan.info()
        plan.destroy()
        if i >= warmup:
            plan_ms.append(1e3 * (t1 - t0))
            fwd_ms.append(tm["fwd"][0])
            bwd_ms.append(tm["bwd_pre"][0] + tm["bwd_main"][0] + tm["bwd_dq"][0])
    area = info["mask_area"]
    fwd_f = 4.0 * area * w.hq * w.d
    r = {"seqlen": S, "hq": w.hq, "hkv": w.hkv, "d": w.d, "mask_area": area, "steps": steps,
         "fwd_ms": statistics.median(fwd_ms), "plan_ms": statistics.median(plan_ms),
         "l2": "flushed before every step (256 MiB write)"}
    r["fwd_tflops"] = fwd_f / (r["fwd_ms"] / 1e3) / 1e12
    r["fwd_frac_measured_burst"] = r["fwd_tflops"] / peaks["bf16_tflops"]
    r["fwd_frac_nominal_2p5"] = r["fwd_tflops"] / NOMINAL_BF16_TFLOPS
    if w.backward:
        r["bwd_ms"] = statistics.median(bwd_ms)
        r["bwd_tflops"] = 2.5 * fwd_f / (r["bwd_ms"] / 1e3) / 1e12
        r["bwd_frac_measured_burst"] = r["bwd_tflops"] / peaks["bf16_tflops"]
        r["bwd_frac_nominal_2p5"] = r["bwd_tflops"] / NOMINAL_BF16_TFLOPS
    r["secondary"] = secondary_bounds(info, w.hq, w.d)
    r["planner"] = planner_throughput(info, r["plan_ms"], peaks["hbm_gbs"])
    # one traced launch of each persistent kernel
    plan = ffa.Plan(w.slices, S, S, stream=stream)
    plan.enable_cta_trace(True)
    out, lse = ffa.fwd(t["q"], t["k"], t["v"], plan, w.scale, stream=stream)
    if w.backward:
        ffa.bwd(t["q"], t["k"], t["v"], out, lse, t["dout"], plan, w.scale, stream=stream)
    plan.check_status(stream)
    r["cta_balance"] = {"fwd": cta_balance(plan.read_cta_trace("fwd", stream))}
    if w.backward:
        r["cta_balance"]["bwd_main"] = cta_balance(plan.read_cta_trace("bwd_main", stream))
    plan.destroy()
    del t, flush
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return r


def gpu_arm(args, rank, world, local):
    import numpy as np
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import flexible_mask_flashattention_gb300 as ffa
    import workloads as W

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = W.workload(args.workload)
    S = w.seqlen
    peaks = load_peaks()
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        t = W.make_tensors(S, w.hq, w.hkv, w.d, w.seed, device=str(dev), with_dout=True)
        q, k, v, dout = t["q"], t["k"], t["v"], t["dout"]
        out = torch.empty_like(q)
        lse = torch.empty((w.hq, S), dtype=torch.float32, device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(ffa.bwd_workspace_size(S, S, w.hq, w.hkv, w.d), dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()

    def step_on(b, plans, before_fwd=None, after_fwd=None, before_bwd=None):
        # The hooks let the end-to-end pipeline start the forward once q, k, v are in (dout may still
        # be arriving) and copy out and lse out while the backward runs.
        plan = ffa.Plan(w.slices, S, S, stream=stream)
        plan.enable_timing(True)
        if before_fwd:
            before_fwd()
        ffa.fwd(b["q"], b["k"], b["v"], plan, w.scale, out=b["out"], lse=b["lse"], stream=stream)
        if after_fwd:
            after_fwd()
        if before_bwd:
            before_bwd()
        ffa.bwd(b["q"], b["k"], b["v"], b["out"], b["lse"], b["dout"], plan, w.scale, dq=b["dq"], dk=b["dk"],
                dv=b["dv"], workspace=ws, stream=stream)
        plans.append(plan)

    bufs0 = {"q": q, "k": k, "v": v, "dout": dout, "out": out, "lse": lse, "dq": dq, "dk": dk, "dv": dv}

    def step(plans):
        step_on(bufs0, plans)

    # warm-up
    for _ in range(args.warmup):
        warm = []
        step(warm)
        warm[-1].check_status(stream)
    info = warm[-1].info() if args.warmup else ffa.Plan(w.slices, S, S, stream=stream).info()
    area = info["mask_area"]
    fwd_f = 4.0 * area * w.hq * w.d
    bwd_f = 2.5 * fwd_f
    torch.cuda.synchronize()

    # timed region
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    plans = []
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step(plans)
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    ms = ev0.elapsed_time(ev1)
    ms = max_over_ranks(ms, world)
    for p in plans:
        p.check_status(stream)
    tk = {"fwd": [0.0, 0], "bwd_pre": [0.0, 0], "bwd_main": [0.0, 0], "bwd_dq": [0.0, 0]}
    launches = 0   # this library's kernels in the timed region: the planner's, fwd's and bwd's
    for p in plans:
        launches += p.info()["plan_launches"]
        for kname, (kms, n) in p.read_timing().items():
            tk[kname][0] += kms
            tk[kname][1] += n
            launches += n
    for p in plans:
        p.destroy()
    ms_step = ms / args.steps
    value = world * args.steps * (fwd_f + bwd_f) / (ms / 1e3) / 1e12
    fwd_ms = tk["fwd"][0] / max(tk["fwd"][1], 1)
    bwd_ms = sum(tk[x][0] for x in ("bwd_pre", "bwd_main", "bwd_dq")) / max(tk["bwd_main"][1], 1)
    main_ms = tk["bwd_main"][0] / max(tk["bwd_main"][1], 1)
    plan_ms = ms_step - fwd_ms - bwd_ms   # plan creation and the calls' host work: all but the kernels
    # plan creation alone, on an idle stream (it waits for its own GPU work, which inside the
    # timed steps includes the previous step's kernels): host wall time, median of 5
    plan_wall = []
    for _ in range(5):
        stream.synchronize()
        t0 = time.perf_counter()
        pw = ffa.Plan(w.slices, S, S, stream=stream)
        plan_wall.append(1e3 * (time.perf_counter() - t0))
        pw.destroy()
    plan_wall_ms = statistics.median(plan_wall)
    if args.only_step:
        # the timed steps alone (for profiling captures): no end-to-end, next-row, trace or side runs
        if rank == 0:
            achieved = bwd_f / (main_ms / 1e3) / 1e12
            print(json.dumps({"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
                              "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
                              "only_step": True, "config": {"workload": w.name, "mask_area": area},
                              "fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "bwd_main_ms": main_ms, "plan_ms": plan_ms,
                              "plan_wall_ms": plan_wall_ms,
                              "roofline": {"kernel": "ffa_bwd_main_kernel", "achieved": achieved,
                                           "peak": peaks["bf16_tflops_sustained"],
                                           "frac": achieved / peaks["bf16_tflops_sustained"]},
                              "gpu_launches": launches, "clocks": clocks}), flush=True)
        return 0

    # end to end through the public API with host buffers.  Every step copies its inputs (q, k, v,
    # dout) from pinned host memory and its results (out, lse, dq, dk, dv) back.  Two measurements:
    # "serial", all of it on the compute stream one step after the other; and the reported one, where
    # the copies run on their own streams into a second set of device tensors, so that step i+1's
    # inputs go in and step i-1's results come out while step i computes (pipeline_order).
    IN, OUT = ("q", "k", "v", "dout"), ("out", "lse", "dq", "dk", "dv")
    h = {n: bufs0[n].cpu().pin_memory() for n in IN}
    ho = {n: torch.empty(bufs0[n].shape, dtype=bufs0[n].dtype, pin_memory=True) for n in OUT}
    h2d = sum(x.numel() * x.element_size() for x in h.values())
    d2h = sum(x.numel() * x.element_size() for x in ho.values())
    with torch.cuda.stream(stream):
        bufs1 = {n: torch.empty_like(x) for n, x in bufs0.items()}
    sets = (bufs0, bufs1)
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def e2e_serial(keep):
        with torch.cuda.stream(stream):
            for n in IN:
                bufs0[n].copy_(h[n], non_blocking=True)
        step(keep)
        with torch.cuda.stream(stream):
            for n in OUT:
                ho[n].copy_(bufs0[n], non_blocking=True)

    FWD_IN, FWD_OUT = ("q", "k", "v"), ("out", "lse")

    def e2e_pipelined(keep, steps):
        # Per step and buffer set: q, k, v go in first and dout after them, so the forward starts
        # before dout has arrived; out and lse go out as soon as the forward is done, dq, dk, dv
        # after the backward.  Only the first step's q, k, v and the last step's dq, dk, dv are not
        # hidden behind compute.
        ev = {key: [torch.cuda.Event() for _ in range(2)] for key in ("qkv", "in", "fwd", "comp", "out")}
        for op, i in pipeline_order(steps):
            b = i % 2
            if op == "h2d":
                if i >= 2:
                    s_in.wait_event(ev["comp"][b])       # step i-2 has finished reading this set's inputs
                with torch.cuda.stream(s_in):
                    for n in FWD_IN:
                        sets[b][n].copy_(h[n], non_blocking=True)
                    ev["qkv"][b].record(s_in)
                    sets[b]["dout"].copy_(h["dout"], non_blocking=True)
                ev["in"][b].record(s_in)
            elif op == "compute":
                def wait_fwd_in(b=b, i=i):
                    # after the plan is built (building it waits for the stream)
                    if i >= 2:
                        stream.wait_event(ev["out"][b])  # step i-2's results have left this set
                    stream.wait_event(ev["qkv"][b])

                def copy_fwd_out(b=b):
                    ev["fwd"][b].record(stream)
                    s_out.wait_event(ev["fwd"][b])
                    with torch.cuda.stream(s_out):
                        for n in FWD_OUT:
                            ho[n].copy_(sets[b][n], non_blocking=True)

                step_on(sets[b], keep, before_fwd=wait_fwd_in, after_fwd=copy_fwd_out,
                        before_bwd=lambda b=b: stream.wait_event(ev["in"][b]))
                ev["comp"][b].record(stream)
            else:
                s_out.wait_event(ev["comp"][b])
                with torch.cuda.stream(s_out):
                    for n in OUT:
                        if n not in FWD_OUT:
                            ho[n].copy_(sets[b][n], non_blocking=True)
                ev["out"][b].record(s_out)

    def timed_e2e(run, warm, first, last):
        keep = []
        warm(keep)
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(first)
        run(keep)
        e1.record(last)
        torch.cuda.synchronize()
        barrier(world)
        ms = max_over_ranks(e0.elapsed_time(e1), world)
        for p in keep:
            p.destroy()
        return ms

    serial_ms = timed_e2e(lambda keep: [e2e_serial(keep) for _ in range(args.steps)], e2e_serial, stream, stream)
    e2e_ms = timed_e2e(lambda keep: e2e_pipelined(keep, args.steps), lambda keep: e2e_pipelined(keep, 2),
                       s_in, s_out)
    del bufs1, sets
    e2e_value = world * args.steps * (fwd_f + bwd_f) / (e2e_ms / 1e3) / 1e12
    # host link rate seen by the serial run: its copies' share of the step, over the bytes moved
    copy_s = (serial_ms - ms_step * args.steps) / 1e3
    copy_gbs = args.steps * (h2d + d2h) / copy_s / 1e9 if copy_s > 0 else None
    serial_value = world * args.steps * (fwd_f + bwd_f) / (serial_ms / 1e3) / 1e12

    # The LSE merge of partial results: ffa_lse_combine on this workload's (out, lse) against a second
    # partial (HBM-bound: it reads two outs and two lses and writes one of each), and ffa_fwd_accumulate
    # against the plain forward on the same plan.
    merge = {}
    with torch.cuda.stream(stream):
        out_b, lse_b = out.clone(), lse.clone() - 0.5
        out_m, lse_m = torch.empty_like(out), torch.empty_like(lse)
        for _ in range(3):
            ffa.lse_combine(out, lse, out_b, lse_b, out=out_m, lse=lse_m, stream=stream)
    torch.cuda.synchronize()
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_comb = 10
    c0.record(stream)
    for _ in range(n_comb):
        ffa.lse_combine(out, lse, out_b, lse_b, out=out_m, lse=lse_m, stream=stream)
    c1.record(stream)
    torch.cuda.synchronize()
    comb_ms = c0.elapsed_time(c1) / n_comb
    comb_bytes = 3 * (out.numel() * out.element_size() + lse.numel() * lse.element_size())
    merge["lse_combine"] = {"ms": comb_ms, "bytes": comb_bytes, "gbs": comb_bytes / comb_ms / 1e6,
                            "frac_of_hbm": comb_bytes / comb_ms / 1e6 / peaks["hbm_gbs"], "bound": "hbm"}
    acc_plan = ffa.Plan(w.slices, S, S, stream=stream)
    acc_plan.enable_timing(True)
    ffa.fwd_accumulate(q, k, v, acc_plan, w.scale, out_m, lse_m, stream=stream)
    acc_plan.check_status(stream)
    acc_ms = acc_plan.read_timing()["fwd"][0]
    acc_plan.destroy()
    merge["fwd_accumulate"] = {"ms": acc_ms, "fwd_ms": fwd_ms, "overhead": acc_ms / fwd_ms - 1.0}
    # The attention sink: ffa_fwd_sink / ffa_bwd_sink once each on the same workload (the backward's
    # preprocess time includes the per-head sink-gradient reduction).
    sink = torch.linspace(-2.0, 2.0, w.hq, device=dev, dtype=torch.float32)
    s_plan = ffa.Plan(w.slices, S, S, stream=stream)
    s_plan.enable_timing(True)
    ffa.fwd_sink(q, k, v, s_plan, w.scale, sink, out=out_m, lse=lse_m, stream=stream)
    dsink = torch.empty_like(sink)
    torch.cuda.synchronize()
    rc = ffa.load_library().ffa_bwd_sink(q.data_ptr(), k.data_ptr(), v.data_ptr(), out_m.data_ptr(), lse_m.data_ptr(),
                                         dout.data_ptr(), S, S, w.hq, w.hkv, w.d, s_plan.handle, float(w.scale),
                                         sink.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                         dsink.data_ptr(), ws.data_ptr(), ws.numel(), stream.cuda_stream)
    if rc != 0:
        raise RuntimeError(f"ffa_bwd_sink failed with status {rc}")
    s_plan.check_status(stream)
    st = s_plan.read_timing()
    s_plan.destroy()
    merge["sink"] = {"fwd_ms": st["fwd"][0], "fwd_plain_ms": fwd_ms,
                     "bwd_ms": st["bwd_pre"][0] + st["bwd_main"][0] + st["bwd_dq"][0], "bwd_plain_ms": bwd_ms,
                     "pre_ms": st["bwd_pre"][0], "pre_plain_ms": tk["bwd_pre"][0] / max(tk["bwd_pre"][1], 1)}
    del out_b, lse_b, out_m, lse_m
    # Range-Gather / Range-Scatter-Reduce (HBM-bound): half of k's rows in 64 ranges gathered; fp32
    # rows of the same shape scatter-reduced into disjoint ranges and, atomically, into overlapping ones.
    rng = np.random.default_rng(1)
    cuts = np.sort(rng.choice(np.arange(1, S), 127, replace=False))
    edges = np.concatenate([[0], cuts, [S]])
    rg = [(int(edges[2 * i]), int(edges[2 * i + 1])) for i in range(64)]
    g_rows = sum(e - s for s, e in rg)
    ov = [(int(s), int(min(S, s + (e - s) * 2))) for s, e in rg]   # each range doubled: neighbours overlap
    o_rows = sum(e - s for s, e in ov)

    def timed(fn, reps=5):
        fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    with torch.cuda.stream(stream):
        gbuf = torch.empty((g_rows,) + tuple(k.shape[1:]), dtype=k.dtype, device=dev)
        acc = torch.zeros(k.shape, dtype=torch.float32, device=dev)
        sbuf = torch.ones((g_rows,) + tuple(k.shape[1:]), dtype=torch.float32, device=dev)
        obuf = torch.ones((o_rows,) + tuple(k.shape[1:]), dtype=torch.float32, device=dev)
    row_b, row_f = k[0].numel() * 2, k[0].numel() * 4
    g_ms = timed(lambda: ffa.range_gather(k, rg, out=gbuf, stream=stream))
    s_ms = timed(lambda: ffa.range_scatter_reduce(sbuf, rg, acc, stream=stream))
    o_ms = timed(lambda: ffa.range_scatter_reduce(obuf, ov, acc, stream=stream))
    hbm = peaks["hbm_gbs"]
    merge["range"] = {
        "gather": {"ms": g_ms, "bytes": 2 * g_rows * row_b, "gbs": 2 * g_rows * row_b / g_ms / 1e6,
                   "frac_of_hbm": 2 * g_rows * row_b / g_ms / 1e6 / hbm},
        "scatter_reduce": {"ms": s_ms, "bytes": 3 * g_rows * row_f, "gbs": 3 * g_rows * row_f / s_ms / 1e6,
                           "frac_of_hbm": 3 * g_rows * row_f / s_ms / 1e6 / hbm},
        "scatter_reduce_overlapping": {"ms": o_ms, "bytes": 3 * o_rows * row_f,
                                       "gbs": 3 * o_rows * row_f / o_ms / 1e6,
                                       "frac_of_hbm": 3 * o_rows * row_f / o_ms / 1e6 / hbm},
        "rows": g_rows, "row_bytes_bf16": row_b}
    del gbuf, acc, sbuf, obuf
    # The dispatch solver (host code): the workload's query chunks onto 8 context-parallel buckets.
    # Balance = largest bucket area / mean, against the plain contiguous split of the chunks.
    chunk, cp = 4096, 8
    if S % (chunk * cp) == 0:
        t0 = time.perf_counter()
        bucket, carea, barea = ffa.dispatch_solve(w.slices, S, S, chunk, cp)
        solve_ms = 1e3 * (time.perf_counter() - t0)
        naive = carea.reshape(cp, -1).sum(axis=1)
        merge["dispatch"] = {"ms": solve_ms, "chunks": int(carea.size), "cp_size": cp, "chunk_size": chunk,
                             "max_over_mean": float(barea.max() / max(barea.mean(), 1)),
                             "contiguous_max_over_mean": float(naive.max() / max(naive.mean(), 1))}

    # Secondary bounds of the headline workload: executed against mask-area MMA work, the planner's
    # bytes over its time, and how evenly one traced launch of each persistent kernel loaded the SMs.
    secondary = secondary_bounds(info, w.hq, w.d)
    planner = planner_throughput(info, plan_wall_ms or plan_ms, peaks["hbm_gbs"])
    tr_plan = ffa.Plan(w.slices, S, S, stream=stream)
    tr_plan.enable_cta_trace(True)
    ffa.fwd(q, k, v, tr_plan, w.scale, out=out, lse=lse, stream=stream)
    ffa.bwd(q, k, v, out, lse, dout, tr_plan, w.scale, dq=dq, dk=dk, dv=dv, workspace=ws, stream=stream)
    tr_plan.check_status(stream)
    balance = {"fwd": cta_balance(tr_plan.read_cta_trace("fwd", stream)),
               "bwd_main": cta_balance(tr_plan.read_cta_trace("bwd_main", stream)),
               "deal": "each CTA pops the next unit of the longest-work-first order from one atomic counter"}
    tr_plan.destroy()
    side = {}
    if not args.no_side_configs:
        for name in SIDE_CONFIGS:
            side[name] = measure_side_config(ffa, W, name, stream, dev, peaks)

    if rank != 0:
        return 0
    # the timing rule between steps: inputs larger than L2 (129 MB on GB300), or else say so
    in_bytes = sum(x.numel() * x.element_size() for x in (q, k, v, dout))
    l2_note = ("inputs larger than L2, no flush" if in_bytes > 129 * 2 ** 20 else
               f"inputs ({in_bytes / 2 ** 20:.1f} MiB) smaller than L2, not flushed: L2-resident timing")
    peak = peaks["bf16_tflops_sustained"]
    achieved = bwd_f / (main_ms / 1e3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "seqlen": S, "hq": w.hq, "hkv": w.hkv, "d": w.d, "docs": len(w.slices),
                   "mask_area": area, "step": "ffa_plan + ffa_fwd + ffa_bwd",
                   "l2": l2_note, "parallelism": f"replicas x{world}"},
        "fwd_tflops": fwd_f / (fwd_ms / 1e3) / 1e12, "bwd_tflops": bwd_f / (bwd_ms / 1e3) / 1e12,
        "fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "plan_ms": plan_ms, "plan_wall_ms": plan_wall_ms,
        "frac_of_peak": {"fwd": fwd_f / (fwd_ms / 1e3) / 1e12 / peaks["bf16_tflops"],
                         "bwd": bwd_f / (bwd_ms / 1e3) / 1e12 / peaks["bf16_tflops"],
                         "step": value / world / peaks["bf16_tflops"],
                         "peak_tflops": peaks["bf16_tflops"], "peak": peaks["source"] + " burst bf16"},
        "frac_of_nominal_2p5": {"fwd": fwd_f / (fwd_ms / 1e3) / 1e12 / NOMINAL_BF16_TFLOPS,
                                "bwd": bwd_f / (bwd_ms / 1e3) / 1e12 / NOMINAL_BF16_TFLOPS,
                                "step": value / world / NOMINAL_BF16_TFLOPS, "peak_tflops": NOMINAL_BF16_TFLOPS},
        "secondary": secondary,
        "wasted_mma_frac": secondary["wasted_mma_frac"],
        "planner": planner,
        "planner_gbs": planner["gbs"],
        "cta_balance": balance,
        "configs": side,
        "roofline": {"kernel": "ffa_bwd_main_kernel", "bound": "tensor", "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak, "traffic": recorded_traffic(w.name),
                     "peak_kind": peaks["source"] + " sustained bf16"},
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "copies": "own streams, double-buffered device tensors; q, k, v go in ahead of dout and out, "
                          "lse come out after the forward, so the copies overlap the neighbouring steps' and "
                          "the other pass's compute", "serial_value": serial_value,
                "copy_gbs_serial": copy_gbs},
        "gpu_launches": launches,
        "clocks": clocks,
        "next_rows": merge,
    }

    if not args.no_cpu_baseline:
        flops, secs, desc = run_oracle_sample(w)
        line["cpu_baseline"] = {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(),
                                "kind": "oracle", "sample": desc}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="varlen_causal_1m")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-side-configs", action="store_true", help="skip the four smaller configurations")
    ap.add_argument("--only-step", action="store_true",
                    help="time the step alone and print a short line (for profiling captures)")
    args = ap.parse_args()
    rank, world, local = dist_setup(args.gpus)
    try:
        if args.impl == "reference":
            return reference_arm(args, rank, world)
        return gpu_arm(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
