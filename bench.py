"""Throughput of the CA-SGD outer iteration on GB300 (samples/s), with rooflines.

A step is one training pass of the workload: `iters` CA-SGD outer iterations
(sample+gather, Gram, recurrence, update) followed by one full-data loss evaluation,
all in the kernels of libcasgd.so.  Default workload: logistic regression on a dense
400,000 x 2,000 BF16 matrix (N(0,1)/sqrt(2000) entries, planted weights, 5% label
flips), b=256, s=32 (Gram 8192 x 8192), eta=0.5, 50 outer iterations per step, seed 0,
synthetic (the epsilon data set it stands in for is not available).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--config 1..5] [--s S] [--sharded]
N > 1 runs under torchrun, one process per GPU: independent replicas (one GPU's
problem per rank, no collective on the data path); value = samples of all ranks / max
time.  `--sharded` instead splits one problem's features over the ranks, with one FP32
all-reduce (NCCL) of the Gram matrix and the margins per outer iteration.  `--impl reference` times the CPU oracle (the plain NumPy statement of the
method) on the host cores, on a bounded sample of the same workload.

`value` comes from K steps called as a user calls them; a second pass of K steps with
CUDA events between the launches gives the per-stage times and the roofline (the
events themselves cost stream time, so that pass is reported apart).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth_inputs as si  # noqa: E402

METRIC = "SGD samples/s per GB300 (CA-SGD); Gram TFLOP/s and % of roofline"
STAGES = ("gather", "gram", "recurrence", "update")
KERNEL_SOURCES = {"gram_tc": ("k_gram_tc.cu",), "gram_simt": ("k_gram_simt.cu",),
                  "gram_recur": ("k_gram_tc.cu", "recur_roles.cuh"),
                  "gram_recur_far": ("k_gram_tc.cu", "recur_roles.cuh"),
                  "recurrence": ("k_recur.cu", "recur_roles.cuh"), "update": ("k_update.cu",),
                  "gather": ("k_prep.cu",)}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=2)
    ap.add_argument("--s", type=int, default=None, help="override s (recipe 4 sweep)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sgd", action="store_true",
                    help="skip the FP32 plain SGD comparison leg")
    ap.add_argument("--m", type=int, default=None,
                    help="override the row count (small profiling captures only)")
    ap.add_argument("--sharded", action="store_true",
                    help="the paper's feature-sharded setting: each rank holds a slice of the "
                         "columns, one FP32 all-reduce of G and the margins per outer iteration "
                         "(torch.distributed, NCCL); strong scaling (one problem)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads' lines (recipes 3, 4 with s = 4..32, 5)")
    ap.add_argument("--config-steps", type=int, default=3,
                    help="timed steps of each other workload (after 1 warm-up step)")
    ap.add_argument("--flags", type=lambda v: int(v, 0), default=0,
                    help="casgd_params_t.flags for profiling variants (e.g. 0x40: Gram and "
                         "recurrence in separate launches)")
    return ap.parse_args()


def workload(cfg: int, s_override, m_override=None):
    r = si.RECIPES[cfg]
    s = s_override or r.s
    iters = r.outer_iters(m=m_override, s=s)
    return r, s, iters


def workload_config(r, s, iters, S, m=None):
    m = r.m if m is None else m
    return {"workload": f"{si.LOSS_NAMES[r.loss]} CA-SGD, dense X {m}x{r.n} BF16, "
                        f"b={r.b}, s={s} (Gram {S}x{S}), eta={r.eta}, {iters} outer iterations "
                        f"+ 1 full-data loss per step, seed 0",
            "m": m, "n": r.n, "b": r.b, "s": s, "S": S, "outer_iters_per_step": iters,
            "loss": si.LOSS_NAMES[r.loss],
            "l2_policy": f"inputs larger than L2: X is {m * ((r.n + 7) // 8 * 8) * 2 / 1e9:.2f} GB "
                         "and each outer iteration gathers fresh random rows"}


def alg_work(n, S, s, b, m):
    """Algorithmic flops/bytes per outer iteration, per stage (strictly block-lower G)."""
    frac = 1.0 - 1.0 / s
    g_bytes = 2.0 * S * S * frac          # 4 bytes x S^2 (1-1/s) / 2 entries
    return {
        "gather": {"bytes": 2.0 * S * n * 2 + 4 * S + 2 * S + 4 * S, "flops": 2.0 * S * n},
        "gram": {"flops": float(n) * S * S * frac, "bytes": 2.0 * S * n + g_bytes},
        "recurrence": {"bytes": g_bytes + 10.0 * S, "flops": 2.0 * S * S * frac / 2},
        "update": {"bytes": 2.0 * S * n + 4.0 * S + 8.0 * n, "flops": 2.0 * S * n},
        "loss": {"bytes": 2.0 * m * ((n + 7) // 8 * 8) + 4.0 * m, "flops": 2.0 * m * n},
    }


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def tensor_peak(pk: dict, clk: dict):
    """The dense BF16 peak a kernel timed in this run is held to: the burst figure,
    unless the clock record of the timed region shows the power cap or an SM clock well
    below its maximum (then the seconds-long sustained figure).  Returns (peak, which)."""
    reasons = clk.get("reasons") or []
    sm, mx = clk.get("sm_mhz"), clk.get("sm_max_mhz")
    low = sm is not None and mx is not None and sm < 0.9 * mx
    if "sw_power_cap" in reasons or low:
        why = "sw_power_cap active" if "sw_power_cap" in reasons else f"SM clock {sm:.0f} of {mx:.0f} MHz"
        return pk["bf16_tflops_sustained"], f"sustained ({why} in the timed region)"
    return pk["bf16_tflops"], ("burst (timed region at full SM clock, no power cap)"
                               if sm is not None else "burst (clocks not sampled)")


def source_hash(kernel: str) -> str:
    """First 16 hex digits of the SHA-256 of the kernel's source files, concatenated."""
    hs = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        hs.update(open(os.path.join(ROOT, "communication_avoiding_step_gb300", "csrc", f),
                       "rb").read())
    return hs.hexdigest()[:16]


def traffic_for(kernel: str, cfg: int):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    d = json.load(open(path)).get(f"{kernel}@config{cfg}")
    if not d:
        return None
    h = source_hash(kernel)
    return d["bytes_per_launch"] if d.get("source_sha256_16") == h else None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            # the sampler is live (first line read) before the timed region starts
            t_end = time.time() + 3.0
            while not self.lines and time.time() < t_end:
                time.sleep(0.01)
            self.lines.clear()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def world_max(value: float, device) -> float:
    """Max of a per-rank value over the process group (identity without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------- CPU side ----
def cpu_sample(cfg, s, budget_s=15.0, max_iters=50):
    """Times the oracle's emulating-mode outer iteration on this host (bounded sample:
    up to one step's 50 outer iterations, stopping once budget_s seconds are spent)."""
    import oracle
    r = si.RECIPES[cfg]
    p = si.make_problem(cfg)
    S = r.b * s
    w = np.zeros(r.n, np.float32)
    done, t_total = 0, 0.0
    while done < max_iters and (t_total < budget_s or done == 0):
        t0 = time.perf_counter()
        w = oracle.outer_step(p.X, p.y, w, r.b, s, r.eta, r.loss, 0, done, mode="emulate")
        t_total += time.perf_counter() - t0
        done += 1
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": S * done / t_total, "unit": "samples/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} outer iteration(s) of the same workload (S={S}) in the oracle's "
                      f"emulating mode (NumPy, BLAS on all host cores), {t_total:.2f} s"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    r, s, iters = workload(args.config, args.s)
    S = r.b * s
    import oracle
    p = si.make_problem(args.config)
    w = np.zeros(r.n, np.float32)
    k = 0
    for _ in range(args.warmup):
        w = oracle.outer_step(p.X, p.y, w, r.b, s, r.eta, r.loss, 0, k, mode="emulate")
        k += 1
    t0 = time.perf_counter()
    for _ in range(args.steps):
        w = oracle.outer_step(p.X, p.y, w, r.b, s, r.eta, r.loss, 0, k, mode="emulate")
        k += 1
    dt = time.perf_counter() - t0
    value = S * args.steps / dt
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    cfgd = workload_config(r, s, iters, S)
    cfgd["reference_step"] = "one outer iteration (bounded sample of the workload)"
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": "samples/s",
           "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": cfgd,
           "cpu_baseline": {"value": value, "unit": "samples/s", "cores": cores, "kind": "oracle",
                            "sample": f"{args.steps} timed outer iterations, emulating mode"},
           "e2e": {"value": value, "unit": "samples/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


# --------------------------------------------------------------------- GPU side ----
GRAM_NAMES = {1: "gram_tc", 2: "gram_simt", 3: "gram_recur", 4: "gram_recur",
              5: "gram_recur_far", 6: "gram_recur_far"}


def stage_times(torch, casgd, data, params, ws, w, iters, steps, k, stream):
    """Per-launch stage times (ms) from `steps` steps with CUDA events between the
    launches; returns (stage_ms_per_launch, total_ms, k, last loss history)."""
    n_ev = iters * casgd.STAGE_EVENTS
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(steps)]
    for row in events:        # torch creates the CUDA event lazily, on first record
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    s0 = torch.cuda.Event(enable_timing=True)
    s1 = torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    hist = None
    for i in range(steps):
        w.zero_()
        hist, _, _ = casgd.train(data, params, w, iters, ws, k0=k, loss_every=iters,
                                 stage_events=events[i])
        k += iters
    s1.record(stream)
    torch.cuda.synchronize()
    stage_ms = {st: 0.0 for st in STAGES}
    for i in range(steps):
        ev = events[i]
        for it in range(iters):
            b0 = it * casgd.STAGE_EVENTS
            for si_, st in enumerate(STAGES):
                stage_ms[st] += ev[b0 + si_].elapsed_time(ev[b0 + si_ + 1])
    per_launch = {st: stage_ms[st] / (steps * iters) for st in STAGES}
    return per_launch, s0.elapsed_time(s1), sum(stage_ms.values()), k, hist


def chain_phase_floor(torch, casgd, data, params, k):
    """The fastest phase of the recurrence's chain in one traced outer iteration (ns
    between alpha_{j-1} and alpha_j stored, j >= 1), or None."""
    import dataclasses
    pt = dataclasses.replace(params, flags=params.flags | casgd.FLAG_TRACE_CHAIN)
    ws = casgd.workspace(data, pt)
    w = torch.zeros(data.n, device="cuda")
    casgd.train(data, pt, w, 2, ws, k0=k)
    tr = casgd.chain_trace(data, pt, ws)
    st = [row[3] for row in tr[:params.s]]
    d = [b - a for a, b in zip(st[:-1], st[1:]) if a and b and b > a]
    del ws
    return min(d) if d else None


def extra_configs(args, torch, casgd, rank, pk):
    """The other workloads of the method (recipes 3, 4 at s = 4, 8, 16, 32, and 5): one
    warm-up and `config_steps` timed steps each, as a user calls them, then as many steps
    with events between the launches for the dominant launch's time."""
    out = {}
    pl = [(3, None), (4, 4), (4, 8), (4, 16), (4, 32), (5, None)]
    stream = torch.cuda.current_stream()
    for cfg, s_ov in pl:
        r, s, iters = workload(cfg, s_ov)
        S = r.b * s
        p = si.make_problem(cfg)
        X32 = torch.from_numpy(p.X).cuda()
        y = torch.from_numpy(p.y).cuda()
        data = casgd.Dataset.from_fp32(X32, y)
        del X32
        params = casgd.Params(r.b, s, r.eta, r.loss, seed=rank)
        ws = casgd.workspace(data, params)
        w = torch.zeros(r.n, device="cuda")
        k = 0
        w.zero_()
        casgd.train(data, params, w, iters, ws, k0=k, loss_every=iters)
        k += iters
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        kind = None
        for _ in range(args.config_steps):
            w.zero_()
            hist, _, kind = casgd.train(data, params, w, iters, ws, k0=k, loss_every=iters)
            k += iters
        t1.record(stream)
        torch.cuda.synchronize()
        el = t0.elapsed_time(t1) / 1e3
        per_launch, _, _, k, _ = stage_times(torch, casgd, data, params, ws, w, iters,
                                             args.config_steps, k, stream)
        work = alg_work(r.n, S, s, r.b, p.m)
        t_g = per_launch["gram"] / 1e3
        name = GRAM_NAMES[kind]
        ent = {"workload": workload_config(r, s, iters, S)["workload"],
               "value": S * iters * args.config_steps / el, "unit": "samples/s",
               "ms_per_step": el * 1e3 / args.config_steps, "steps": args.config_steps,
               "dominant_kernel": name, "dominant_ms_per_launch": per_launch["gram"],
               "other_ms_per_iteration": {st: per_launch[st] for st in STAGES if st != "gram"},
               "final_loss": hist[0] if hist else None}
        tf = work["gram"]["flops"] / t_g / 1e12
        tb = work["gram"]["bytes"] / t_g / 1e9
        ent["tensor"] = {"achieved_TFLOP/s": tf, "frac": tf / pk["bf16_tflops"],
                         "peak": pk["bf16_tflops"], "peak_source": f"{pk['source']} bf16 burst"}
        ent["hbm_by_algorithmic_bytes"] = {
            "achieved_GB/s": tb, "frac": tb / pk["hbm_gbs"], "peak": pk["hbm_gbs"],
            "note": "bytes of the stored-G algorithm (Y read, G written); the far-forming "
                    "launch never moves G below the band, so this can exceed 1"}
        floor = chain_phase_floor(torch, casgd, data, params, k) if kind in (5, 6) else None
        if floor:
            t_lat = s * floor / 1e9
            ent["latency"] = {"bound": "chain", "phase_floor_us": floor / 1e3,
                              "bound_us": t_lat * 1e6, "frac": t_lat / t_g,
                              "note": "s phases x the fastest measured chain phase (alpha_j "
                                      "stored after alpha_{j-1}, one traced iteration)"}
        bound = "tensor" if ent["tensor"]["frac"] >= (ent.get("latency") or {}).get("frac", 0) \
            else "chain latency"
        ent["bound"] = bound
        out[f"config{cfg}" + (f"_s{s}" if cfg == 4 else "")] = ent
        del ws, data, w
        torch.cuda.empty_cache()
    return out


def run_sharded(args):
    """Feature-sharded CA-SGD over the ranks of a torchrun job (one rank: the exchange is
    the identity).  Every rank draws the same rows; rank q holds columns
    [q*n/N, (q+1)*n/N) of X and of w.  A step = `iters` outer iterations; value = the
    problem's samples per second (every rank works on the same samples)."""
    import torch
    import communication_avoiding_step_gb300 as casgd

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    casgd.load()
    r, s, iters = workload(args.config, args.s, args.m)
    S = r.b * s
    p = si.make_problem(args.config, m=args.m)
    c0, c1 = r.n * rank // world, r.n * (rank + 1) // world
    X32 = torch.from_numpy(np.ascontiguousarray(p.X[:, c0:c1])).cuda()
    data = casgd.Dataset.from_fp32(X32, torch.from_numpy(p.y).cuda())
    del X32
    params = casgd.Params(r.b, s, r.eta, r.loss, seed=0, flags=args.flags)
    ws = casgd.workspace_sharded(data, params)
    xbuf = casgd.exchange_buffer(params)
    w = torch.zeros(c1 - c0, device="cuda")
    all_reduce = dist.all_reduce if dist else None
    k = 0
    for _ in range(args.warmup):
        w.zero_()
        casgd.train_sharded(data, params, w, iters, ws, xbuf, all_reduce, k0=k)
        k += iters
    stream = torch.cuda.current_stream()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    launches = 0
    with ClockSampler(local) as clocks:
        t0.record(stream)
        for _ in range(args.steps):
            w.zero_()
            n_l, _ = casgd.train_sharded(data, params, w, iters, ws, xbuf, all_reduce, k0=k)
            launches += n_l
            k += iters
        t1.record(stream)
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    elapsed = world_max(t0.elapsed_time(t1) / 1e3, torch.device("cuda", local))
    if rank == 0:
        xb = xbuf.numel() * 4
        out = {"metric": METRIC, "value": S * iters * args.steps / elapsed, "unit": "samples/s",
               "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
               "ms_per_step": elapsed * 1e3 / args.steps, "higher_is_better": True,
               "scaling": "strong", "vs_baseline": None, "dtype": "bf16",
               "data": "synthetic",
               "config": dict(workload_config(r, s, iters, S, p.m),
                              sharded=f"features split over {world} rank(s); one FP32 "
                                      f"all-reduce of {xb / 1e6:.1f} MB per outer iteration"),
               "parallelism": f"feature-sharded x{world}", "gpu_launches": launches,
               "clocks": clocks.summary()}
        print(json.dumps(out), flush=True)
    if dist:
        dist.destroy_process_group()


def run_ours(args):
    import torch
    import communication_avoiding_step_gb300 as casgd

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    casgd.load()

    r, s, iters = workload(args.config, args.s, args.m)
    S = r.b * s
    p = si.make_problem(args.config, m=args.m)
    X32 = torch.from_numpy(p.X).cuda()
    y = torch.from_numpy(p.y).cuda()
    data = casgd.Dataset.from_fp32(X32, y)
    if args.no_sgd:
        del X32
    torch.cuda.synchronize()
    params = casgd.Params(r.b, s, r.eta, r.loss, seed=rank, flags=args.flags)
    ws = casgd.workspace(data, params)
    w = torch.zeros(r.n, device="cuda")
    stream = torch.cuda.current_stream()

    def step(k0, events=None):
        w.zero_()
        hist, launches, kind = casgd.train(data, params, w, iters, ws, k0=k0,
                                           loss_every=iters, stage_events=events)
        return hist, launches, kind

    k = 0
    for _ in range(args.warmup):
        step(k)
        k += iters
    n_ev = iters * casgd.STAGE_EVENTS
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
              for _ in range(args.steps)]
    for row in events:        # torch creates the CUDA event lazily, on first record
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    launches_total = 0
    # The timed region runs the K steps as a user calls them.  A second pass of K steps
    # then records CUDA events between the launches for the per-stage times and the
    # roofline: each event costs about 2 us of stream time and keeps consecutive launches
    # from overlapping, so those steps are timed separately (ms_per_step_stage_pass).
    with ClockSampler(local) as clocks:
        start.record(stream)
        for i in range(args.steps):
            hist, launches, kind = step(k)
            launches_total += launches
            k += iters
        end.record(stream)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        # A third pass times the dominant launch as it runs in the timed region: two
        # events per step only, before the launch of iteration 1 and after that of
        # iteration iters-2, so the launches between them follow one another as they
        # do without events (the period includes the short gap between two launches).
        period_ms = None
        if iters >= 4:
            n_between = iters - 2
            pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                     for _ in range(args.steps)]
            for a_, b_ in pairs:
                a_.record(stream)
                b_.record(stream)
            torch.cuda.synchronize()
            for i in range(args.steps):
                row = [None] * n_ev
                row[1 * casgd.STAGE_EVENTS + 1] = pairs[i][0]
                row[(iters - 2) * casgd.STAGE_EVENTS + 2] = pairs[i][1]
                step(k, row)
                k += iters
            torch.cuda.synchronize()
            period_ms = sum(a_.elapsed_time(b_) for a_, b_ in pairs) / (args.steps * n_between)
        s_start = torch.cuda.Event(enable_timing=True)
        s_end = torch.cuda.Event(enable_timing=True)
        s_start.record(stream)
        for i in range(args.steps):
            hist, _, _ = step(k, events[i])  # the final-loss comparison uses the last step
            k += iters
        s_end.record(stream)
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    elapsed = world_max(start.elapsed_time(end) / 1e3, torch.device("cuda", local))
    stage_pass = world_max(s_start.elapsed_time(s_end) / 1e3, torch.device("cuda", local))
    stage_ms = {st: 0.0 for st in STAGES}
    for i in range(args.steps):
        ev = events[i]
        for it in range(iters):
            b0 = it * casgd.STAGE_EVENTS
            for si_, st in enumerate(STAGES):
                stage_ms[st] += ev[b0 + si_].elapsed_time(ev[b0 + si_ + 1])
    per_launch_ms = {st: stage_ms[st] / (args.steps * iters) for st in STAGES}
    loss_ms = (stage_pass * 1e3 - sum(stage_ms.values())) / args.steps  # loss + host gaps

    samples = S * iters * args.steps * world
    value = samples / elapsed
    pk = peaks()
    work = alg_work(r.n, S, s, r.b, p.m)
    # kind 3/4/5/6: the Gram (4: of the next iteration; 5/6: forming the far sums), the
    # recurrence and the update share one launch (its time is the "gram" stage; the
    # "recurrence" and "update" stages then hold only the gaps between events); kind 6
    # also gathers the rows there, two iterations ahead, where the shapes allow (the
    # "gather" stage then holds the prologue's gathers spread over the step)
    gram_name = GRAM_NAMES[kind]
    fused_gather = kind == 6 and per_launch_ms["gather"] < 0.05 * per_launch_ms["gram"]
    stages_out = {}
    for st in STAGES:
        t = per_launch_ms[st] / 1e3
        ent = {"ms_per_launch": per_launch_ms[st],
               "GB/s": work[st]["bytes"] / t / 1e9 if t > 0 else None}
        if st == "gram":
            ent["TFLOP/s"] = work[st]["flops"] / t / 1e12 if t > 0 else None
            ent["kernel"] = gram_name
        elif (st in ("recurrence", "update") and kind in (3, 4, 5, 6)) or \
                (st == "gather" and fused_gather):
            ent["GB/s"] = None
            ent["note"] = "runs inside the shared launch (the gram stage)"
        stages_out[st] = ent
    dom = max(STAGES, key=lambda st: per_launch_ms[st])
    t_dom = per_launch_ms[dom] / 1e3
    dur_src = "stage pass: CUDA events around every launch (no overlap between launches)"
    if dom == "gram" and period_ms is not None and kind == 6:
        # one launch per outer iteration: the launch period of the steady state
        t_dom = period_ms / 1e3
        dur_src = ("launch period: CUDA events around launches 1 .. iters-2 of each step, "
                   "none between them (includes the gap between two launches)")
    if dom == "gram":
        achieved = work["gram"]["flops"] / t_dom / 1e12
        peak, which = tensor_peak(pk, clocks.summary())
        roof = {"kernel": gram_name, "bound": "tensor", "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_source": f"{pk['source']} bf16 dense, {which}",
                "traffic": traffic_for(gram_name, args.config)}
    else:
        achieved = work[dom]["bytes"] / t_dom / 1e9
        peak = pk["hbm_gbs"]
        roof = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peak,
                "unit": "GB/s", "frac": achieved / peak, "peak_source": f"{pk['source']} HBM copy",
                "traffic": traffic_for(dom, args.config)}
    roof["units_per_launch"] = "one outer iteration (S rows)"
    roof["duration_ms"] = t_dom * 1e3
    roof["duration_source"] = dur_src

    # ---- end to end: host buffers, copies inside the timed region ----------------
    # ---- FP32 plain minibatch SGD on the same rows (the paper's comparison) -----
    sgd = None
    if not args.no_sgd:
        sws = casgd.sgd_workspace(r.b)
        wsg = torch.zeros(r.n, device="cuda")
        sgd_params = casgd.Params(r.b, 1, r.eta, r.loss, seed=rank)
        nsteps = iters * s  # one CA-SGD step's minibatches
        casgd.sgd_fp32(X32, y, sgd_params, wsg, nsteps, sws, q0=0)  # warm-up
        torch.cuda.synchronize()
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for i in range(args.steps):
            wsg.zero_()
            casgd.sgd_fp32(X32, y, sgd_params, wsg, nsteps, sws, q0=(i + 1) * nsteps)
        s1.record(stream)
        torch.cuda.synchronize()
        sgd_elapsed = s0.elapsed_time(s1) / 1e3
        # final loss on the rows of the last timed CA-SGD step, from w = 0
        wsg.zero_()
        casgd.sgd_fp32(X32, y, sgd_params, wsg, nsteps, sws, q0=(k - iters) * s)
        f_sgd = casgd.loss(data, r.loss, wsg, ws)
        st = casgd.get_status(sws)
        value_sgd = S * iters * args.steps / sgd_elapsed
        f_ca = hist[0] if hist else None
        sgd = {"value": value_sgd, "unit": "samples/s",
               "kind": "FP32 plain minibatch SGD on FP32 X (casgd_sgd_fp32), the same rows",
               "steps_per_rep": nsteps, "ms_per_rep": sgd_elapsed * 1e3 / args.steps,
               "ca_sgd_over_sgd": value / value_sgd if value_sgd > 0 else None,
               "final_loss": f_sgd, "ca_sgd_final_loss": f_ca,
               "final_loss_gap": abs(f_ca - f_sgd) / f_sgd if f_ca is not None else None,
               "status": st}
        del X32

    e2e = None
    e2e_overlapped = None
    if not args.no_e2e:
        Xh = data.X.cpu().pin_memory()
        yh = data.y.cpu().pin_memory()
        wh = torch.zeros(r.n).pin_memory()
        e_steps = max(2, min(args.steps, 5))
        h2d = Xh.numel() * 2 + yh.numel() * 4 + wh.numel() * 4
        # (1) The C-ABI call with host buffers (casgd_train_host): per step it copies X, y
        # and w0 from pinned host memory into the device buffers, runs the step's
        # iterations and the loss, and copies w back to the host -- all inside the timed
        # region, one step after the other.
        Xd = torch.empty_like(data.X)
        yd = torch.empty_like(data.y)
        dset = casgd.Dataset(Xd, yd, r.n)
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(e_steps):
            wh.zero_()
            hist, _, _ = casgd.train_host(Xh, yh, wh, dset, w, params, iters, ws, k0=k,
                                          loss_every=iters)
            k += iters
        t1.record(stream)
        torch.cuda.synchronize()
        e_el = world_max(t0.elapsed_time(t1) / 1e3, torch.device("cuda", local))
        e2e = {"value": S * iters * e_steps * world / e_el, "unit": "samples/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": wh.numel() * 4 + 8,
               "steps": e_steps,
               "copies": "casgd_train_host (C ABI, host buffers): X, y, w0 copied in and w "
                         "copied back each step, steps one after the other"}
        # (2) The same through the binding with the copy of step i+1's X and y on a copy
        # stream into a second device buffer while step i computes.
        w_out = torch.empty(r.n).pin_memory()
        Xd2 = [Xd, torch.empty_like(data.X)]
        yd2 = [yd, torch.empty_like(data.y)]
        dsets = [casgd.Dataset(Xd2[i], yd2[i], r.n) for i in range(2)]
        copy_stream = torch.cuda.Stream()
        ready = [torch.cuda.Event() for _ in range(2)]
        wh.zero_()
        torch.cuda.synchronize()

        def copy_inputs(i):
            with torch.cuda.stream(copy_stream):
                Xd2[i].copy_(Xh, non_blocking=True)
                yd2[i].copy_(yh, non_blocking=True)
                ready[i].record(copy_stream)

        t0.record(stream)
        copy_stream.wait_event(t0)
        copy_inputs(0)
        for i in range(e_steps):
            cur = i % 2
            if i + 1 < e_steps:  # buffer 1-cur was last read by step i-1, which is done
                copy_inputs(1 - cur)
            stream.wait_event(ready[cur])
            w.copy_(wh, non_blocking=True)
            casgd.train(dsets[cur], params, w, iters, ws, k0=k, loss_every=iters)
            w_out.copy_(w, non_blocking=True)
            k += iters
        t1.record(stream)
        torch.cuda.synchronize()
        e_el2 = world_max(t0.elapsed_time(t1) / 1e3, torch.device("cuda", local))
        e2e_overlapped = {"value": S * iters * e_steps * world / e_el2, "unit": "samples/s",
                          "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": w_out.numel() * 4 + 8,
                          "steps": e_steps,
                          "copies": "through the binding: each step's X and y on a copy "
                                    "stream, overlapping the previous step's compute (two "
                                    "device buffers)"}
        del Xd, yd, Xd2, yd2, dset, dsets

    configs = None
    if not args.no_configs and args.m is None and args.flags == 0:
        del data, ws
        torch.cuda.empty_cache()
        configs = extra_configs(args, torch, casgd, rank, pk)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_sample(args.config, s)

    if rank == 0:
        out = {"metric": METRIC, "value": value, "unit": "samples/s", "n_gpus": world,
               "steps": args.steps, "warmup": args.warmup,
               "ms_per_step": elapsed * 1e3 / args.steps, "higher_is_better": True,
               "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
               "config": dict(workload_config(r, s, iters, S, p.m),
                              **({"flags": hex(args.flags)} if args.flags else {})),
               "parallelism": "replicas" if world > 1 else "single",
               "gpu_launches": launches_total,
               "roofline": roof, "stages": stages_out,
               "loss_and_gaps_ms_per_step": loss_ms,
               "ms_per_step_stage_pass": stage_pass * 1e3 / args.steps,
               "gram_tflops": stages_out["gram"]["TFLOP/s"],
               "final_loss": hist[0] if hist else None,
               "clocks": clocks.summary(), "e2e": e2e, "e2e_overlapped": e2e_overlapped,
               "cpu_baseline": cpu,
               "fp32_sgd": sgd, "configs": configs}
        print(json.dumps(out), flush=True)
    if dist:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.sharded:
        run_sharded(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
