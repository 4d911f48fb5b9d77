#!/usr/bin/env python
"""Benchmark of the fused TP-reduce + MoE finalize + residual + RMSNorm op.

One step = one call of the whole fused path (routed gather-sum, shared add,
rank sum, residual add, RMSNorm) on one batch of synthetic input.  The
headline workload is the bandwidth-bound prefill shape: R = 8 rank partials,
K = 10 routed experts per token, H = 8192, T = 8192 tokens per GPU (12.2 GB of
algorithmic traffic per call, far larger than the 129 MB L2, so no flush is
needed between calls).  Inputs are drawn on the device with a seeded
generator (gen.make_inputs); nothing is read from disk.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line (rank 0).  value = algorithmic bytes of all ranks / the
slowest rank's device time (GB/s); ms_per_step = device time per call.
Extra keys: roofline (dominant kernel against the measured HBM copy peak),
cpu_baseline (the CPU oracle on a bounded sample), e2e (same metric through
the public binding with pinned host buffers and the host<->device copies
inside the timed region), clocks (nvidia-smi during the timed region),
gpu_launches, and sweep (µs/call and GB/s vs T for every workload, L2-cold
by rotating inputs, timed by CUDA-graph replay).

--impl reference times the CPU oracle (the slow, plain fp64 restatement of
the method; no GPU) on a bounded sample of the same workload and prints the
same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "µs/call and achieved HBM GB/s (% of GB300 roofline) vs tokens T, 1 GPU"
UNIT = "GB/s"
HEADLINE = ("prefill", 8192)
FALLBACK_HBM_GBS = 6800.0
REGIMES = {"auto": 0, "cluster": 1, "stream": 2, "oneshot": 3, "split": 4}
REGIME_NAMES = {1: "cluster", 2: "stream", 3: "oneshot", 4: "split"}


def parse_regime(tok: str):
    """'auto' | 'cluster' | 'stream' | 'oneshot' | 'split' | 'c<N>' (cluster regime, N CTAs
    per row) | 's<N>' (split regime, N CTAs per row)."""
    if tok.startswith("c") and tok[1:].isdigit():
        return REGIMES["cluster"], int(tok[1:])
    if tok.startswith("s") and tok[1:].isdigit():
        return REGIMES["split"], int(tok[1:])
    return REGIMES[tok], 0
CPU_SAMPLE_T = 512
WARM_CALLS = 64  # calls per graph in the L2-warm sweep (all on the one input set)
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "stream_rows_prefill_traffic.json")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=500)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=HEADLINE[0],
                   choices=["tiny", "ar_only", "dsv3_decode", "glm_gemma", "prefill"],
                   help="shape of the timed call (the headline is prefill)")
    p.add_argument("--tokens", type=int, default=HEADLINE[1], help="T per GPU")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-sweep", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=16)
    p.add_argument("--e2e-streams", type=int, default=1,
                   help="streams the per-step host->device input copies are spread over")
    p.add_argument("--regime", default="auto",
                   help="force a kernel regime for the timed call: auto, cluster, stream, "
                        "oneshot or c<N> (cluster regime with N CTAs per row)")
    p.add_argument("--gated", action="store_true",
                   help="time the gated shared-expert variant (shared partials scaled by a "
                        "per-token sigmoid gate)")
    p.add_argument("--stage-bytes", type=int, default=0,
                   help="target ring-slot bytes of the streaming kernels (0 = automatic)")
    p.add_argument("--sweep-regimes", default="auto",
                   help="comma list of regimes timed in the sweep (same tokens as --regime)")
    p.add_argument("--sweep-only", default="",
                   help="comma list of workloads to sweep (default: all)")
    p.add_argument("--pdl", action="store_true",
                   help="headline and e2e workspaces launch with programmatic dependent launch")
    p.add_argument("--sweep-pdl", choices=["off", "on", "both"], default="both",
                   help="sweep points without / with programmatic dependent launch (AR_WS_PDL)")
    p.add_argument("--sweep-perm", choices=["random", "expert_sorted"], default="random",
                   help="routing permutation of the sweep's inputs: a random permutation of the "
                        "expert rows, or the expert-sorted order a real MoE dispatch produces")
    p.add_argument("--sweep-mode", choices=["rotate", "scatter", "warm"], default="rotate",
                   help="rotate: L2-cold, each call gathers within its own expert block; "
                        "scatter: L2-cold, gathers spread over all sets' rows; "
                        "warm: one input set replayed (L2-warm)")
    return p.parse_args()


def headline_config(name: str, T: int, world: int) -> dict:
    from gen import CONFIGS, problem_bytes
    cfg = CONFIGS[name]
    R, K, H = cfg.R, cfg.K, cfg.H
    b = problem_bytes(R, K, H, T)
    return {"workload": f"{name} R={R} K={K} H={H} T={T} per GPU, bf16 in/out, "
                        f"fp32 accumulate, residual_out bf16",
            "R": R, "K": K, "H": H, "T": T, "bytes_per_step_per_gpu": b,
            "l2": (f"inputs {b / 1e9:.3g} GB per call per GPU, larger than the 129 MB L2: no flush"
                   if b > 3 * 129e6 else f"inputs {b / 1e6:.3g} MB per call: L2-warm (not a roofline figure)"),
            "parallelism": f"token rows sharded, {world} independent GPU(s), no collective"}


def rank_seed(cfg_index: int, T: int, rank: int) -> int:
    """Seed of rank `rank`'s own T token rows (weak scaling: disjoint shards)."""
    return 1_000_003 * cfg_index + T + 7919 * rank


def aggregate_gbs(bytes_per_rank: int, steps: int, max_ms: float, world: int) -> float:
    """Whole-job GB/s: the bytes every rank processed over the slowest rank's time."""
    return world * bytes_per_rank * steps / (max_ms * 1e-3) / 1e9


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


HOST_SIDE_MARK = "// ------------------------------------------------------------------ host side"


def kernel_source_sha() -> str:
    """Hash of the streaming kernel's device code: stream_rows.cu up to its
    host-side section, and the device header arf_common.cuh, with comments
    and blank lines dropped -- so an edited comment or a host-side change
    (planning, launch, declarations) does not void a traffic capture."""
    import re
    h = hashlib.sha256()
    for name in ("stream_rows.cu", "arf_common.cuh"):
        with open(os.path.join(ROOT, "tp_reduce_moe_gb300", "csrc", name)) as f:
            text = f.read()
        if name == "stream_rows.cu":
            text = text[:text.index(HOST_SIDE_MARK)]
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update("\n".join(line.rstrip() for line in text.splitlines() if line.strip()).encode())
    return h.hexdigest()[:16]


# ------------------------------------------------------------------ clocks
def smi_device_id(torch, local: int) -> str:
    """nvidia-smi id of the CUDA device (its UUID: CUDA_VISIBLE_DEVICES may remap indices)."""
    try:
        u = str(torch.cuda.get_device_properties(local).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(local)


class ClockSampler:
    """nvidia-smi samples (200 ms) kept only while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.samples, self.active = [], False
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(device_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.5)   # let nvidia-smi come up before the timed region

    def _read(self):
        for line in self.proc.stdout:
            if self.active:
                self.samples.append([x.strip() for x in line.split(",")])

    def start(self):
        self.active = True

    def stop(self):
        time.sleep(0.25)
        self.active = False
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.samples:
            return None
        sm = [float(s[1]) for s in self.samples if len(s) > 2 and s[1].replace(".", "").isdigit()]
        mx = [float(s[2]) for s in self.samples if len(s) > 2 and s[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for s in self.samples:
            for i, n in enumerate(names):
                if len(s) > 5 + i and s[5 + i].lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(self.samples)}


# ------------------------------------------------------------------ CPU oracle
def cpu_oracle_run(min_seconds: float, seed: int, reps_max: int = 1000, one_thread_passes: int = 0):
    """Time the CPU oracle on a bounded sample of the headline workload: T=512
    token rows drawn with the same recipe (R=8, K=10, H=8192), repeated until
    at least min_seconds have passed.  Returns (GB/s, threads, sample text,
    per-pass seconds, GB/s on one thread over one_thread_passes passes or
    None)."""
    import oracle
    from gen import make_inputs, problem_bytes
    from tests._util import oracle_args
    cores = len(os.sched_getaffinity(0))
    oracle.set_num_threads(cores)
    inp = make_inputs(HEADLINE[0], CPU_SAMPLE_T, seed=seed)
    a = oracle_args(inp)
    call = lambda: oracle.ar_finalize_rmsnorm_ref(a["E"], a["perm"], a["w"], a["S"], a["residual"],
                                                  a["gamma"], a["weight_bias"], a["eps"])
    call()  # page in
    times = []
    t_all = time.perf_counter()
    while (time.perf_counter() - t_all < min_seconds or len(times) < 3) and len(times) < reps_max:
        t0 = time.perf_counter()
        call()
        times.append(time.perf_counter() - t0)
    b = problem_bytes(inp["R"], inp["K"], inp["H"], CPU_SAMPLE_T)
    gbs = b * len(times) / sum(times) / 1e9
    sample = (f"{CPU_SAMPLE_T} token rows of the prefill workload (R=8, K=10, H=8192) drawn with its "
              f"recipe, {b / 1e9:.3f} GB per pass, {len(times)} passes in {sum(times):.1f} s")
    threads = oracle.num_threads()
    gbs1 = None
    if one_thread_passes > 0:
        oracle.set_num_threads(1)
        try:
            t0 = time.perf_counter()
            for _ in range(one_thread_passes):
                call()
            gbs1 = b * one_thread_passes / (time.perf_counter() - t0) / 1e9
        finally:
            oracle.set_num_threads(threads)
    return gbs, threads, sample, times, gbs1


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    from gen import CONFIGS, make_inputs, problem_bytes
    from tests._util import oracle_args
    cores = len(os.sched_getaffinity(0))
    oracle.set_num_threads(cores)
    inp = make_inputs(HEADLINE[0], CPU_SAMPLE_T, seed=7)
    a = oracle_args(inp)
    call = lambda: oracle.ar_finalize_rmsnorm_ref(a["E"], a["perm"], a["w"], a["S"], a["residual"],
                                                  a["gamma"], a["weight_bias"], a["eps"])
    for _ in range(max(args.warmup, 0)):
        call()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        call()
        times.append(time.perf_counter() - t0)
    b = problem_bytes(inp["R"], inp["K"], inp["H"], CPU_SAMPLE_T)
    value = b * len(times) / sum(times) / 1e9
    sample = (f"{CPU_SAMPLE_T} token rows of the prefill workload (R=8, K=10, H=8192) per step, "
              f"drawn with its recipe ({b / 1e9:.3f} GB per step)")
    cfg = CONFIGS[HEADLINE[0]]
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * sum(times) / len(times), 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": headline_config(HEADLINE[0], args.tokens, args.gpus),
            "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm
def main_ours(args):
    import torch
    import torch.distributed as dist

    import tp_reduce_moe_gb300 as arf
    from gen import CONFIGS, make_inputs, problem_bytes
    from tp_reduce_moe_gb300 import build as arbuild

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    if rank == 0 or world == 1:
        arbuild.build()
    if world > 1:
        dist.barrier()
    arf.load_library()

    def barrier():
        if world > 1:
            dist.barrier()

    def rank_max(x: float) -> float:
        return max_over_ranks(x, world, dev)

    cfg = CONFIGS[args.workload]
    T = args.tokens
    R, K, H = cfg.R, cfg.K, cfg.H
    # weak scaling: every rank draws and reduces its own T token rows
    d = make_inputs(cfg, T, seed=rank_seed(cfg.index, T, rank), device=dev)
    ws = arf.ar_workspace_create(R, K, H, T, cfg.eps, device=local,
                                 flags=arf.AR_WS_PDL if args.pdl else 0)
    force, csize = parse_regime(args.regime)
    arf.ar_workspace_set_regime(ws, force)
    arf.ar_workspace_set_cluster_size(ws, csize)
    arf.ar_workspace_set_stage_bytes(ws, args.stage_bytes)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    r_out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    gate = None
    if args.gated:
        from gen import make_gate_logits
        gate = make_gate_logits(T, device=dev)

    def step():
        if K == 0:
            arf.ar_rmsnorm(ws, d["S"], d["residual"], d["gamma"], d["weight_bias"], d["eps"],
                           out=out, residual_out=r_out, stream=stream)
        else:
            arf.ar_finalize_rmsnorm(ws, d["E"], d["perm"], d["w"], d["S"], d["residual"], d["gamma"],
                                    d["weight_bias"], d["eps"], out=out, residual_out=r_out,
                                    stream=stream, shared_gate=gate)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    regime, ctas = arf.ar_workspace_last_regime(ws)
    plan = {k: v for k, v in arf.ar_workspace_last_plan(ws).items() if v and k not in ("regime", "ctas_per_row")}

    clocks = ClockSampler(smi_device_id(torch, local))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_begin.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier()
    clocks.stop()
    total_ms = t_begin.elapsed_time(t_end)
    launch_ms = [a.elapsed_time(b) for a, b in ev]
    dev_err = arf.ar_workspace_device_error(ws)
    if dev_err:
        raise RuntimeError(f"device error word {dev_err:#x} after the timed region")
    total_ms = rank_max(total_ms)
    bytes_step = problem_bytes(R, K, H, T)
    value = aggregate_gbs(bytes_step, args.steps, total_ms, world)
    ms_per_step = total_ms / args.steps
    avg_launch_ms = statistics.fmean(launch_ms)

    peak, peak_kind = peaks()
    achieved = bytes_step / (avg_launch_ms * 1e-3) / 1e9
    traffic = None
    try:
        with open(PROFILE_TRAFFIC) as f:
            prof = json.load(f)
        if prof.get("kernel_source_sha") == kernel_source_sha():
            traffic = int(prof["dram_bytes_per_row"] * T)
    except (OSError, ValueError, KeyError):
        pass
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "peak_source": f"{peak_kind} HBM copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                if peak_kind == "measured" else "fallback 6.8 TB/s",
                "kernel": "cluster_rows_kernel" if regime == arf.AR_REGIME_ONESHOT else "stream_rows_kernel",
                "algorithmic_bytes_per_launch": bytes_step}

    # ---------------------------------------------- end to end (host buffers)
    e2e = None
    if not args.no_e2e and K > 0:
        e2e = run_e2e(args, arf, torch, d, ws, dev, stream, bytes_step, barrier, rank_max, world)

    sweep = None
    if not args.no_sweep and rank == 0:
        sweep = run_sweep(arf, torch, dev, stream, peak, args.sweep_regimes.split(","),
                          [w for w in args.sweep_only.split(",") if w], args.sweep_mode,
                          gated=args.gated,
                          pdls={"off": (False,), "on": (True,), "both": (False, True)}[args.sweep_pdl],
                          perm_kind=args.sweep_perm)
    # The L2-hot numbers beside the cold ones: the decode workloads at their
    # configured T with one input set replayed (inputs that fit the L2 stay
    # there).
    sweep_warm = None
    if not args.no_sweep and rank == 0 and args.sweep_mode == "rotate" and not args.sweep_only:
        sweep_warm = run_sweep(arf, torch, dev, stream, peak, ("auto",), ("ar_only", "dsv3_decode", "glm_gemma"),
                               "warm", gated=args.gated, pdls=(False,), perm_kind=args.sweep_perm, extra=False)

    cpu = None
    if not args.no_cpu and rank == 0 and world == 1:
        gbs, cores, sample, _, gbs1 = cpu_oracle_run(10.0, seed=7, one_thread_passes=2)
        cpu = {"value": round(gbs, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": sample, "value_1_thread": round(gbs1, 3)}

    ws.destroy()
    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
                "data": "synthetic",
                "config": headline_config(args.workload, T, world),
                "us_per_call": round(1e3 * ms_per_step, 3),
                "regime": REGIME_NAMES.get(regime, "?"), "ctas": ctas, "plan": plan, "gated": bool(args.gated),
                "pdl": bool(args.pdl),
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": args.steps, "clocks": clocks.summary(), "sweep": sweep,
                "sweep_warm": sweep_warm}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_e2e(args, arf, torch, d, ws, dev, stream, bytes_step, barrier, rank_max, world):
    """Same call through the public binding, inputs from pinned host memory:
    each step copies every input host->device, runs the op and copies out and
    residual_out back, all inside the timed region.  The device inputs are
    double-buffered, so step i's host->device copies overlap step i-1's kernel
    and read-back (as a serving loop would), never the copies of another step."""
    R = len(d["E"])
    ins = [*d["E"], *d["S"], d["residual"], d["gamma"], d["perm"], d["w"]]
    host = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in ins]
    for h, x in zip(host, ins):
        h.copy_(x)
    sets = [ins, [torch.empty_like(x) for x in ins]]
    T, H = d["T"], d["H"]
    h_out = torch.empty((T, H), dtype=torch.bfloat16, pin_memory=True)
    h_rout = torch.empty((T, H), dtype=torch.bfloat16, pin_memory=True)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    r_out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    h2d = sum(x.numel() * x.element_size() for x in ins)
    d2h = 2 * T * H * 2

    copy_streams = [torch.cuda.Stream(dev) for _ in range(max(1, args.e2e_streams))]
    last_read = [None, None]  # per input set: the kernel that last read it

    def step(i, start=None):
        cur = sets[i % 2]
        for j, (h, x) in enumerate(zip(host, cur)):
            cs = copy_streams[j % len(copy_streams)]
            if start is not None:
                cs.wait_event(start)
            if last_read[i % 2] is not None:
                cs.wait_event(last_read[i % 2])
            with torch.cuda.stream(cs):
                x.copy_(h, non_blocking=True)
        for cs in copy_streams:
            ev = torch.cuda.Event()
            ev.record(cs)
            stream.wait_event(ev)
        E, S = cur[:R], cur[R:2 * R]
        residual, gamma, perm, w = cur[2 * R:]
        arf.ar_finalize_rmsnorm(ws, E, perm, w, S, residual, gamma, d["weight_bias"], d["eps"],
                                out=out, residual_out=r_out, stream=stream)
        ev = torch.cuda.Event()
        ev.record(stream)
        last_read[i % 2] = ev
        with torch.cuda.stream(stream):
            h_out.copy_(out, non_blocking=True)
            h_rout.copy_(r_out, non_blocking=True)

    for i in range(2):
        step(i)
    torch.cuda.synchronize()
    barrier()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    n = max(1, args.e2e_steps)
    a.record(stream)
    for i in range(n):
        step(i, start=a if i == 0 else None)
    b.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms = rank_max(a.elapsed_time(b)) / n
    # The host link on its own (after the timed region): the largest input's
    # pinned host->device copy, best of three -- the bound the e2e step meets.
    big = max(range(len(host)), key=lambda j: host[j].numel() * host[j].element_size())
    nbytes = host[big].numel() * host[big].element_size()
    link = 0.0
    for _ in range(3):
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        with torch.cuda.stream(stream):
            sets[0][big].copy_(host[big], non_blocking=True)
        c1.record(stream)
        torch.cuda.synchronize()
        link = max(link, nbytes / (c0.elapsed_time(c1) * 1e-3) / 1e9)
    del host, sets
    return {"value": round(world * bytes_step / (ms * 1e-3) / 1e9, 2), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 3),
            "h2d_gbs": round(h2d / (ms * 1e-3) / 1e9, 2), "host_link_gbs": round(link, 2),
            "steps": n, "copy_streams": len(copy_streams),
            "overlap": "inputs double-buffered: a step's host->device copies overlap the previous "
                       "step's kernel and read-back",
            "api": "tp_reduce_moe_gb300.ar_finalize_rmsnorm"}


# Token counts swept beyond each workload's configured ones: the mid-range decode
# T where the regime tables switch kernels and ring variants.
SWEEP_EXTRA_T = {"dsv3_decode": (24, 32, 36, 48, 72, 96, 112, 160, 192, 256)}


def run_sweep(arf, torch, dev, stream, peak, regimes=("auto",), only=(), mode="rotate",
              gated=False, pdls=(False,), perm_kind="random", extra=True):
    """µs/call vs T for every workload: L2-cold by rotating through disjoint
    input sets (>= 3x L2 in total; each set gathers only within its own block
    of expert rows, like successive layers), timed by replaying a CUDA graph
    of one call per set."""
    from gen import CONFIGS, make_inputs, problem_bytes
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    res = []
    for name in ("ar_only", "dsv3_decode", "glm_gemma", "prefill"):
        if only and name not in only:
            continue
        cfg = CONFIGS[name]
        for T in sorted(set(cfg.Ts) | set(SWEEP_EXTRA_T.get(name, ()) if extra else ())):
            if name == "prefill" and T == HEADLINE[1]:
                continue
            for regime_name in regimes:
                for pdl in pdls:
                    res.append(sweep_point(arf, torch, dev, stream, peak, l2, cfg, name, T,
                                           *parse_regime(regime_name), mode=mode,
                                           gated=gated and cfg.K > 0, pdl=pdl, perm_kind=perm_kind))
    from gen import MHC_SHAPES
    for name, shp in MHC_SHAPES.items():
        if only and name not in only and "mhc" not in only:
            continue
        for T in shp["Ts"]:
            for pdl in pdls:
                res.append(sweep_mhc_point(arf, torch, dev, stream, peak, l2, name, shp, T, mode, pdl))
    return res


def sweep_mhc_point(arf, torch, dev, stream, peak, l2, name, shp, T, mode="rotate", pdl=False):
    """One T of the all-reduce + mHC write-back (ar_mhc_post), timed like the
    main sweep: a CUDA graph of one call per disjoint input set (>= 3x L2)."""
    from gen import make_mhc_inputs, mhc_problem_bytes
    R, H, hc = shp["R"], shp["H"], shp["hc"]
    b = mhc_problem_bytes(R, H, hc, T)
    n_sets = 1 if mode == "warm" else int(min(8192, max(2, math.ceil(3 * l2 / b))))
    inp = make_mhc_inputs(R, H, hc, T * n_sets, seed=5 + T, device=dev)
    P, x, post, comb = inp["P"], inp["x"], inp["post"], inp["comb"]
    out = torch.empty_like(x)
    ws = arf.ar_workspace_create(R, 0, H, T, 1e-6, device=dev.index, flags=arf.AR_WS_PDL if pdl else 0)

    def call(i):
        sl = slice(i * T, (i + 1) * T)
        arf.ar_mhc_post(ws, [p[sl] for p in P], x[sl], post[sl], comb[sl], out=out[sl])

    for i in range(min(n_sets, 4)):
        call(i)
    torch.cuda.synchronize()
    # warm: the one input set called WARM_CALLS times per graph (a graph of
    # one call would time the graph launch, not the call)
    calls = WARM_CALLS if mode == "warm" else n_sets
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(calls):
            call(i % n_sets)
    g.replay()
    torch.cuda.synchronize()
    per = []
    reps = 4 if mode == "warm" else 1
    for _ in range(3):
        a = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            g.replay()
        e.record(stream)
        torch.cuda.synchronize()
        per.append(a.elapsed_time(e) * 1e3 / (calls * reps))
    us = statistics.median(per)
    gbs = b / (us * 1e-6) / 1e9
    err = arf.ar_workspace_device_error(ws)
    del g, inp, out, P, x, post, comb
    ws.destroy()
    torch.cuda.empty_cache()
    return {"workload": name, "R": R, "K": 0, "H": H, "hc": hc, "T": T, "us_per_call": round(us, 3),
            "GBps": round(gbs, 1), "frac_of_hbm_peak": round(gbs / peak, 4), "regime": "mhc_post",
            "ctas": None, "forced": False, "calls_per_graph": calls, "mode": mode, "gated": False,
            "pdl": pdl, "device_error": err}


def sweep_point(arf, torch, dev, stream, peak, l2, cfg, name, T, force, csize=0, mode="rotate",
                gated=False, pdl=False, perm_kind="random"):
    """One (workload, T, regime) point of the sweep."""
    from gen import make_gate_logits, make_inputs, problem_bytes
    b = problem_bytes(cfg.R, cfg.K, cfg.H, T)
    n_sets = int(min(8192, max(2, math.ceil(3 * l2 / b))))
    if mode == "warm":
        n_sets = 1
    big = make_inputs(cfg, T * n_sets, seed=11 + T, device=dev, perm_kind=perm_kind,
                      perm_blocks=n_sets if mode == "rotate" else 1)
    ws = arf.ar_workspace_create(cfg.R, cfg.K, cfg.H, T, cfg.eps, device=dev.index,
                                 flags=arf.AR_WS_PDL if pdl else 0)
    arf.ar_workspace_set_regime(ws, force)
    arf.ar_workspace_set_cluster_size(ws, csize)
    outs = torch.empty((n_sets, T, cfg.H), dtype=torch.bfloat16, device=dev)
    routs = torch.empty((n_sets, T, cfg.H), dtype=torch.bfloat16, device=dev)
    gates = make_gate_logits(T * n_sets, device=dev) if gated else None

    def call(i, st):
        sl = slice(i * T, (i + 1) * T)
        S = [x[sl] for x in big["S"]] if big["S"] is not None else None
        if cfg.K == 0:
            arf.ar_rmsnorm(ws, S, big["residual"][sl], big["gamma"], 0.0, cfg.eps,
                           out=outs[i], residual_out=routs[i], stream=st)
        else:
            arf.ar_finalize_rmsnorm(ws, big["E"], big["perm"][sl], big["w"][sl], S,
                                    big["residual"][sl], big["gamma"], 0.0, cfg.eps,
                                    out=outs[i], residual_out=routs[i], stream=st,
                                    rows_e=big["rows_e"],
                                    shared_gate=gates[sl] if gates is not None else None)

    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    try:
        with torch.cuda.stream(side):
            for i in range(min(n_sets, 8)):
                call(i, side)
    except arf.ArfuseError as e:  # a forced regime with no plan for this shape
        ws.destroy()
        return {"workload": name, "T": T, "regime": REGIME_NAMES.get(force, "auto"), "ctas": csize,
                "forced": True, "unsupported": arf.ar_status_string(e.status)}
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize()
    regime, ctas = arf.ar_workspace_last_regime(ws)
    plan = {k: v for k, v in arf.ar_workspace_last_plan(ws).items() if v and k not in ("regime", "ctas_per_row")}
    calls = WARM_CALLS if mode == "warm" else n_sets
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cs = torch.cuda.current_stream(dev)
        for i in range(calls):
            call(i % n_sets, cs)
    g.replay()
    torch.cuda.synchronize()
    per = []
    reps = 4 if mode == "warm" else 1
    for _ in range(3):
        a = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            g.replay()
        e.record(stream)
        torch.cuda.synchronize()
        per.append(a.elapsed_time(e) * 1e3 / (calls * reps))
    us = statistics.median(per)
    gbs = b / (us * 1e-6) / 1e9
    err = arf.ar_workspace_device_error(ws)
    del g, big, outs, routs
    ws.destroy()
    torch.cuda.empty_cache()
    return {"workload": name, "R": cfg.R, "K": cfg.K, "H": cfg.H, "T": T,
            "us_per_call": round(us, 3), "GBps": round(gbs, 1),
            "frac_of_hbm_peak": round(gbs / peak, 4),
            "regime": REGIME_NAMES.get(regime, "?"), "ctas": ctas, "plan": plan,
            "forced": force != 0, "calls_per_graph": calls, "mode": mode, "perm": perm_kind,
            "gated": gated,
            "pdl": pdl, "device_error": err}


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return main_ours(args)


if __name__ == "__main__":
    sys.exit(main())
