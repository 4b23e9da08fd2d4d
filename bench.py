#!/usr/bin/env python
"""MoE-layer forward benchmark (one JSON line on rank 0).

Workload: the DeepSeek-V3-shaped layer (T=16384 tokens, D=7168, I=2048,
256 routed experts, top-8, one shared expert with I_s=2048, sigmoid router
with a bias that gives the experts a Zipf(1.1) load), BF16, synthetic seeded
inputs (moe_inputs).  A step is one moe_fwd call: router + top-k, schedule,
persistent dispatch/expert-FFN/combine kernel.  Throughput is tokens/s and
effective TFLOP/s = 6 T (k + 1) D I / t ("Mixture-of-Kittens", Sec. 4.1).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs N independent replicas (one process per GPU, launched by
torch.distributed.run): the layer has no data-parallel exchange on one node,
so value = all replicas' tokens / max-over-ranks time ("scaling": "weak").
--impl reference times the fp64 CPU oracle (the only reference this build
has) on a bounded token sample per step, on rank 0.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

REPO = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, REPO)

import moe_inputs as mi  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
SMI_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
REASON_NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
METRIC = "MoE-layer fwd tokens/s (DSV3 shape, 16K tok)"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="dsv3", choices=sorted(mi.CONFIGS))
    ap.add_argument("--minibatch", type=int, default=8192)
    ap.add_argument("--ring-slots", type=int, default=4)
    ap.add_argument("--gather-ctas", type=int, default=8)
    ap.add_argument("--lag", type=int, default=1)
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="target CPU time of the oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--tokens", type=int, default=0,
                    help="profiling only: a smaller case with this many tokens (uniform routing)")
    ap.add_argument("--experts", type=int, default=0,
                    help="profiling only: a smaller case with this many routed experts (uniform routing)")
    return ap.parse_args()


def select_workload(args):
    """The named workload, or (profiling only) a smaller case of the same D, I,
    k, I_s with --tokens / --experts and uniform routing."""
    shape = mi.CONFIGS[args.workload]
    if not args.tokens and not args.experts:
        return shape, mi.make_inputs(shape)
    T = args.tokens or shape.T
    E = args.experts or shape.E
    small = mi.custom_shape(T, shape.D, shape.I, E, shape.k, shape.I_s, score=shape.score,
                            config_id=shape.config_id + 1000)
    return small, mi.make_inputs(small, calibration={"beta": None, "redraw": {}})


def load_peaks():
    path = os.path.join(REPO, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return FALLBACK_PEAKS, "fallback"


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={SMI_FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], 0.0, set()
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx = max(mx, float(parts[2]))
                except ValueError:
                    continue
                for name, flag in zip(REASON_NAMES, parts[5:9]):
                    if flag.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- distributed
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != n_gpus and world > 1:
        raise SystemExit(f"--gpus {n_gpus} but WORLD_SIZE {world}")
    return world, rank, local


# ----------------------------------------------------------------------------- oracle timing
def time_oracle(inp, seconds: float):
    """Oracle on a contiguous token slice sized for about `seconds` of CPU time."""
    import oracle
    probe = 2 * max(1, oracle.num_threads())
    t0 = time.perf_counter()
    oracle.moe_fwd_inputs(inp, rows=np.arange(probe))
    per_tok = (time.perf_counter() - t0) / probe
    n = int(max(probe, min(inp.T, seconds / max(per_tok, 1e-9))))
    t0 = time.perf_counter()
    oracle.moe_fwd_inputs(inp, rows=np.arange(n))
    dt = time.perf_counter() - t0
    return {"value": n / dt, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"first {n} tokens of the {inp.shape.name} workload (T={inp.shape.T}), fp64, "
                      f"{dt:.1f} s; per-token cost is constant (k+1 expert FFNs)",
            "seconds": dt}


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    import oracle
    shape, inp = select_workload(args)
    per_step_tokens = None
    times = []
    total_steps = args.warmup + args.steps
    budget = 150.0  # seconds of oracle work for the whole run
    probe = 2 * max(1, oracle.num_threads())
    t0 = time.perf_counter()
    oracle.moe_fwd_inputs(inp, rows=np.arange(probe))
    per_tok = (time.perf_counter() - t0) / probe
    per_step_tokens = int(max(1, min(shape.T, budget / total_steps / max(per_tok, 1e-9))))
    rows = np.arange(per_step_tokens)
    for i in range(total_steps):
        t0 = time.perf_counter()
        oracle.moe_fwd_inputs(inp, rows=rows)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    total = sum(times)
    value = per_step_tokens * len(times) / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * total / len(times), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(shape, args, "oracle on host cores"),
        "tflops": shape.flops(per_step_tokens) * len(times) / total / 1e12,
        "cpu_baseline": {"kind": "oracle", "cores": oracle.num_threads(), "value": value, "unit": "tokens/s",
                         "sample": f"first {per_step_tokens} tokens of the {shape.name} workload per step, fp64"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(shape, args, extra=None):
    cfg = {"workload": f"{shape.name}: DeepSeek-V3-shaped MoE layer forward" if shape.name.startswith("dsv3")
           else f"{shape.name} MoE layer forward",
           "T": shape.T, "D": shape.D, "I": shape.I, "E": shape.E, "k": shape.k, "I_s": shape.I_s,
           "score": shape.score, "load": "Zipf(1.1) via router bias" if shape.load == "zipf" else shape.load,
           "precision": shape.precision, "minibatch": args.minibatch, "ring_slots": args.ring_slots,
           "gather_ctas": args.gather_ctas, "lag": args.lag,
           "l2": "inputs larger than L2 (expert weights 22.5 GB, x 235 MB for dsv3); no flush",
           "parallelism": "replicas"}
    if extra:
        cfg["note"] = extra
    return cfg


# ----------------------------------------------------------------------------- our arm
def run_ours(args, world, rank, local):
    import torch
    import routing_grouped_expert_gemm_gb300 as rg
    from routing_grouped_expert_gemm_gb300 import build as rgbuild

    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    rgbuild.build()
    t_gen = time.perf_counter()
    shape, inp = select_workload(args)
    t_gen = time.perf_counter() - t_gen
    if shape.precision != "bf16":
        raise SystemExit("only the bf16 path is benchmarked by this arm")

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()

    T = shape.T
    plan = rg.moe_plan_create(T, shape.D, shape.I, shape.E, shape.k, shape.I_s, score_fn=shape.score,
                              minibatch=args.minibatch, ring_slots=args.ring_slots, gather_ctas=args.gather_ctas,
                              lag=args.lag)
    w = {"W_router": dev(inp.w_router),
         "b_router": None if inp.b_router is None else torch.from_numpy(inp.b_router).cuda(),
         "W_up": dev(inp.w_up), "W_gate": dev(inp.w_gate), "W_down": dev(inp.w_down)}
    if shape.I_s:
        w.update(Ws_up=dev(inp.ws_up), Ws_gate=dev(inp.ws_gate), Ws_down=dev(inp.ws_down))
    x = dev(inp.x)
    ws_bytes = rg.moe_workspace_bytes(plan, T)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.empty((T, shape.D), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        rg.moe_fwd(plan, T, x, w, out, ws, ws_bytes, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    status = rg.moe_get_status(plan, ws, stream=stream)
    if status != 0:
        raise SystemExit(f"device status {status} after warm-up")

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # ---- device-resident timed region (per-launch events on the launching stream)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    for e4 in ev:  # torch creates the CUDA event at its first record
        for e in e4:
            e.record(stream)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(args.steps):
        rg.moe_plan_set_timing_events(plan, ev[i])
        step()
    end.record(stream)
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop()
    rg.moe_plan_set_timing_events(plan, None)
    status = rg.moe_get_status(plan, ws, stream=stream)
    if status != 0:
        raise SystemExit(f"device status {status} in the timed region")
    elapsed_ms = start.elapsed_time(end)
    router_ms = [e[0].elapsed_time(e[1]) for e in ev]
    sched_ms = [e[1].elapsed_time(e[2]) for e in ev]
    mega_ms = [e[2].elapsed_time(e[3]) for e in ev]
    step_ms = [e[0].elapsed_time(e[3]) for e in ev]

    # ---- end to end: pinned host x in, host out back, every step
    e2e = None
    if not args.no_e2e:
        x_host = torch.from_numpy(np.ascontiguousarray(inp.x).view(np.int16)).view(torch.bfloat16).pin_memory()
        out_host = torch.empty((T, shape.D), dtype=torch.bfloat16).pin_memory()
        x_in = torch.empty_like(x)
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(3):
            x_in.copy_(x_host, non_blocking=True)
            rg.moe_fwd(plan, T, x_in, w, out, ws, ws_bytes, stream=stream)
            out_host.copy_(out, non_blocking=True)
        barrier()
        torch.cuda.synchronize()
        s0.record(stream)
        for _ in range(args.steps):
            x_in.copy_(x_host, non_blocking=True)
            rg.moe_fwd(plan, T, x_in, w, out, ws, ws_bytes, stream=stream)
            out_host.copy_(out, non_blocking=True)
        s1.record(stream)
        torch.cuda.synchronize()
        barrier()
        e2e_ms = s0.elapsed_time(s1)
        e2e = {"ms": e2e_ms, "h2d": x_host.numel() * 2, "d2h": out_host.numel() * 2}

    # ---- max over ranks
    def allmax(v):
        if world == 1:
            return v
        import torch.distributed as dist
        t = torch.tensor([v], dtype=torch.float64, device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    elapsed_ms = allmax(elapsed_ms)
    if e2e:
        e2e["ms"] = allmax(e2e["ms"])
    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0

    peaks, peak_src = load_peaks()
    flops = shape.flops(T)
    mega_mean = sum(mega_ms) / len(mega_ms)
    achieved = flops / (mega_mean / 1000.0) / 1e12
    peak = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
    value = world * T * args.steps / (elapsed_ms / 1000.0)
    line = {
        "metric": METRIC,
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded normal inputs, random-init weights)",
        "config": workload_config(shape, args),
        "tflops": world * flops * args.steps / (elapsed_ms / 1000.0) / 1e12,
        "tflops_frac_of_peak": (world * flops * args.steps / (elapsed_ms / 1000.0) / 1e12) / (world * peak),
        "ms_median_step": statistics.median(step_ms),
        "phases_ms_mean": {"router_topk": sum(router_ms) / len(router_ms), "schedule": sum(sched_ms) / len(sched_ms),
                           "megakernel": mega_mean},
        "roofline": {"kernel": "moe_megakernel", "bound": "tensor", "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak, "traffic": None,
                     "peak_source": f"{peak_src} bf16 sustained (kernel timed inside a long loop)",
                     "frac_of_burst_peak": achieved / float(peaks["bf16_tflops"])},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
        "input_generation_s": t_gen,
    }
    if e2e:
        line["e2e"] = {"value": world * T * args.steps / (e2e["ms"] / 1000.0), "unit": "tokens/s",
                       "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"]}
    if world == 1 and not args.no_cpu_baseline:
        cb = time_oracle(inp, args.cpu_seconds)
        line["cpu_baseline"] = {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")}
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    world, rank, local = dist_setup(args.gpus)
    if args.impl == "reference":
        return run_reference(args, world, rank)
    return run_ours(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
