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
--impl reference times the fp64 CPU oracle (there is no other reference
implementation) on a bounded token sample per step, on rank 0.
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
    ap.add_argument("--no-mxfp8", action="store_true", help="skip the MXFP8 sub-measurement")
    ap.add_argument("--no-backward", action="store_true", help="skip the forward + backward measurement")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the minibatch sweep (512 / 2048 / 8192 / 32768 and ring vs over-allocation)")
    ap.add_argument("--gather-ctas-mx", type=int, default=6, help="gather CTAs for the MXFP8 layer")
    ap.add_argument("--dispatch", choices=["ring", "direct", "spread"], default="spread",
                    help="BF16 layer: how the routed tokens reach the expert tiles (spread: every GEMM CTA "
                         "fills the ring, measured fastest on every workload; ring: --gather-ctas CTAs fill it)")
    ap.add_argument("--dispatch-mx", choices=["ring", "direct", "spread"], default="spread",
                    help="MXFP8 layer: the same choice (spread measured fastest on DSV3)")
    ap.add_argument("--mma-pair", type=int, default=1, choices=[0, 1],
                    help="CTA-pair (cta_group::2) expert tiles, BF16 and MXFP8 (measured fastest on DSV3)")
    ap.add_argument("--raster", type=int, default=0, help="up/gate tile order: M-tiles per group (0 = default)")
    ap.add_argument("--pad-odd-tiles", type=int, default=0, choices=[0, 1],
                    help="CTA pairs: 1 runs an expert segment's odd last M-tile with an empty partner instead of "
                         "splitting it over the pair (bf16; MXFP8 always pads)")
    ap.add_argument("--plain-launch", action="store_true",
                    help="profiling only: launch the persistent kernel without the cooperative attribute, "
                         "so that ncu can replay the CTA-pair kernel")
    ap.add_argument("--gemm-ctas", type=int, default=0, help="CTAs that run expert tiles (0 = all remaining SMs)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="profiling only: a smaller case with this many tokens (uniform routing)")
    ap.add_argument("--route-only", action="store_true",
                    help="profiling only: time the routing stage alone (moe_route_static: router + top-k + "
                         "schedule) on the workload's x and router; no expert weights on the device")
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
                            config_id=shape.config_id + 1000, precision=shape.precision)
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


def reduce_max(v: float, world: int) -> float:
    """Max of v over all ranks (the slowest replica sets the time).  Works with
    the nccl (GPU tensor) and gloo (CPU tensor) backends."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world: int, tokens_per_step: int, steps: int, elapsed_ms: float) -> float:
    """Whole-job tokens/s of `world` independent replicas timed together."""
    return world * tokens_per_step * steps / (elapsed_ms / 1000.0)


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
        "config": workload_config(shape, args),
        "note": "oracle on host cores",
        "tflops": shape.flops(per_step_tokens) * len(times) / total / 1e12,
        "cpu_baseline": {"kind": "oracle", "cores": oracle.num_threads(), "value": value, "unit": "tokens/s",
                         "sample": f"first {per_step_tokens} tokens of the {shape.name} workload per step, fp64"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(shape, args):
    cfg = {"workload": f"{shape.name}: DeepSeek-V3-shaped MoE layer forward" if shape.name.startswith("dsv3")
           else f"{shape.name} MoE layer forward",
           "T": shape.T, "D": shape.D, "I": shape.I, "E": shape.E, "k": shape.k, "I_s": shape.I_s,
           "score": shape.score, "load": "Zipf(1.1) via router bias" if shape.load == "zipf" else shape.load,
           "precision": shape.precision, "minibatch": args.minibatch, "ring_slots": args.ring_slots,
           "gather_ctas": (args.gather_ctas_mx if shape.precision == "mxfp8" else args.gather_ctas)
           if dispatch_of(shape, args) == "ring" else 0,
           "lag": args.lag, "dispatch": dispatch_of(shape, args),
           "mma_pair": args.mma_pair, "raster": args.raster,
           "pad_odd_tiles": (args.pad_odd_tiles if shape.precision == "bf16" else 1) if args.mma_pair else None,
           "gemm_ctas": args.gemm_ctas or "all remaining SMs",
           "l2": l2_note(shape),
           "parallelism": "replicas"}
    return cfg


def dispatch_of(shape, args) -> str:
    return args.dispatch_mx if shape.precision == "mxfp8" else args.dispatch


def l2_note(shape) -> str:
    """The timing rule this workload meets: its inputs are larger than L2."""
    routed = shape.E * 3 * shape.D * shape.I
    wbytes = (routed * 33 / 32 if shape.precision == "mxfp8" else routed * 2) + 3 * shape.D * shape.I_s * 2
    xbytes = shape.T * shape.D * 2
    return f"inputs larger than L2 (expert weights {wbytes / 1e9:.1f} GB, x {xbytes / 1e6:.0f} MB); no flush"


# ----------------------------------------------------------------------------- recorded DRAM traffic
# the sources that decide what the persistent kernel launch does: its code, the task
# schedule, the plan and launch set-up, the MXFP8 layouts and the C header (the router,
# the backward pass and the layout probes are separate launches)
TRAFFIC_SOURCES = ("api.cu", "common.cuh", "megakernel.cu", "mxfp8.cu", "plan.cuh", "ptx.cuh", "schedule.cu")


def kernel_sources_hash() -> str:
    """sha256 over the persistent kernel's sources and the C header: a recorded ncu
    traffic figure applies only to the kernel it was taken from."""
    import hashlib
    root = os.path.dirname(os.path.abspath(__file__))
    csrc = os.path.join(root, "routing_grouped_expert_gemm_gb300", "csrc")
    files = [os.path.join(csrc, f) for f in TRAFFIC_SOURCES]
    files.append(os.path.join(root, "include", "moe.h"))
    h = hashlib.sha256()
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def recorded_traffic(key: str, cfg: dict):
    """(dram__bytes_read.sum + dram__bytes_write.sum of one persistent-kernel
    launch, the record's note) from profiles/traffic_<key>.txt, if it was taken
    from these sources and this launch configuration; else (None, None)."""
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "profiles", f"traffic_{key}.txt")
    if not os.path.exists(path):
        return None, None
    rec = {}
    with open(path) as fh:
        for line in fh:
            parts = line.split(None, 1)
            if len(parts) == 2 and not line.startswith("#"):
                rec[parts[0]] = parts[1].strip()
    if rec.get("sources_sha256") != kernel_sources_hash():
        return None, None
    for k in ("minibatch", "ring_slots", "gather_ctas", "mma_pair", "raster", "dispatch", "pad_odd_tiles",
              "gemm_ctas"):
        if k in rec and str(cfg.get(k)) != rec[k]:
            return None, None
    try:
        return float(rec["dram_bytes_per_launch"]), rec.get("note", "")
    except (KeyError, ValueError):
        return None, None


def attach_traffic(roof: dict, shape, cfg: dict) -> dict:
    """The roofline's `traffic`: a recorded ncu figure of these sources and this
    launch configuration, else null."""
    key = f"{shape.name}_{shape.precision}"
    traffic, note = recorded_traffic(key, cfg)
    roof["traffic"] = traffic
    roof["traffic_note"] = (f"{note} (profiles/traffic_{key}.txt)" if traffic
                            else "no ncu capture for these sources and this launch configuration")
    return roof


# ----------------------------------------------------------------------------- our arm
class Runner:
    """One workload on the device: plan, weights (MXFP8 quantised outside any
    timed region), workspace, and a timed loop of moe_fwd calls."""

    def __init__(self, rg, torch, shape, inp, args, world, share=None, **knobs):
        """share: an earlier Runner of the same workload whose device weights and
        input are reused; knobs: plan settings that replace the arguments'."""
        self.rg, self.torch, self.shape, self.inp, self.args, self.world = rg, torch, shape, inp, args, world
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
        T = shape.T
        plan_kw = dict(minibatch=args.minibatch, ring_slots=args.ring_slots,
                       gather_ctas=args.gather_ctas_mx if shape.precision == "mxfp8" else args.gather_ctas,
                       lag=args.lag, dispatch=dispatch_of(shape, args), raster=args.raster,
                       gemm_ctas=args.gemm_ctas, mma_pair=args.mma_pair, plain_launch=int(args.plain_launch),
                       pad_odd_tiles=args.pad_odd_tiles)
        plan_kw.update(knobs)
        self.knobs = plan_kw
        self.plan = rg.moe_plan_create(T, shape.D, shape.I, shape.E, shape.k, shape.I_s, score_fn=shape.score,
                                       precision=shape.precision, **plan_kw)
        self.stream = torch.cuda.current_stream()
        self.launches = 3  # router (+ MXFP8 x quantisation), schedule, persistent kernel
        self.ws_bytes = rg.moe_workspace_bytes(self.plan, T)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device="cuda")
        if share is not None:
            self.w, self.x, self.out = share.w, share.x, share.out
            return
        w = {"W_router": dev(inp.w_router),
             "b_router": None if inp.b_router is None else torch.from_numpy(inp.b_router).cuda()}
        for name, arr, rows, K in (("W_up", inp.w_up, shape.E * shape.I, shape.D),
                                   ("W_gate", inp.w_gate, shape.E * shape.I, shape.D),
                                   ("W_down", inp.w_down, shape.E * shape.D, shape.I)):
            wd = dev(arr)
            if shape.precision == "mxfp8":  # pre-quantised weights (MoK Sec. 3.4), not timed
                q = torch.empty((rows, K), dtype=torch.uint8, device="cuda")
                sc = torch.empty(rg.moe_mxfp8_scale_bytes(rows, K), dtype=torch.uint8, device="cuda")
                rg.moe_quantize_mxfp8(self.plan, wd, rows, K, q, sc)
                torch.cuda.synchronize()
                del wd
                w[name], w[name + "_scale"] = q, sc
            else:
                w[name] = wd
        if shape.I_s:
            w.update(Ws_up=dev(inp.ws_up), Ws_gate=dev(inp.ws_gate), Ws_down=dev(inp.ws_down))
        self.w = w
        self.x = dev(inp.x)
        self.out = torch.empty((T, shape.D), dtype=torch.bfloat16, device="cuda")

    def step(self, x=None):
        self.rg.moe_fwd(self.plan, self.shape.T, self.x if x is None else x, self.w, self.out, self.ws,
                        self.ws_bytes, stream=self.stream)

    def barrier(self):
        if self.world > 1:
            import torch.distributed as dist
            dist.barrier()

    def status(self):
        return self.rg.moe_get_status(self.plan, self.ws, stream=self.stream)

    def timed(self, steps, warmup, sampler=None):
        torch, rg = self.torch, self.rg
        for _ in range(warmup):
            self.step()
        torch.cuda.synchronize()
        if self.status() != 0:
            raise SystemExit(f"device status {self.status()} after warm-up")
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
        for e4 in ev:  # torch creates the CUDA event at its first record
            for e in e4:
                e.record(self.stream)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        if sampler:
            sampler.start()
            time.sleep(0.3)
        self.barrier()
        torch.cuda.synchronize()
        start.record(self.stream)
        for i in range(steps):
            rg.moe_plan_set_timing_events(self.plan, ev[i])
            self.step()
        end.record(self.stream)
        torch.cuda.synchronize()
        self.barrier()
        clocks = sampler.stop() if sampler else None
        rg.moe_plan_set_timing_events(self.plan, None)
        if self.status() != 0:
            raise SystemExit(f"device status {self.status()} in the timed region")
        phases = rg.moe_get_phase_times(self.plan, self.ws, stream=self.stream)  # the last timed launch
        return {"elapsed_ms": start.elapsed_time(end), "phase_stamps_ms": phases,
                "router_ms": [e[0].elapsed_time(e[1]) for e in ev],
                "sched_ms": [e[1].elapsed_time(e[2]) for e in ev],
                "mega_ms": [e[2].elapsed_time(e[3]) for e in ev],
                "step_ms": [e[0].elapsed_time(e[3]) for e in ev], "clocks": clocks}

    def e2e(self, steps, pipelined=True):
        """pinned host x -> device, forward, device -> pinned host out, every step.

        pipelined: input copies, forwards and output copies run on three
        streams with two device input and output buffers, so that step i + 1's
        input copy and step i - 1's output copy overlap step i's forward (each
        step still moves its own input and result); otherwise copy, forward
        and copy run in sequence."""
        torch = self.torch
        x_host = torch.from_numpy(np.ascontiguousarray(self.inp.x).view(np.int16)).view(torch.bfloat16).pin_memory()
        outs_host = [torch.empty((self.shape.T, self.shape.D), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        x_in = [torch.empty_like(self.x) for _ in range(2)]
        outs = [self.out, torch.empty_like(self.out)]
        # the streams are created here: work on torch's legacy default stream
        # would serialise with every other stream; and one stream for both
        # copy directions would queue step i + 1's input copy behind step i's
        # output copy, which waits for step i's forward
        comp = torch.cuda.Stream() if pipelined else self.stream
        cs = torch.cuda.Stream() if pipelined else self.stream
        cs_out = torch.cuda.Stream() if pipelined else self.stream
        Ev = torch.cuda.Event

        def run(n):
            in_free, out_free = [None, None], [None, None]
            for i in range(n):
                b = i & 1
                with torch.cuda.stream(cs):
                    if in_free[b] is not None:
                        cs.wait_event(in_free[b])
                    x_in[b].copy_(x_host, non_blocking=True)
                    ready = Ev()
                    ready.record(cs)
                comp.wait_event(ready)
                if out_free[b] is not None:
                    comp.wait_event(out_free[b])
                self.rg.moe_fwd(self.plan, self.shape.T, x_in[b], self.w, outs[b], self.ws, self.ws_bytes,
                                stream=comp)
                done = Ev()
                done.record(comp)
                in_free[b] = done
                with torch.cuda.stream(cs_out):
                    cs_out.wait_event(done)
                    outs_host[b].copy_(outs[b], non_blocking=True)
                    copied = Ev()
                    copied.record(cs_out)
                out_free[b] = copied

        run(3)
        self.barrier()
        torch.cuda.synchronize()
        s0, s1 = Ev(enable_timing=True), Ev(enable_timing=True)
        s0.record(cs)  # before the first input copy
        run(steps)
        s1.record(cs_out)  # after the last output copy, which followed the last forward
        torch.cuda.synchronize()
        self.barrier()
        return {"ms": s0.elapsed_time(s1), "h2d": x_host.numel() * 2, "d2h": outs_host[0].numel() * 2}


def flops_split(shape, T=None):
    """(routed, shared) expert-FFN FLOPs of one forward (Sec. 4.1's 6 T k D I
    and 6 T D I_s)."""
    T = shape.T if T is None else T
    return 6.0 * T * shape.k * shape.D * shape.I, 6.0 * T * shape.D * shape.I_s


def tensor_roofline(shape, kernel_ms, bf16_peak, peak_src, burst_peak):
    """Roofline of the persistent kernel: achieved TFLOP/s against the time the
    work takes at peak.  BF16: every FLOP at the BF16 peak.  MXFP8: the routed
    FLOPs at 2x the BF16 peak (the dense MXFP8 rate, MoK Sec. 4.1) and the
    shared expert's (BF16) at 1x, so the peak is the blended rate."""
    routed, shared = flops_split(shape)
    total = routed + shared
    mx = shape.precision == "mxfp8"

    def at_peak_s(p):
        return (routed / (2.0 * p) if mx else routed / p) + shared / p
    achieved = total / (kernel_ms / 1000.0) / 1e12
    blended = total / at_peak_s(bf16_peak * 1e12) / 1e12
    blended_burst = total / at_peak_s(burst_peak * 1e12) / 1e12
    return {"kernel": "moe_megakernel", "bound": "tensor", "achieved": achieved, "peak": blended,
            "unit": "TFLOP/s", "frac": achieved / blended,
            "peak_source": f"{peak_src} bf16 sustained (kernel timed inside a long loop)"
                           + ("; routed FLOPs at 2x (MXFP8 dense), shared-expert FLOPs at 1x (BF16)" if mx else ""),
            "frac_of_burst_peak": achieved / blended_burst}


def phase_bandwidths(shape, res, hbm_peak):
    """HBM figures of the phases that move data rather than multiply, from the
    last timed launch: the router's read of x (CUDA events), the ring fill
    (bytes gathered over the window until the last minibatch was marked
    gathered; overlapped with the expert tiles and paced by the ring) and the
    final combine pass (it runs alone: staging rows + g read, output written)."""
    T, D, k, kY = shape.T, shape.D, shape.k, shape.k + shape.n_shared
    router_ms = statistics.mean(res["router_ms"])
    router_bytes = T * D * 2 + shape.E * D * 2
    fill_bytes = T * k * D * (2 + 2 if shape.precision == "bf16" else 2 + 1 + 1 / 32)
    comb_bytes = T * kY * D * 2 + T * D * 2 + T * k * 4
    st = res.get("phase_stamps_ms") or {}
    out = {"router": {"bytes": router_bytes, "ms": router_ms, "GB/s": router_bytes / router_ms / 1e6}}
    if st.get("last_fill"):
        out["ring_fill"] = {"bytes": fill_bytes, "window_ms": st["last_fill"],
                            "GB/s": fill_bytes / st["last_fill"] / 1e6,
                            "note": "x rows read + ring rows written (MXFP8: bf16 read, codes + scales written) "
                                    "over kernel start .. last minibatch gathered; overlapped, paced by the ring"}
    if st.get("combine_start") is not None and st.get("combine_end") is not None:
        ms = st["combine_end"] - st["combine_start"]
        if ms > 0:
            out["combine"] = {"bytes": comb_bytes, "ms": ms, "GB/s": comb_bytes / ms / 1e6,
                              "frac_of_hbm_peak": comb_bytes / ms / 1e6 / hbm_peak}
    out["hbm_peak_GB/s"] = hbm_peak
    return out


def minibatch_sweep(run, steps, warmup):
    """tokens/s of the same layer (same device weights) at the minibatch sizes
    MoK Sec. 3.2 sweeps, 4 ring slots each (32768 x 4 holds every route: the
    over-allocated buffer of Sec. 3.3), and ring vs over-allocation at the
    default minibatch (4 slots: the ring wraps; T k / b slots: it never does)."""
    shape = run.shape
    R = shape.T * shape.k
    base = run.knobs["minibatch"]
    points = [(b, 4) for b in (512, 2048, 8192, 32768)]
    points.append((base, max(4, -(-R // base))))
    out = []
    for b, slots in points:
        r = Runner(run.rg, run.torch, shape, run.inp, run.args, run.world, share=run, minibatch=b, ring_slots=slots)
        res = r.timed(steps, warmup)
        out.append({"minibatch": b, "ring_slots": slots, "wraps": slots * b < R,
                    "tokens_per_s": shape.T * steps / (res["elapsed_ms"] / 1000.0),
                    "ms_per_step": res["elapsed_ms"] / steps,
                    "megakernel_ms": statistics.mean(res["mega_ms"])})
        del r
    ring = next(p for p in out if p["minibatch"] == base and p["ring_slots"] == 4)
    full = out[-1]
    return {"points": out,
            "ring_vs_overallocation": {"minibatch": base, "ring_ms": ring["ms_per_step"],
                                       "overallocated_ms": full["ms_per_step"],
                                       "ring_overhead": ring["ms_per_step"] / full["ms_per_step"] - 1.0},
            "best_over_worst": max(p["tokens_per_s"] for p in out[:4]) / min(p["tokens_per_s"] for p in out[:4])}


def backward_flops(shape):
    """(phase 0, phase 1) FLOPs the backward executes: the replayed up/gate
    projections and dh' = W_down^T dO (6 T k D I routed, 6 T D I_s shared), then
    dx (4 T k D I), dW_down (2 T k D I) and dW_up, dW_gate (4 T k D I), and the
    shared expert's alike.  The pages count the backward as 2x the forward's
    6 T (k + 1) D I without the replay ("Mixture-of-Kittens", Sec. 4.1)."""
    R = shape.T * shape.k
    sh = shape.T * shape.I_s
    return 6.0 * R * shape.D * shape.I + 6.0 * sh * shape.D, 10.0 * R * shape.D * shape.I + 10.0 * sh * shape.D


def backward_timing(run, steps, warmup, bf16_peak, burst_peak, peak_src, sampler=None):
    """A training step of the layer: moe_fwd then moe_bwd (upstream gradient
    dO ~ N(0, 1), seeded), every gradient written.  Events bracket the
    forward's and the backward's phases."""
    torch, rg, shape = run.torch, run.rg, run.shape
    T = shape.T
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    dO = dev(mi.grad_out(shape))
    bf = torch.bfloat16
    g = {"dx": torch.empty((T, shape.D), dtype=bf, device="cuda"),
         "dW_router": torch.empty((shape.E, shape.D), dtype=torch.float32, device="cuda"),
         "db_router": torch.empty(shape.E, dtype=torch.float32, device="cuda") if run.inp.b_router is not None
         else None,
         "dW_up": torch.empty((shape.E, shape.I, shape.D), dtype=bf, device="cuda"),
         "dW_gate": torch.empty((shape.E, shape.I, shape.D), dtype=bf, device="cuda"),
         "dW_down": torch.empty((shape.E, shape.D, shape.I), dtype=bf, device="cuda")}
    if shape.I_s:
        g.update(dWs_up=torch.empty((shape.I_s, shape.D), dtype=bf, device="cuda"),
                 dWs_gate=torch.empty((shape.I_s, shape.D), dtype=bf, device="cuda"),
                 dWs_down=torch.empty((shape.D, shape.I_s), dtype=bf, device="cuda"))
    wsb = rg.moe_bwd_workspace_bytes(run.plan, T)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")

    def step():
        run.step()
        rg.moe_bwd(run.plan, T, run.x, run.w, dO, run.ws, g, ws, wsb, stream=run.stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    if rg.moe_get_status(run.plan, ws, stream=run.stream) != 0:
        raise SystemExit("backward: device status after warm-up")
    fev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    bev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    for e in [x for ev in fev + bev for x in ev]:
        e.record(run.stream)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.3)
    start.record(run.stream)
    for i in range(steps):
        rg.moe_plan_set_timing_events(run.plan, fev[i])
        rg.moe_plan_set_bwd_timing_events(run.plan, bev[i])
        step()
    end.record(run.stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    rg.moe_plan_set_timing_events(run.plan, None)
    rg.moe_plan_set_bwd_timing_events(run.plan, None)
    if rg.moe_get_status(run.plan, ws, stream=run.stream) != 0:
        raise SystemExit("backward: device status in the timed region")
    el = start.elapsed_time(end)
    mean = lambda xs: sum(xs) / len(xs)
    ph = {"gather": mean([b[0].elapsed_time(b[1]) for b in bev]),
          "replay_and_activation_grad_gemm": mean([b[1].elapsed_time(b[2]) for b in bev]),
          "input_and_weight_grad_gemm": mean([b[2].elapsed_time(b[3]) for b in bev]),
          "router_and_dx_combine": mean([b[3].elapsed_time(b[4]) for b in bev])}
    bwd_ms = mean([b[0].elapsed_time(b[4]) for b in bev])
    fwd_ms = mean([f[0].elapsed_time(f[3]) for f in fev])
    f0, f1 = backward_flops(shape)
    fl_fwd = shape.flops()
    roof = {}
    for name, fl, ms in (("bwd_gemm_phase0", f0, ph["replay_and_activation_grad_gemm"]),
                         ("bwd_gemm_phase1", f1, ph["input_and_weight_grad_gemm"])):
        ach = fl / (ms / 1000.0) / 1e12
        roof[name] = {"kernel": name, "bound": "tensor", "achieved": ach, "peak": bf16_peak, "unit": "TFLOP/s",
                      "frac": ach / bf16_peak, "frac_of_burst_peak": ach / burst_peak,
                      "flops_per_launch": fl, "ms": ms,
                      "peak_source": f"{peak_src} bf16 sustained"}
    del ws, g
    return {"workload": f"{shape.name}: forward + backward (every gradient), dO ~ N(0, 1) seeded",
            "fwd_bwd_tokens_per_s": T * steps / (el / 1000.0), "ms_per_step": el / steps,
            "fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "bwd_phases_ms": ph,
            "bwd_tflops_pages_convention": 2.0 * fl_fwd / (bwd_ms / 1000.0) / 1e12,
            "bwd_tflops_executed": (f0 + f1) / (bwd_ms / 1000.0) / 1e12,
            "bwd_flops_note": "pages: backward = 2x the forward's 6T(k+1)DI; executed adds the replayed "
                              "up/gate projections (16 T k D I + 16 T D I_s in all)",
            "roofline": roof, "gpu_launches_per_step": run.launches + 8, "clocks": clocks}


def scheduling_comparison(run, steps, warmup):
    """The one-CTA persistent kernel with its units claimed by the cooperative
    grid from the global counter, against the same kernel scheduled by cluster
    launch control (MoK Sec. 3.4: one CTA per task launched, running CTAs
    cancel pending launches and take their tokens).  Same weights; the outputs
    are bitwise equal (tests/test_gpu_clc.py)."""
    out = {}
    for name, clc in (("counter", 0), ("cluster_launch_control", 1)):
        r = Runner(run.rg, run.torch, run.shape, run.inp, run.args, run.world, share=run, mma_pair=0, clc=clc)
        res = r.timed(steps, warmup)
        out[name] = {"ms_per_step": res["elapsed_ms"] / steps, "megakernel_ms": statistics.mean(res["mega_ms"]),
                     "tokens_per_s": run.shape.T * steps / (res["elapsed_ms"] / 1000.0)}
        del r
    out["note"] = "one CTA per tile (mma_pair 0), the dispatch of the main line"
    return out


def run_route_only(args):
    """The routing stage alone (router GEMM + top-k + g, then the schedule) on
    the workload's x and router weights, through moe_route_static: a small
    device footprint (x and W_r only) for profiling the router kernel."""
    import torch
    import routing_grouped_expert_gemm_gb300 as rg
    from routing_grouped_expert_gemm_gb300 import build as rgbuild
    rgbuild.build()
    shape = mi.CONFIGS[args.workload]
    inp = mi.make_inputs(shape, weights=False)
    T = min(shape.T, rg.MOE_ROUTE_STATIC_MAX_TOKENS)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    x, wr = dev(inp.x[:T]), dev(inp.w_router)
    b = None if inp.b_router is None else torch.from_numpy(inp.b_router).cuda()
    plan = rg.moe_plan_create(T, shape.D, shape.I, shape.E, shape.k, shape.I_s, score_fn=shape.score)
    i32 = dict(dtype=torch.int32, device="cuda")
    o = [torch.empty((T, shape.k), **i32), torch.empty((T, shape.k), dtype=torch.float32, device="cuda"),
         torch.empty(shape.E, **i32), torch.empty(shape.E + 1, **i32), torch.empty((T * shape.k, 3), **i32),
         torch.empty(T * shape.k, **i32)]
    for _ in range(args.warmup):
        rg.moe_route_static(plan, T, x, wr, b, *o)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        rg.moe_route_static(plan, T, x, wr, b, *o)
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) / args.steps * 1000.0
    print(json.dumps({"route_only": shape.name, "T": T, "us_per_call": us,
                      "x_read_GB/s": T * shape.D * 2 / (us * 1e-6) / 1e9}), flush=True)
    return 0


def run_ours(args, world, rank, local):
    import torch
    import routing_grouped_expert_gemm_gb300 as rg
    from routing_grouped_expert_gemm_gb300 import build as rgbuild

    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    rgbuild.build()

    def allmax(v):
        return reduce_max(v, world)

    peaks, peak_src = load_peaks()
    bf16_peak = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
    burst_peak = float(peaks["bf16_tflops"])
    hbm_peak = float(peaks["hbm_gbs"])

    t_gen = time.perf_counter()
    shape, inp = select_workload(args)
    t_gen = time.perf_counter() - t_gen
    run = Runner(rg, torch, shape, inp, args, world)
    res = run.timed(args.steps, args.warmup, ClockSampler(local))
    e2e = None if args.no_e2e else run.e2e(args.steps)
    e2e_serial = None if args.no_e2e else run.e2e(args.steps, pipelined=False)
    T = shape.T
    elapsed_ms = allmax(res["elapsed_ms"])
    if e2e:
        e2e["ms"] = allmax(e2e["ms"])
        e2e_serial["ms"] = allmax(e2e_serial["ms"])
    flops = shape.flops(T)
    mega_mean = sum(res["mega_ms"]) / len(res["mega_ms"])
    cfg = workload_config(shape, args)
    roof = attach_traffic(tensor_roofline(shape, mega_mean, bf16_peak, peak_src, burst_peak), shape, cfg)
    line = {
        "metric": METRIC,
        "value": replica_throughput(world, T, args.steps, elapsed_ms), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if shape.precision == "bf16" else "mxfp8 (e4m3 + e8m0) routed, bf16 shared",
        "data": "synthetic (seeded normal inputs, random-init weights)",
        "config": cfg,
        "tflops": world * flops * args.steps / (elapsed_ms / 1000.0) / 1e12,
        "ms_median_step": statistics.median(res["step_ms"]),
        "phases_ms_mean": {"router_topk": statistics.mean(res["router_ms"]),
                           "schedule": statistics.mean(res["sched_ms"]), "megakernel": mega_mean},
        "roofline": roof,
        "phase_bandwidth": phase_bandwidths(shape, res, hbm_peak),
        "gpu_launches": run.launches * args.steps,
        "clocks": res["clocks"],
        "input_generation_s": t_gen,
    }
    line["tflops_frac_of_peak"] = line["tflops"] / (world * roof["peak"])
    if e2e:
        # copies on a second stream overlap the neighbouring steps' forwards;
        # "serial": copy in, forward, copy out one after the other
        line["e2e"] = {"value": replica_throughput(world, T, args.steps, e2e["ms"]), "unit": "tokens/s",
                       "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                       "copies": "pipelined: input copies, forwards, output copies on three streams, "
                                 "two device input/output buffers",
                       "serial_value": replica_throughput(world, T, args.steps, e2e_serial["ms"])}
    sweep_steps = max(3, args.steps // 4)
    full_size = not (args.tokens or args.experts)
    if not args.no_backward and shape.precision == "bf16":
        line["backward"] = backward_timing(run, max(3, args.steps // 2), 3, bf16_peak, burst_peak, peak_src,
                                           ClockSampler(local))
    if not args.no_sweep and full_size:
        line["minibatch_sweep"] = minibatch_sweep(run, sweep_steps, 3)
        line["scheduling"] = scheduling_comparison(run, sweep_steps, 3)
    cpu = None
    if world == 1 and not args.no_cpu_baseline and rank == 0:
        cb = time_oracle(inp, args.cpu_seconds)
        cpu = {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")}
        line["cpu_baseline"] = cpu
    del run
    torch.cuda.empty_cache()

    # the same layer in MXFP8 (routed experts), its own seeded inputs, uniform routing
    if not args.no_mxfp8 and args.workload == "dsv3" and full_size:
        mshape = mi.CONFIGS["dsv3_mxfp8"]
        minp = mi.make_inputs(mshape)
        mrun = Runner(rg, torch, mshape, minp, args, world)
        mres = mrun.timed(args.steps, args.warmup, ClockSampler(local))
        m_el = allmax(mres["elapsed_ms"])
        m_mega = statistics.mean(mres["mega_ms"])
        line["mxfp8"] = {
            "workload": "dsv3_mxfp8: DSV3 shape, uniform routing, routed experts MXFP8, shared expert BF16",
            "value": replica_throughput(world, mshape.T, args.steps, m_el), "unit": "tokens/s",
            "ms_per_step": m_el / args.steps, "tflops": world * mshape.flops() * args.steps / (m_el / 1000.0) / 1e12,
            "config": workload_config(mshape, args),
            "phases_ms_mean": {"router_topk": statistics.mean(mres["router_ms"]),
                               "schedule": statistics.mean(mres["sched_ms"]), "megakernel": m_mega},
            "roofline": attach_traffic(tensor_roofline(mshape, m_mega, bf16_peak, peak_src, burst_peak), mshape,
                                       workload_config(mshape, args)),
            "phase_bandwidth": phase_bandwidths(mshape, mres, hbm_peak),
            "gpu_launches": mrun.launches * args.steps,
            "clocks": mres["clocks"],
        }
        if not args.no_sweep:
            line["mxfp8"]["minibatch_sweep"] = minibatch_sweep(mrun, sweep_steps, 3)
        del mrun
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    world, rank, local = dist_setup(args.gpus)
    if args.impl == "reference":
        return run_reference(args, world, rank)
    if args.route_only:
        return run_route_only(args)
    return run_ours(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
