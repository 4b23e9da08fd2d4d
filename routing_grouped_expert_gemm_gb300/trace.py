"""Per-role timing of the persistent kernel (the MOE_TRACE build).

    python -m routing_grouped_expert_gemm_gb300.trace [workload] ['{"gather_ctas": 8, ...}']

Builds the MOE_TRACE variant of the library (every wait of the persistent
kernel timed with clock64 in registers and added to per-CTA slots once, at
the end), runs a few forwards of a seeded workload from moe_inputs and
prints, per role, the mean and maximum time per CTA spent in each kind of
wait or epilogue (BF16 or MXFP8 workloads; clock64 cycles converted at the SM
clock measured over the run), plus the mean time from a stage's TMA issue to
its full barrier being seen by the MMA issuer.  The timed waits perturb the kernel a
little: use it to see where time goes, not for throughput figures.
"""
from __future__ import annotations

import json
import os
import sys

# the trace variant must be chosen before the package loads its library
os.environ["MOE_TRACE_BUILD"] = "1"

NAMES = ["start", "end", "prod_dep", "prod_empty", "mma_full", "mma_tempty", "epi_tfull", "epi_busy",
         "gather_wait", "gather_busy", "final_wait", "last_task", "epi_R1", "epi_R2", "epi_S1", "epi_S2",
         "tma_lat_ns", "tma_stages", "g_loadwait", "g_storewait", "start_clk", "end_clk", "combine"]
SLOTS = len(NAMES)  # the kernel's TRACE_SLOTS


def main(argv: list[str]) -> int:
    import numpy as np
    import torch

    import moe_inputs as mi
    import routing_grouped_expert_gemm_gb300 as rg
    from routing_grouped_expert_gemm_gb300 import build

    # `python -m` imports the package (and fixes its library path) before this
    # module runs: point it at the trace variant before the library is loaded
    rg.LIB_PATH = build.build(trace=True)
    if rg._lib is not None and rg._lib._name != rg.LIB_PATH:
        raise SystemExit("trace: the regular library is already loaded in this process")
    name = argv[0] if argv else "dsv3"
    cfg = json.loads(argv[1]) if len(argv) > 1 else {}
    shape = mi.CONFIGS[name]
    inp = mi.make_inputs(shape)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    w = {"W_router": dev(inp.w_router),
         "b_router": None if inp.b_router is None else torch.from_numpy(inp.b_router).cuda(),
         "W_up": dev(inp.w_up), "W_gate": dev(inp.w_gate), "W_down": dev(inp.w_down)}
    if shape.I_s:
        w.update(Ws_up=dev(inp.ws_up), Ws_gate=dev(inp.ws_gate), Ws_down=dev(inp.ws_down))
    x = dev(inp.x)
    T = shape.T
    out = torch.empty((T, shape.D), dtype=torch.bfloat16, device="cuda")
    plan = rg.moe_plan_create(T, shape.D, shape.I, shape.E, shape.k, shape.I_s, score_fn=shape.score,
                              precision=shape.precision, **cfg)
    if shape.precision == "mxfp8":  # routed weights as E4M3 codes + block scales
        for nm, rows, K in (("W_up", shape.E * shape.I, shape.D), ("W_gate", shape.E * shape.I, shape.D),
                            ("W_down", shape.E * shape.D, shape.I)):
            q = torch.empty((rows, K), dtype=torch.uint8, device="cuda")
            sc = torch.empty(rg.moe_mxfp8_scale_bytes(rows, K), dtype=torch.uint8, device="cuda")
            rg.moe_quantize_mxfp8(plan, w[nm], rows, K, q, sc)
            torch.cuda.synchronize()
            w[nm], w[nm + "_scale"] = q, sc
        torch.cuda.empty_cache()
    wsb = rg.moe_workspace_bytes(plan, T)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    for _ in range(4):
        rg.moe_fwd(plan, T, x, w, out, ws, wsb)
    torch.cuda.synchronize()
    status = rg.moe_get_status(plan, ws)
    print("status", status)
    # the trace slots are the last section of the workspace: [1024 CTAs, SLOTS] int64
    tr = ws[wsb - SLOTS * 1024 * 8:].view(torch.int64).view(1024, SLOTS).cpu().numpy()
    tr = tr[tr[:, 0] != 0]  # CTAs that ran
    start = tr[:, 0].min()
    dur_us = (tr[:, 1] - start) / 1e3
    # clock64 cycles per us over each CTA's run: the SM clock it actually ran at
    clk = float(np.median((tr[:, 21] - tr[:, 20]) / np.maximum(tr[:, 1] - tr[:, 0], 1) * 1e3))
    print("kernel span us: max %.0f  min %.0f   SM clock %.0f MHz" % (dur_us.max(), dur_us.min(), clk))
    G = cfg.get("gather_ctas", 8) if cfg.get("dispatch", "ring") == "ring" else 0
    for label, rows in (("gather", tr[:G]), ("gemm", tr[G:])):
        if len(rows) == 0:
            continue
        print(label)
        for i in list(range(2, 16)) + [18, 19, 22]:
            if i == 11:
                continue
            v = rows[:, i] / clk
            v = v[v > 0] if (v > 0).any() else v
            if v.max() > 0:
                print("  %-12s mean %8.0f us  max %8.0f" % (NAMES[i], v.mean(), v.max()))
        lat, n = rows[:, 16], rows[:, 17]
        if n.sum() > 0:
            print("  tma issue->full seen: mean %.2f us over %d stages" % (lat.sum() / n.sum() / 1e3, n.sum()))
        ends = (rows[:, 1] - start) / 1e3
        print("  end (us from first start): mean %.0f min %.0f max %.0f" % (ends.mean(), ends.min(), ends.max()))
    return 0 if status == 0 else 1


if __name__ == "__main__":
    sys.exit(main(sys.argv[1:]))
