"""Writes tests/golden/router_calibration.json: per workload, the router bias
and the list of x rows redrawn by the top-k gap rule.  Calls only the oracle
(for the fp64 router logits) and the seeded input generator.

Input recipe (synthetic stand-in for the pages' standard-normal router logits
and inputs, "Mixture-of-Kittens: MoE Megakernel for NVL72s" Sec. 4.1):
  * uniform-load workloads keep beta = None (no bias);
  * the Zipf workload ("dsv3") targets per-expert route counts that follow
    Zipf(1.1) over expert ids, water-filled with cap T, and finds beta by a
    fixed number of deterministic steps beta_e += 0.5 (ln(target_e + 1) -
    ln(count_e + 1)), counts taken from the top-k of the biased fp64 logits;
    beta is then rounded to fp32 (the precision the library takes it in);
  * gap rule: a token whose k-th and (k+1)-th biased logits differ by less than
    1e-3 gets its x row redrawn from the stream (seed, x | attempt << 32),
    attempt = 1, 2, ... until the gap holds.  The top-k is then decided
    identically in fp32 and fp64.

Usage: python tests/golden/make_router_calibration.py [workload ...]
"""
import json
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import moe_inputs as mi  # noqa: E402
import oracle  # noqa: E402

GAP = 1e-3
ZIPF_STEPS = 400


def topk_counts(logits_b, k, E):
    sel = np.argpartition(-logits_b, k - 1, axis=1)[:, :k]
    return np.bincount(sel.reshape(-1), minlength=E)


def kth_gap(logits_b, k):
    part = -np.partition(-logits_b, k, axis=1)[:, :k + 1]
    part.sort(axis=1)
    return part[:, 1] - part[:, 0]  # (k-th largest) - ((k+1)-th largest)


def calibrate(name):
    shape = mi.CONFIGS[name]
    T, D, E, k = shape.T, shape.D, shape.E, shape.k
    t0 = time.time()
    attempt = np.zeros(T, dtype=np.int32)
    x = mi.x_rows(shape.seed, T, D, attempt)
    wr = mi.make_inputs(shape, T=1, weights=False, calibration={"beta": None, "redraw": {}}).w_router
    logits = oracle.router_logits(x, wr, None)
    rec = {"seed": shape.seed, "T": T, "E": E, "k": k, "gap": GAP}
    beta = None
    if shape.load == "zipf":
        target = mi.zipf_targets(E, T * k, T, shape.zipf_s)
        b = np.zeros(E)
        for _ in range(ZIPF_STEPS):
            cnt = topk_counts(logits + b, k, E)
            b += 0.5 * (np.log(target + 1.0) - np.log(cnt + 1.0))
        beta = b.astype(np.float32)
        rec["zipf_s"] = shape.zipf_s
        rec["zipf_steps"] = ZIPF_STEPS
        rec["target_counts"] = target.tolist()
    bb = np.zeros(E) if beta is None else beta.astype(np.float64)
    redraw = {}
    for _round in range(50):
        bad = np.nonzero(kth_gap(logits + bb, k) < GAP)[0]
        if bad.size == 0:
            break
        for t in bad:
            attempt[t] += 1
            redraw[int(t)] = int(attempt[t])
        rows = np.stack([mi.x_rows(shape.seed, T, D, attempt, int(t), 1)[0] for t in bad])
        logits[bad] = oracle.router_logits(rows, wr, None)
    else:
        raise RuntimeError("gap rule did not converge")
    rec["beta"] = None if beta is None else [float(v) for v in beta]
    rec["redraw"] = {str(t): a for t, a in sorted(redraw.items())}
    rec["histogram"] = topk_counts(logits + bb, k, E).tolist()
    rec["min_gap"] = float(kth_gap(logits + bb, k).min())
    print(f"{name}: {len(redraw)} rows redrawn, min gap {rec['min_gap']:.3g}, "
          f"max count {max(rec['histogram'])}, min count {min(rec['histogram'])}, {time.time() - t0:.0f}s",
          flush=True)
    return rec


def main(names):
    path = os.path.join(HERE, "router_calibration.json")
    data = {}
    if os.path.exists(path):
        with open(path) as f:
            data = json.load(f)
    for name in names:
        data[name] = calibrate(name)
        with open(path, "w") as f:
            json.dump(data, f, indent=1, sort_keys=True)


if __name__ == "__main__":
    main(sys.argv[1:] or ["tiny", "qwen3", "dsv3", "dsv3_mxfp8", "kimi_k2"])
