"""Seeded synthetic inputs for the MoE-layer forward (shared by the CUDA path's
tests/bench and by the fp64 oracle's tests).

This module holds no arithmetic of the MoE method: it draws standard-normal
values from a counter-based generator (``gen.c``), scales them by 1/sqrt(fan_in)
and rounds them to bf16.  The router bias that shapes the expert load and the
list of x rows that were redrawn (the top-k gap rule) are *data*, read from
``tests/golden/router_calibration.json``; that file is written by
``tests/golden/make_router_calibration.py``, which calls only the oracle.

Workloads (Mixture-of-Kittens: MoE Megakernel for NVL72s, Sec. 4.1: router
logits and inputs drawn from a standard normal; shapes from Sec. 4.1 and the
DeepSeek-V3-style layer of the vendor blog post):

=============  =====  ====  ====  ===  ==  ====  ========  ==========
name             T     D     I     E   k   I_s   score     load
=============  =====  ====  ====  ===  ==  ====  ========  ==========
tiny            256   256   128   16   4   128   sigmoid   uniform
qwen3          8192  4096  1536  128   8     0   softmax   uniform
dsv3          16384  7168  2048  256   8  2048   sigmoid   Zipf(1.1)
dsv3_mxfp8    16384  7168  2048  256   8  2048   sigmoid   uniform
kimi_k2       32768  7168  2048  384   8  2048   sigmoid   uniform
=============  =====  ====  ====  ===  ==  ====  ========  ==========

x ~ N(0,1); W_up, W_gate, W_r ~ N(0, 1/D); W_down ~ N(0, 1/I); shared-expert
weights likewise with I_s.  Seeds are ``20261202 + config_id``.
"""
from __future__ import annotations

import ctypes
import json
import math
import os
import subprocess
import sys
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_REPO = os.path.dirname(_HERE)
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_LIB_DIR, "libmoe_inputs.so")
CALIBRATION_PATH = os.path.join(_REPO, "tests", "golden", "router_calibration.json")

# tensor ids of the counter-based streams
TID_X, TID_WR, TID_WUP, TID_WGATE, TID_WDOWN = 1, 2, 3, 4, 5
TID_WS_UP, TID_WS_GATE, TID_WS_DOWN = 6, 7, 8
TID_DOUT = 9  # upstream gradient dL/d out of a backward pass
SEED_BASE = 20261202


@dataclass(frozen=True)
class MoEShape:
    name: str
    T: int
    D: int
    I: int
    E: int
    k: int
    I_s: int
    score: str  # "sigmoid" | "softmax"
    load: str  # "uniform" | "zipf"
    precision: str = "bf16"  # "bf16" | "mxfp8"
    config_id: int = 0
    zipf_s: float = 1.1

    @property
    def seed(self) -> int:
        return SEED_BASE + self.config_id

    @property
    def routes(self) -> int:
        return self.T * self.k

    @property
    def n_shared(self) -> int:
        return 1 if self.I_s > 0 else 0

    def flops(self, T: int | None = None) -> float:
        """Expert-FFN FLOPs of one forward: 6 T (k + n_shared) D I (Sec. 4.1)."""
        T = self.T if T is None else T
        routed = 6.0 * T * self.k * self.D * self.I
        shared = 6.0 * T * self.D * self.I_s
        return routed + shared


CONFIGS: dict[str, MoEShape] = {
    "tiny": MoEShape("tiny", 256, 256, 128, 16, 4, 128, "sigmoid", "uniform", config_id=0),
    "qwen3": MoEShape("qwen3", 8192, 4096, 1536, 128, 8, 0, "softmax", "uniform", config_id=1),
    "dsv3": MoEShape("dsv3", 16384, 7168, 2048, 256, 8, 2048, "sigmoid", "zipf", config_id=2),
    "dsv3_mxfp8": MoEShape("dsv3_mxfp8", 16384, 7168, 2048, 256, 8, 2048, "sigmoid", "uniform",
                           precision="mxfp8", config_id=3),
    "kimi_k2": MoEShape("kimi_k2", 32768, 7168, 2048, 384, 8, 2048, "sigmoid", "uniform", config_id=4),
    # The pages' four evaluated layer shapes (one shared expert each; its width
    # is not given, read as I), 16384 tokens on one GPU, uniform routing; the
    # _mxfp8 twins draw the same inputs (same config_id) with MXFP8 routed experts.
    "kimi_k27": MoEShape("kimi_k27", 16384, 7168, 2048, 384, 8, 2048, "sigmoid", "uniform", config_id=5),
    "glm52": MoEShape("glm52", 16384, 6144, 2048, 256, 8, 2048, "sigmoid", "uniform", config_id=6),
    "qwen35": MoEShape("qwen35", 16384, 4096, 1024, 512, 10, 1024, "sigmoid", "uniform", config_id=7),
    "dsv4pro": MoEShape("dsv4pro", 16384, 7168, 3072, 384, 6, 3072, "sigmoid", "uniform", config_id=8),
}
for _n in ("kimi_k27", "glm52", "qwen35", "dsv4pro"):
    _b = CONFIGS[_n]
    CONFIGS[_n + "_mxfp8"] = MoEShape(_n + "_mxfp8", _b.T, _b.D, _b.I, _b.E, _b.k, _b.I_s, _b.score, _b.load,
                                      precision="mxfp8", config_id=_b.config_id)


# --------------------------------------------------------------------------- build / load
_lib = None


def build(verbose: bool = False) -> str:
    """Compile gen.c into moe_inputs/_build/libmoe_inputs.so (gcc, OpenMP if present)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    src = os.path.join(_HERE, "gen.c")
    base = ["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-std=c11", src, "-o", _LIB_PATH, "-lm"]
    for extra in (["-fopenmp"], []):
        cmd = base[:1] + extra + base[1:]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            if verbose:
                print(" ".join(cmd))
            return _LIB_PATH
    raise RuntimeError("building moe_inputs failed:\n" + r.stderr)


def _load():
    global _lib
    if _lib is not None:
        return _lib
    src = os.path.join(_HERE, "gen.c")
    if not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
        build()
    lib = ctypes.CDLL(_LIB_PATH)
    u64, i64, dbl, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
    lib.gen_normal_bf16.argtypes = [u64, u64, u64, u64, dbl, vp]
    lib.gen_normal_f64.argtypes = [u64, u64, u64, u64, dbl, vp]
    lib.gen_rows_bf16.argtypes = [u64, u64, i64, i64, i64, vp, dbl, vp]
    lib.gen_num_threads.restype = ctypes.c_int
    _lib = lib
    return lib


def num_threads() -> int:
    return int(_load().gen_num_threads())


# --------------------------------------------------------------------------- raw draws
def normal_bf16(seed: int, tid: int, n: int, scale: float = 1.0, start: int = 0,
                out: np.ndarray | None = None) -> np.ndarray:
    """bf16 bit patterns (uint16) of scale * N(0,1) draws n..; C-contiguous."""
    if out is None:
        out = np.empty(n, dtype=np.uint16)
    assert out.dtype == np.uint16 and out.flags.c_contiguous and out.size == n
    _load().gen_normal_bf16(seed, tid, start, n, scale, out.ctypes.data)
    return out


def normal_f64(seed: int, tid: int, n: int, scale: float = 1.0, start: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _load().gen_normal_f64(seed, tid, start, n, scale, out.ctypes.data)
    return out


def x_rows(seed: int, T: int, D: int, attempt: np.ndarray | None, row0: int = 0,
           rows: int | None = None, out: np.ndarray | None = None) -> np.ndarray:
    """Rows [row0, row0+rows) of x (uint16 bf16 bits, shape [rows, D])."""
    rows = T - row0 if rows is None else rows
    if out is None:
        out = np.empty((rows, D), dtype=np.uint16)
    assert out.dtype == np.uint16 and out.flags.c_contiguous and out.size == rows * D
    att = None
    if attempt is not None:
        attempt = np.ascontiguousarray(attempt, dtype=np.int32)
        assert attempt.size == T
        att = attempt.ctypes.data
    _load().gen_rows_bf16(seed, TID_X, row0, rows, D, att, 1.0, out.ctypes.data)
    return out


def bf16_bits_to_f32(a: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float32."""
    return (a.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest-even) and return bit patterns (uint16)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


# --------------------------------------------------------------------------- load shaping
def zipf_targets(E: int, routes: int, cap: int, s: float) -> np.ndarray:
    """Per-expert route counts following Zipf(s) over ranks 1..E (expert id =
    rank - 1), water-filled so that no expert exceeds ``cap`` (a token picks an
    expert at most once, so at most T routes reach one expert); integer counts
    summing to ``routes`` by largest remainder."""
    w = np.array([1.0 / (r ** s) for r in range(1, E + 1)])
    capped = np.zeros(E, dtype=bool)
    tgt = np.zeros(E)
    while True:
        remaining = routes - cap * capped.sum()
        free = ~capped
        tgt = np.where(capped, float(cap), remaining * w / w[free].sum())
        over = free & (tgt > cap)
        if not over.any():
            break
        capped |= over
    base = np.floor(tgt).astype(np.int64)
    short = routes - int(base.sum())
    order = np.argsort(-(tgt - base), kind="stable")
    base[order[:short]] += 1
    return base


def load_calibration(name: str) -> dict:
    """Router bias and redrawn-row attempts for workload ``name`` (see
    tests/golden/make_router_calibration.py)."""
    if not os.path.exists(CALIBRATION_PATH):
        raise FileNotFoundError(CALIBRATION_PATH)
    with open(CALIBRATION_PATH) as f:
        data = json.load(f)
    if name not in data:
        raise KeyError(f"no calibration for workload {name!r} in {CALIBRATION_PATH}")
    return data[name]


# --------------------------------------------------------------------------- full input sets
@dataclass
class MoEInputs:
    shape: MoEShape
    T: int
    x: np.ndarray  # uint16 [T, D]
    w_router: np.ndarray  # uint16 [E, D]
    b_router: np.ndarray | None  # float32 [E] or None
    w_up: np.ndarray | None = None  # uint16 [E, I, D]
    w_gate: np.ndarray | None = None
    w_down: np.ndarray | None = None  # uint16 [E, D, I]
    ws_up: np.ndarray | None = None  # uint16 [I_s, D]
    ws_gate: np.ndarray | None = None
    ws_down: np.ndarray | None = None  # uint16 [D, I_s]
    attempt: np.ndarray | None = None  # int32 [T_full]
    meta: dict = field(default_factory=dict)


def expert_weights(seed: int, D: int, I: int, which: str, e0: int, ne: int) -> np.ndarray:
    """Experts [e0, e0+ne) of W_up / W_gate ([ne, I, D]) or W_down ([ne, D, I])."""
    if which == "up":
        tid, inner, scale = TID_WUP, (I, D), 1.0 / math.sqrt(D)
    elif which == "gate":
        tid, inner, scale = TID_WGATE, (I, D), 1.0 / math.sqrt(D)
    elif which == "down":
        tid, inner, scale = TID_WDOWN, (D, I), 1.0 / math.sqrt(I)
    else:
        raise ValueError(which)
    per = inner[0] * inner[1]
    out = np.empty((ne,) + inner, dtype=np.uint16)
    normal_bf16(seed, tid, ne * per, scale, start=e0 * per, out=out.reshape(-1))
    return out


def make_inputs(shape: MoEShape | str, T: int | None = None, weights: bool = True,
                calibration: dict | None = None, seed: int | None = None) -> MoEInputs:
    """Draw a workload's inputs.  ``T`` < shape.T takes the first T tokens of the
    full workload (the same rows, bit for bit).  ``calibration`` overrides the
    stored router bias / redraw list (used by the calibration script itself and
    by unit tests on random shapes); ``seed`` overrides the workload seed."""
    if isinstance(shape, str):
        shape = CONFIGS[shape]
    T = shape.T if T is None else T
    seed = shape.seed if seed is None else seed
    if calibration is None:
        try:
            calibration = load_calibration(shape.name)
        except (FileNotFoundError, KeyError):
            if shape.load == "zipf":
                raise
            calibration = {"beta": None, "redraw": {}}
    T_full = max(shape.T, T)
    attempt = np.zeros(T_full, dtype=np.int32)
    for t, a in calibration.get("redraw", {}).items():
        if int(t) < T_full:
            attempt[int(t)] = int(a)
    D, I, E, I_s = shape.D, shape.I, shape.E, shape.I_s
    x = x_rows(seed, T_full, D, attempt, 0, T)
    w_router = normal_bf16(seed, TID_WR, E * D, 1.0 / math.sqrt(D)).reshape(E, D)
    beta = calibration.get("beta")
    b_router = None if beta is None else np.asarray(beta, dtype=np.float32)
    inp = MoEInputs(shape, T, x, w_router, b_router, attempt=attempt,
                    meta={"seed": seed, "calibration": {k: v for k, v in calibration.items() if k != "redraw"}})
    if weights:
        inp.w_up = expert_weights(seed, D, I, "up", 0, E)
        inp.w_gate = expert_weights(seed, D, I, "gate", 0, E)
        inp.w_down = expert_weights(seed, D, I, "down", 0, E)
        if I_s > 0:
            inp.ws_up = normal_bf16(seed, TID_WS_UP, I_s * D, 1.0 / math.sqrt(D)).reshape(I_s, D)
            inp.ws_gate = normal_bf16(seed, TID_WS_GATE, I_s * D, 1.0 / math.sqrt(D)).reshape(I_s, D)
            inp.ws_down = normal_bf16(seed, TID_WS_DOWN, D * I_s, 1.0 / math.sqrt(I_s)).reshape(D, I_s)
    return inp


def grad_out(shape: MoEShape | str, T: int | None = None, seed: int | None = None) -> np.ndarray:
    """Upstream gradient dL/d out of a backward pass: bf16 bit patterns of
    N(0, 1) draws, [T, D], rows 0..T-1 of the workload's full [shape.T, D]
    draw (the same rows for any T)."""
    if isinstance(shape, str):
        shape = CONFIGS[shape]
    T = shape.T if T is None else T
    seed = shape.seed if seed is None else seed
    return normal_bf16(seed, TID_DOUT, T * shape.D).reshape(T, shape.D)


def custom_shape(T: int, D: int, I: int, E: int, k: int, I_s: int, score: str = "sigmoid",
                 config_id: int = 100, precision: str = "bf16") -> MoEShape:
    """An ad-hoc shape for unit tests (uniform load, no stored calibration)."""
    return MoEShape(f"custom_{config_id}", T, D, I, E, k, I_s, score, "uniform",
                    precision=precision, config_id=config_id)
