"""fp64 CPU oracle for the MoE-layer forward -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg import this package.  The CUDA library never does, and this package never
imports the CUDA library: the two share no code.  Only the seeded input
generator (``moe_inputs``) serves both.

The arithmetic lives in ``moe_oracle.c`` (plain loops in fp64, OpenMP over
tokens), ``alg1.py`` (Algorithm 1 for any number of ranks) and ``backward.py``
(the layer's backward pass by the chain rule, fp64 numpy, pinned in
``tests/test_oracle_backward.py``).  Every function
follows "Mixture-of-Kittens: MoE Megakernel for NVL72s" as cited in those
files.  Parity status of each function (what pins it) is listed in the tests
``tests/test_oracle_pins.py``; absolute layer values beyond those pins have no
printed worked example in the source pages.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from .alg1 import alg1_schedule, sort_key_schedule  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_LIB_DIR, "liboracle.so")

SCORE = {"sigmoid": 0, "softmax": 1}


def build(verbose: bool = False) -> str:
    """Compile moe_oracle.c into oracle/_build/liboracle.so with gcc."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    src = os.path.join(_HERE, "moe_oracle.c")
    base = ["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
            src, "-o", _LIB_PATH, "-lm"]
    err = ""
    for extra in (["-fopenmp"], []):
        cmd = base[:1] + extra + base[1:]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            if verbose:
                print(" ".join(cmd))
            return _LIB_PATH
        err = r.stderr
    raise RuntimeError("building the oracle failed:\n" + err)


class _Layer(ctypes.Structure):
    _fields_ = [
        ("D", ctypes.c_int64), ("I", ctypes.c_int64), ("E", ctypes.c_int64),
        ("k", ctypes.c_int64), ("I_s", ctypes.c_int64), ("score_fn", ctypes.c_int),
        ("x", ctypes.c_void_p), ("Wr", ctypes.c_void_p), ("beta", ctypes.c_void_p),
        ("Wup", ctypes.c_void_p), ("Wgate", ctypes.c_void_p), ("Wdown", ctypes.c_void_p),
        ("Wup_q", ctypes.c_void_p), ("Wup_s", ctypes.c_void_p),
        ("Wgate_q", ctypes.c_void_p), ("Wgate_s", ctypes.c_void_p),
        ("Wdown_q", ctypes.c_void_p), ("Wdown_s", ctypes.c_void_p),
        ("mx", ctypes.c_int),
        ("Ws_up", ctypes.c_void_p), ("Ws_gate", ctypes.c_void_p), ("Ws_down", ctypes.c_void_p),
    ]


_lib = None


def _load():
    global _lib
    if _lib is not None:
        return _lib
    src = os.path.join(_HERE, "moe_oracle.c")
    if not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
        build()
    lib = ctypes.CDLL(_LIB_PATH)
    i64, vp = ctypes.c_int64, ctypes.c_void_p
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_router_logits.argtypes = [vp, i64, vp, i64, vp, vp, i64, vp]
    lib.oracle_topk.argtypes = [vp, i64, i64, i64, ctypes.c_int, vp, vp]
    lib.oracle_topk.restype = ctypes.c_int
    lib.oracle_moe_fwd.argtypes = [ctypes.POINTER(_Layer), vp, i64, vp, vp, vp]
    lib.oracle_moe_fwd.restype = ctypes.c_int
    lib.oracle_schedule.argtypes = [vp, i64, i64, i64, vp, vp, vp, vp]
    lib.oracle_schedule.restype = ctypes.c_int
    lib.oracle_mx_quantize_f64.argtypes = [vp, i64, i64, vp, vp]
    lib.oracle_mx_quantize_bf16.argtypes = [vp, i64, i64, vp, vp]
    lib.oracle_mx_dequantize.argtypes = [vp, vp, i64, i64, vp]
    lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_value.restype = ctypes.c_double
    lib.oracle_e4m3_encode.argtypes = [ctypes.c_double]
    lib.oracle_e4m3_encode.restype = ctypes.c_uint8
    _lib = lib
    return lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ router
def router_logits(x, w_router, b_router=None, rows=None) -> np.ndarray:
    """fp64 logits x[t] . W_r[e] + beta[e] for the listed rows of x (bf16 bits)."""
    x, w_router = _c(x, np.uint16), _c(w_router, np.uint16)
    b_router = _c(b_router, np.float32)
    D = x.shape[1]
    E = w_router.shape[0]
    rows = None if rows is None else _c(rows, np.int64)
    n = x.shape[0] if rows is None else rows.size
    out = np.empty((n, E), dtype=np.float64)
    _load().oracle_router_logits(_ptr(x), D, _ptr(rows), n, _ptr(w_router), _ptr(b_router), E, _ptr(out))
    return out


def topk(logits, k: int, score: str = "sigmoid"):
    """(topk_idx int32 [n,k] in ascending expert id, g fp64 [n,k])."""
    logits = _c(logits, np.float64)
    n, E = logits.shape
    idx = np.empty((n, k), dtype=np.int32)
    g = np.empty((n, k), dtype=np.float64)
    rc = _load().oracle_topk(_ptr(logits), n, E, k, SCORE[score], _ptr(idx), _ptr(g))
    if rc != 0:
        raise ValueError("oracle_topk: bad k")
    return idx, g


# ------------------------------------------------------------------ layer
def moe_fwd(shape, x, w_router, b_router, w_up=None, w_gate=None, w_down=None,
            ws_up=None, ws_gate=None, ws_down=None, rows=None, mx=None):
    """fp64 forward for the listed token rows.

    ``mx`` = None (bf16 experts) or a dict with uint8 arrays
    {up_q, up_s, gate_q, gate_s, down_q, down_s} (MXFP8 experts; the token and
    the gated activation are MX-quantised inside).  Returns (out fp64 [n, D],
    topk_idx int32 [n, k], g fp64 [n, k])."""
    x = _c(x, np.uint16)
    D, I, E, k = shape.D, shape.I, shape.E, shape.k
    keep = []

    def hold(a, dt):
        a = _c(a, dt)
        keep.append(a)
        return _ptr(a)

    L = _Layer()
    L.D, L.I, L.E, L.k, L.I_s = D, I, E, k, shape.I_s
    L.score_fn = SCORE[shape.score]
    L.x = hold(x, np.uint16)
    L.Wr = hold(w_router, np.uint16)
    L.beta = hold(b_router, np.float32) if b_router is not None else None
    if mx is None:
        L.mx = 0
        L.Wup, L.Wgate, L.Wdown = hold(w_up, np.uint16), hold(w_gate, np.uint16), hold(w_down, np.uint16)
    else:
        L.mx = 1
        L.Wup_q, L.Wup_s = hold(mx["up_q"], np.uint8), hold(mx["up_s"], np.uint8)
        L.Wgate_q, L.Wgate_s = hold(mx["gate_q"], np.uint8), hold(mx["gate_s"], np.uint8)
        L.Wdown_q, L.Wdown_s = hold(mx["down_q"], np.uint8), hold(mx["down_s"], np.uint8)
    if ws_up is not None:
        L.Ws_up, L.Ws_gate, L.Ws_down = hold(ws_up, np.uint16), hold(ws_gate, np.uint16), hold(ws_down, np.uint16)
    rows_a = None if rows is None else _c(rows, np.int64)
    n = x.shape[0] if rows_a is None else rows_a.size
    out = np.empty((n, D), dtype=np.float64)
    idx = np.empty((n, k), dtype=np.int32)
    g = np.empty((n, k), dtype=np.float64)
    rc = _load().oracle_moe_fwd(ctypes.byref(L), _ptr(rows_a), n, _ptr(out), _ptr(idx), _ptr(g))
    if rc != 0:
        raise ValueError(f"oracle_moe_fwd failed ({rc})")
    return out, idx, g


def moe_fwd_inputs(inp, rows=None, mx=None):
    """moe_fwd on a moe_inputs.MoEInputs bundle."""
    return moe_fwd(inp.shape, inp.x, inp.w_router, inp.b_router, inp.w_up, inp.w_gate, inp.w_down,
                   inp.ws_up, inp.ws_gate, inp.ws_down, rows=rows, mx=mx)


# ------------------------------------------------------------------ schedule
def schedule(topk_idx, E: int):
    """Single-rank Algorithm 1: (M int32[E], S int32[E+1], sched int32[T*k,3], route_row int32[T*k])."""
    topk_idx = _c(topk_idx, np.int32)
    T, k = topk_idx.shape
    M = np.empty(E, dtype=np.int32)
    S = np.empty(E + 1, dtype=np.int32)
    sched = np.empty((T * k, 3), dtype=np.int32)
    route_row = np.empty(T * k, dtype=np.int32)
    rc = _load().oracle_schedule(_ptr(topk_idx), T, k, E, _ptr(M), _ptr(S), _ptr(sched), _ptr(route_row))
    if rc != 0:
        raise ValueError("oracle_schedule: expert index out of range")
    return M, S, sched, route_row


# ------------------------------------------------------------------ MXFP8
def mx_quantize(v, K: int | None = None):
    """OCP MX v1.0 MXFP8 (E4M3, 32-element blocks along the last axis).
    ``v`` is uint16 (bf16 bits) or float64.  Returns (codes uint8, scales uint8)."""
    v = np.asarray(v)
    K = v.shape[-1] if K is None else K
    assert K % 32 == 0
    rows = v.size // K
    q = np.empty(v.shape, dtype=np.uint8)
    s = np.empty(v.shape[:-1] + (K // 32,), dtype=np.uint8)
    if v.dtype == np.uint16:
        v = _c(v, np.uint16)
        _load().oracle_mx_quantize_bf16(_ptr(v), rows, K, _ptr(q), _ptr(s))
    else:
        v = _c(v, np.float64)
        _load().oracle_mx_quantize_f64(_ptr(v), rows, K, _ptr(q), _ptr(s))
    return q, s


def mx_dequantize(q, s) -> np.ndarray:
    q, s = _c(q, np.uint8), _c(s, np.uint8)
    K = q.shape[-1]
    out = np.empty(q.shape, dtype=np.float64)
    _load().oracle_mx_dequantize(_ptr(q), _ptr(s), q.size // K, K, _ptr(out))
    return out


def e4m3_value(code: int) -> float:
    return float(_load().oracle_e4m3_value(code))


def e4m3_encode(v: float) -> int:
    return int(_load().oracle_e4m3_encode(v))
