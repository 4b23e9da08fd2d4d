"""Python binding of the MoE-layer forward C ABI (``include/moe.h``).

Argument marshalling only: every step of the forward runs in the CUDA library
``_lib/libmoe_gb300.so`` (built by ``build.py``).  There is no fallback: if the
library is missing or cannot be loaded, every entry point raises.  PyTorch is
used only to hand over device pointers and streams.

Entry points keep the C names: ``moe_plan_create``, ``moe_plan_destroy``,
``moe_workspace_bytes``, ``moe_quantize_mxfp8``, ``moe_mxfp8_scale_bytes``,
``moe_fwd``, ``moe_bwd_workspace_bytes``, ``moe_bwd``, ``moe_get_status``,
``moe_get_phase_times``, ``moe_route_static``, ``moe_error_string``.
"""
from __future__ import annotations

import ctypes
import os
import re

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libmoe_gb300.so")
if os.environ.get("MOE_TRACE_BUILD") == "1":  # profiling only: the MOE_TRACE variant of the same library
    LIB_PATH = os.path.join(_HERE, "_lib", "libmoe_gb300_trace.so")
elif os.environ.get("MOE_DEBUG_BUILD") == "1":  # debugging only: the MOE_DEBUG_LOG variant
    LIB_PATH = os.path.join(_HERE, "_lib", "libmoe_gb300_dbg.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "moe.h")
TESTING_HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "moe_testing.h")
# test hooks (one-tile probes of tensor-core encodings), a library of their own
TESTING_LIB_PATH = os.path.join(_HERE, "_lib", "libmoe_gb300_testing.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED_SHAPE = -2
MOE_ERR_WORKSPACE_TOO_SMALL = -3
MOE_ERR_CUDA = -4
MOE_ERR_UNSUPPORTED_DEVICE = -5
MOE_ERR_STATIC_SCRATCH_TOO_SMALL = -6
MOE_ROUTE_STATIC_MAX_TOKENS = 16384
MOE_STATUS_OK, MOE_STATUS_TIMEOUT, MOE_STATUS_SCHEDULE_INVALID, MOE_STATUS_STAGING_OVERFLOW = 0, 1, 2, 3
MOE_SCORE_SIGMOID, MOE_SCORE_SOFTMAX = 0, 1
MOE_PREC_BF16, MOE_PREC_MXFP8 = 0, 1
MOE_DISPATCH_RING, MOE_DISPATCH_DIRECT, MOE_DISPATCH_SPREAD = 0, 1, 2


class MoEError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {moe_error_string(code)} ({code})")


class moe_config(ctypes.Structure):
    _fields_ = [("T_max", ctypes.c_int64), ("D", ctypes.c_int64), ("I", ctypes.c_int64), ("E", ctypes.c_int64),
                ("k", ctypes.c_int64), ("I_s", ctypes.c_int64), ("score_fn", ctypes.c_int32),
                ("precision", ctypes.c_int32), ("minibatch", ctypes.c_int32), ("ring_slots", ctypes.c_int32),
                ("gather_ctas", ctypes.c_int32), ("gemm_ctas", ctypes.c_int32), ("lag", ctypes.c_int32),
                ("timeout_ms", ctypes.c_int32), ("dispatch", ctypes.c_int32), ("l2_prefetch", ctypes.c_int32),
                ("mma_pair", ctypes.c_int32), ("raster", ctypes.c_int32),
                ("test_unfilled_minibatch", ctypes.c_int32), ("clc", ctypes.c_int32),
                ("plain_launch", ctypes.c_int32), ("pad_odd_tiles", ctypes.c_int32)]


class moe_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "W_router", "b_router", "W_up", "W_gate", "W_down", "W_up_scale", "W_gate_scale", "W_down_scale",
        "Ws_up", "Ws_gate", "Ws_down")]


class moe_grads(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "dx", "dW_router", "db_router", "dW_up", "dW_gate", "dW_down", "dWs_up", "dWs_gate", "dWs_down")]


class moe_outputs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "out", "topk_idx", "topk_w", "expert_counts", "expert_offsets", "sched", "route_row")]


_lib = None


def lib():
    """The loaded CUDA library (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing (run routing_grouped_expert_gemm_gb300/build.py)")
    L = ctypes.CDLL(LIB_PATH)
    vp, i64, sz, i32p = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.POINTER(ctypes.c_int)
    L.moe_plan_create.argtypes = [ctypes.POINTER(moe_config), ctypes.POINTER(vp)]
    L.moe_plan_create.restype = ctypes.c_int
    L.moe_plan_destroy.argtypes = [vp]
    L.moe_plan_destroy.restype = ctypes.c_int
    L.moe_workspace_bytes.argtypes = [vp, i64]
    L.moe_workspace_bytes.restype = sz
    L.moe_quantize_mxfp8.argtypes = [vp, vp, i64, i64, vp, vp, vp]
    L.moe_quantize_mxfp8.restype = ctypes.c_int
    L.moe_mxfp8_scale_bytes.argtypes = [i64, i64]
    L.moe_mxfp8_scale_bytes.restype = sz
    L.moe_fwd.argtypes = [vp, i64, vp, ctypes.POINTER(moe_weights), ctypes.POINTER(moe_outputs), vp, sz, vp]
    L.moe_fwd.restype = ctypes.c_int
    L.moe_get_status.argtypes = [vp, vp, i32p, vp]
    L.moe_get_status.restype = ctypes.c_int
    L.moe_plan_set_timing_events.argtypes = [vp, ctypes.POINTER(vp)]
    L.moe_plan_set_timing_events.restype = ctypes.c_int
    L.moe_plan_set_bwd_timing_events.argtypes = [vp, ctypes.POINTER(vp)]
    L.moe_plan_set_bwd_timing_events.restype = ctypes.c_int
    L.moe_bwd_workspace_bytes.argtypes = [vp, i64]
    L.moe_bwd_workspace_bytes.restype = sz
    L.moe_bwd.argtypes = [vp, i64, vp, ctypes.POINTER(moe_weights), vp, vp, ctypes.POINTER(moe_grads), vp, sz, vp]
    L.moe_bwd.restype = ctypes.c_int
    L.moe_get_phase_times.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_double), vp]
    L.moe_get_phase_times.restype = ctypes.c_int
    L.moe_route_static.argtypes = [vp, i64, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.moe_route_static.restype = ctypes.c_int
    L.moe_route_static_scratch_bytes.argtypes = []
    L.moe_route_static_scratch_bytes.restype = sz
    L.moe_error_string.argtypes = [ctypes.c_int]
    L.moe_error_string.restype = ctypes.c_char_p
    _lib = L
    return L


_testing_lib = None


def testing_lib():
    """The test-hook library (one-tile probes; raises if it was not built)."""
    global _testing_lib
    if _testing_lib is not None:
        return _testing_lib
    if not os.path.exists(TESTING_LIB_PATH):
        raise RuntimeError(f"test-hook library not built: {TESTING_LIB_PATH} is missing")
    L = ctypes.CDLL(TESTING_LIB_PATH)
    vp = ctypes.c_void_p
    L.moe_testing_mx_tile.argtypes = [vp, vp, vp, vp, ctypes.c_int, vp]
    L.moe_testing_mx_tile.restype = ctypes.c_int
    L.moe_testing_pair_tile.argtypes = [vp, vp, vp, vp, ctypes.c_int, vp]
    L.moe_testing_pair_tile.restype = ctypes.c_int
    L.moe_testing_pair_mma_time.argtypes = [vp, vp, vp, vp, ctypes.c_int, ctypes.c_int, vp, vp]
    L.moe_testing_pair_mma_time.restype = ctypes.c_int
    L.moe_testing_pair_mx_tile.argtypes = [vp, vp, vp, vp, vp, ctypes.c_int, vp]
    L.moe_testing_pair_mx_tile.restype = ctypes.c_int
    L.moe_testing_mn_tile.argtypes = [vp, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, vp]
    L.moe_testing_mn_tile.restype = ctypes.c_int
    L.moe_testing_tma3d_load.argtypes = [vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, vp]
    L.moe_testing_tma3d_load.restype = ctypes.c_int
    _testing_lib = L
    return L


def declared_functions(header: str | None = None) -> list[str]:
    """Function names declared in one header (default: include/moe.h, the ABI)."""
    text = open(header or HEADER_PATH).read()
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char\*)\s+(moe_\w+)\s*\(", text, flags=re.M)))


def _ptr(v) -> int | None:
    if v is None:
        return None
    if isinstance(v, int):
        return v
    return int(v.data_ptr())  # torch tensor


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def moe_error_string(code: int) -> str:
    return lib().moe_error_string(code).decode()


class Plan:
    """Owns a moe_plan*; released by moe_plan_destroy (or garbage collection)."""

    def __init__(self, handle: int, cfg: moe_config):
        self.handle = handle
        self.cfg = cfg

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.moe_plan_destroy(self.handle)
            self.handle = None


def moe_plan_create(T_max, D, I, E, k, I_s=0, score_fn=MOE_SCORE_SIGMOID, precision=MOE_PREC_BF16, minibatch=0,
                    ring_slots=0, gather_ctas=0, gemm_ctas=0, lag=1, timeout_ms=0, dispatch=MOE_DISPATCH_RING,
                    l2_prefetch=0, mma_pair=0, raster=0, test_unfilled_minibatch=0, clc=0, plain_launch=0,
                    pad_odd_tiles=0) -> Plan:
    if isinstance(score_fn, str):
        score_fn = {"sigmoid": MOE_SCORE_SIGMOID, "softmax": MOE_SCORE_SOFTMAX}[score_fn]
    if isinstance(precision, str):
        precision = {"bf16": MOE_PREC_BF16, "mxfp8": MOE_PREC_MXFP8}[precision]
    if isinstance(dispatch, str):
        dispatch = {"ring": MOE_DISPATCH_RING, "direct": MOE_DISPATCH_DIRECT, "spread": MOE_DISPATCH_SPREAD}[dispatch]
    cfg = moe_config(T_max, D, I, E, k, I_s, score_fn, precision, minibatch, ring_slots, gather_ctas, gemm_ctas,
                     lag, timeout_ms, dispatch, l2_prefetch, mma_pair, raster, test_unfilled_minibatch, clc, plain_launch,
                     pad_odd_tiles)
    h = ctypes.c_void_p()
    rc = lib().moe_plan_create(ctypes.byref(cfg), ctypes.byref(h))
    if rc != MOE_OK:
        raise MoEError(rc, "moe_plan_create")
    return Plan(h.value, cfg)


def moe_plan_destroy(plan: Plan) -> None:
    if plan.handle:
        lib().moe_plan_destroy(plan.handle)
        plan.handle = None


def moe_workspace_bytes(plan: Plan, T: int) -> int:
    return int(lib().moe_workspace_bytes(plan.handle, T))


def moe_mxfp8_scale_bytes(rows: int, K: int) -> int:
    return int(lib().moe_mxfp8_scale_bytes(rows, K))


def moe_quantize_mxfp8(plan: Plan, W, rows: int, K: int, q, scales, stream=None) -> None:
    rc = lib().moe_quantize_mxfp8(plan.handle, _ptr(W), rows, K, _ptr(q), _ptr(scales), _stream(stream))
    if rc != MOE_OK:
        raise MoEError(rc, "moe_quantize_mxfp8")


def moe_fwd(plan: Plan, T: int, x, weights: dict, out, workspace, workspace_bytes: int | None = None,
            topk_idx=None, topk_w=None, expert_counts=None, expert_offsets=None, sched=None, route_row=None,
            stream=None) -> None:
    """weights: dict with keys of moe_weights (W_router, b_router, W_up, ...)."""
    w = moe_weights(**{k: _ptr(v) for k, v in weights.items()})
    o = moe_outputs(_ptr(out), _ptr(topk_idx), _ptr(topk_w), _ptr(expert_counts), _ptr(expert_offsets),
                    _ptr(sched), _ptr(route_row))
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    rc = lib().moe_fwd(plan.handle, T, _ptr(x), ctypes.byref(w), ctypes.byref(o), _ptr(workspace),
                       workspace_bytes, _stream(stream))
    if rc != MOE_OK:
        raise MoEError(rc, "moe_fwd")


def moe_bwd_workspace_bytes(plan: Plan, T: int) -> int:
    return int(lib().moe_bwd_workspace_bytes(plan.handle, T))


def moe_bwd(plan: Plan, T: int, x, weights: dict, dO, fwd_workspace, grads: dict, workspace,
            workspace_bytes: int | None = None, stream=None) -> None:
    """Backward pass: ``grads`` has keys of moe_grads (dx, dW_router, db_router,
    dW_up, dW_gate, dW_down, dWs_up, dWs_gate, dWs_down); ``fwd_workspace`` is
    the workspace of the moe_fwd call on the same x and weights."""
    w = moe_weights(**{k: _ptr(v) for k, v in weights.items()})
    g = moe_grads(**{k: _ptr(v) for k, v in grads.items()})
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    rc = lib().moe_bwd(plan.handle, T, _ptr(x), ctypes.byref(w), _ptr(dO), _ptr(fwd_workspace), ctypes.byref(g),
                       _ptr(workspace), workspace_bytes, _stream(stream))
    if rc != MOE_OK:
        raise MoEError(rc, "moe_bwd")


def moe_get_status(plan: Plan, workspace, stream=None) -> int:
    st = ctypes.c_int(-1)
    rc = lib().moe_get_status(plan.handle, _ptr(workspace), ctypes.byref(st), _stream(stream))
    if rc != MOE_OK:
        raise MoEError(rc, "moe_get_status")
    return st.value


def moe_get_phase_times(plan: Plan, workspace, stream=None) -> dict:
    """Phase stamps of the last forward on ``workspace`` (ms after the persistent
    kernel's start; None where the phase did not happen)."""
    arr = (ctypes.c_double * 3)()
    rc = lib().moe_get_phase_times(plan.handle, _ptr(workspace), arr, _stream(stream))
    if rc != MOE_OK:
        raise MoEError(rc, "moe_get_phase_times")
    keys = ("last_fill", "combine_start", "combine_end")
    return {k: (None if v < 0 else float(v)) for k, v in zip(keys, arr)}


def moe_plan_set_timing_events(plan: Plan, events) -> None:
    """events: four torch.cuda.Event (created with enable_timing) or None."""
    if events is None:
        rc = lib().moe_plan_set_timing_events(plan.handle, None)
    else:
        arr = (ctypes.c_void_p * 4)(*[int(e.cuda_event) for e in events])
        rc = lib().moe_plan_set_timing_events(plan.handle, arr)
    if rc != MOE_OK:
        raise MoEError(rc, "moe_plan_set_timing_events")


def moe_plan_set_bwd_timing_events(plan: Plan, events) -> None:
    """events: five torch.cuda.Event (created with enable_timing) or None."""
    if events is None:
        rc = lib().moe_plan_set_bwd_timing_events(plan.handle, None)
    else:
        arr = (ctypes.c_void_p * 5)(*[int(e.cuda_event) for e in events])
        rc = lib().moe_plan_set_bwd_timing_events(plan.handle, arr)
    if rc != MOE_OK:
        raise MoEError(rc, "moe_plan_set_bwd_timing_events")


def moe_route_static(plan: Plan, T: int, x, W_router, b_router, topk_idx, topk_w, expert_counts, expert_offsets,
                     sched, route_row, device_status=None, stream=None) -> None:
    """Routing stage (top-k, g, counts, offsets, schedule table) that allocates
    nothing: its scratch is a fixed array inside the library, for callers that
    cannot call cudaMalloc.  Calls that overlap on the GPU race on that array."""
    rc = lib().moe_route_static(plan.handle, T, _ptr(x), _ptr(W_router), _ptr(b_router), _ptr(topk_idx),
                                _ptr(topk_w), _ptr(expert_counts), _ptr(expert_offsets), _ptr(sched),
                                _ptr(route_row), _ptr(device_status), _stream(stream))
    if rc != MOE_OK:
        raise MoEError(rc, "moe_route_static")


def moe_route_static_scratch_bytes() -> int:
    return int(lib().moe_route_static_scratch_bytes())
