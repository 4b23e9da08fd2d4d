"""Helpers for the GPU tests: move seeded inputs to the device and call the
C ABI through the Python binding."""
from __future__ import annotations

import numpy as np
import torch

import moe_inputs as mi
import routing_grouped_expert_gemm_gb300 as rg


def to_dev_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to("cuda")


def bf16_dev_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


class Layer:
    """Device copies of one workload's parameters plus a plan and workspace."""

    def __init__(self, inp: mi.MoEInputs, T_max: int | None = None, shared: bool = True, weights: dict | None = None,
                 **plan_kw):
        """weights: the device parameters of an earlier Layer of the same
        workload (shared instead of uploaded again)."""
        s = inp.shape
        self.shape = s
        self.T_max = T_max or inp.T
        self.plan = rg.moe_plan_create(self.T_max, s.D, s.I, s.E, s.k, s.I_s, score_fn=s.score,
                                       precision=s.precision, **plan_kw)
        self.mx = s.precision == "mxfp8"
        if weights is not None:
            self.w = weights
            self.ws_bytes = rg.moe_workspace_bytes(self.plan, self.T_max)
            self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device="cuda")
            return
        self.w = {
            "W_router": to_dev_bf16(inp.w_router),
            "b_router": None if inp.b_router is None else torch.from_numpy(inp.b_router).to("cuda"),
            "W_up": to_dev_bf16(inp.w_up),
            "W_gate": to_dev_bf16(inp.w_gate),
            "W_down": to_dev_bf16(inp.w_down),
        }
        if self.mx:  # routed weights quantised on the GPU (codes + scale blocks)
            self.w_bf16 = {k: self.w[k] for k in ("W_up", "W_gate", "W_down")}
            for name, rows, K in (("W_up", s.E * s.I, s.D), ("W_gate", s.E * s.I, s.D), ("W_down", s.E * s.D, s.I)):
                q = torch.empty((rows, K), dtype=torch.uint8, device="cuda")
                sc = torch.empty(rg.moe_mxfp8_scale_bytes(rows, K), dtype=torch.uint8, device="cuda")
                rg.moe_quantize_mxfp8(self.plan, self.w[name], rows, K, q, sc)
                self.w[name] = q
                self.w[name + "_scale"] = sc
        if shared and s.I_s > 0:
            self.w.update(Ws_up=to_dev_bf16(inp.ws_up), Ws_gate=to_dev_bf16(inp.ws_gate),
                          Ws_down=to_dev_bf16(inp.ws_down))
        self.ws_bytes = rg.moe_workspace_bytes(self.plan, self.T_max)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device="cuda")

    def run(self, x: torch.Tensor, T: int | None = None, export: bool = True, poison: bool = False) -> dict:
        s = self.shape
        T = x.shape[0] if T is None else T
        out = torch.empty((T, s.D), dtype=torch.bfloat16, device="cuda")
        res = {"out": out}
        if export:
            R = T * s.k
            res.update(topk_idx=torch.empty((T, s.k), dtype=torch.int32, device="cuda"),
                       topk_w=torch.empty((T, s.k), dtype=torch.float32, device="cuda"),
                       expert_counts=torch.empty(s.E, dtype=torch.int32, device="cuda"),
                       expert_offsets=torch.empty(s.E + 1, dtype=torch.int32, device="cuda"),
                       sched=torch.empty((R, 3), dtype=torch.int32, device="cuda"),
                       route_row=torch.empty(R, dtype=torch.int32, device="cuda"))
        if poison:
            self.ws.fill_(0xFF)  # bf16 0xFFFF is NaN: any unwritten read shows up
            out.fill_(float("nan"))
        rg.moe_fwd(self.plan, T, x, self.w, out, self.ws, self.ws_bytes,
                   **{k: v for k, v in res.items() if k != "out"})
        status = rg.moe_get_status(self.plan, self.ws)
        res["status"] = status
        return res


def rel_l2(a: np.ndarray, b: np.ndarray) -> float:
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def check_out(gpu: np.ndarray, ref: np.ndarray, rel_tol: float = 1e-2, maxabs_frac: float = 3e-2):
    """Tolerance for bf16 outputs: rel-L2 <= 1e-2 and max-abs <= 3e-2 * rms(out)."""
    assert np.isfinite(gpu).all(), "non-finite output"
    rel = rel_l2(gpu, ref)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    mabs = float(np.abs(gpu - ref).max())
    assert rel <= rel_tol, f"rel-L2 {rel:.3g} > {rel_tol}"
    assert mabs <= maxabs_frac * rms, f"max-abs {mabs:.3g} > {maxabs_frac} * rms {rms:.3g}"
    return rel, mabs / rms


def scale_blocks_to_rows(blocks: np.ndarray, rows: int, K: int) -> np.ndarray:
    """Library scale layout (512-byte blocks [rows/128][K/128]) -> [rows, K/32]."""
    b = blocks.reshape(rows // 128, K // 128, 32, 4, 4)  # [rb, kg, r%32, (r%128)//32, kb]
    return b.transpose(0, 3, 2, 1, 4).reshape(rows, K // 32)
