"""fp64 reference of the MoE layer's backward pass -- TEST INFRASTRUCTURE.

Only the tests import this module.  It shares nothing with the CUDA library.

"Mixture-of-Kittens: MoE Megakernel for NVL72s" trains the layer of Sec. 2.1
(Eq. MoE): Sec. 3.3 "Ring-Aware Forward Replay" recomputes forward
intermediates inside the backward pass, and Sec. 3.4 "Router Weight Gradient
Computation" takes the router-weight gradient from the inner product of the
gated activation h and the down projection's input gradient (W_down^T dO),
SonicMoE-style, instead of materialising the expert output.  Given an upstream
gradient dO = dL/d out, ``moe_bwd`` returns dL/d(every input) by the chain rule
written out on the forward's definition, in float64 numpy, with no rounding:

  forward, token t, slot j with expert e = idx[t, j]:
    l = W_r x + beta;  s = sigmoid(l), or softmax(l) over all E
    top-k on l (higher wins, ties to the lower expert id; slots in ascending id)
    g_j = s_e / sum_{selected} s;   a_u = W_up[e] x,  a_g = W_gate[e] x
    h = SiLU(a_g) * a_u;   y_j = W_down[e] h
    out = f_s(x) + sum_j g_j y_j   (f_s: the shared expert, same FFN, weight 1)

  backward:
    dy_j = g_j dO;  dg_j = <dO, y_j> = <W_down[e]^T dO, h>
    dh = W_down[e]^T dy_j;  dW_down[e] += dy_j h^T
    da_u = dh * SiLU(a_g);  da_g = dh * a_u * SiLU'(a_g),
        SiLU'(z) = sigma(z) (1 + z (1 - sigma(z)))
    dW_up[e] += da_u x^T;  dW_gate[e] += da_g x^T;  dx += W_up[e]^T da_u + W_gate[e]^T da_g
    g = s_sel / S (S = sum of the selected s): ds_e = (dg_j - sum_i g_i dg_i) / S for the
        selected experts, 0 for the others
    sigmoid: dl = ds * s (1 - s);  softmax: dl = s * (ds - <s, ds>)
    dW_r += dl x^T;  dbeta += dl;  dx += W_r^T dl

The selection is piecewise constant in l: no gradient flows through it (the
finite-difference pins keep every perturbation inside one selection).
"""
from __future__ import annotations

import numpy as np


def _sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def _silu(z):
    return z * _sigmoid(z)


def _dsilu(z):
    sg = _sigmoid(z)
    return sg * (1.0 + z * (1.0 - sg))


def select(logits: np.ndarray, k: int) -> np.ndarray:
    """Top-k experts per row: higher logit first, ties to the lower id; each row
    listed in ascending expert id (the slot order).  int64 [T, k]."""
    order = np.argsort(-logits, axis=1, kind="stable")  # stable: equal logits keep ascending id
    return np.sort(order[:, :k], axis=1)


def scores(logits: np.ndarray, score: str) -> np.ndarray:
    if score == "sigmoid":
        return _sigmoid(logits)
    if score == "softmax":
        z = np.exp(logits - logits.max(axis=1, keepdims=True))
        return z / z.sum(axis=1, keepdims=True)
    raise ValueError(score)


def moe_fwd(p: dict, k: int, score: str) -> dict:
    """Forward on float64 arrays.  ``p``: x [T,D], w_router [E,D], b_router [E] or
    None, w_up / w_gate [E,I,D], w_down [E,D,I], ws_up / ws_gate [I_s,D] and
    ws_down [D,I_s] or None.  Returns out [T,D] plus the intermediates the
    backward uses."""
    x = p["x"]
    T, D = x.shape
    E = p["w_router"].shape[0]
    logits = x @ p["w_router"].T
    if p.get("b_router") is not None:
        logits = logits + p["b_router"][None, :]
    idx = select(logits, k)
    s = scores(logits, score)
    s_sel = np.take_along_axis(s, idx, axis=1)
    S = s_sel.sum(axis=1)
    g = s_sel / S[:, None]
    out = np.zeros((T, D))
    a_u = np.zeros((T, k, p["w_up"].shape[1]))
    a_g = np.zeros_like(a_u)
    y = np.zeros((T, k, D))
    for e in range(E):
        tt, jj = np.nonzero(idx == e)
        if tt.size == 0:
            continue
        xe = x[tt]
        au, ag = xe @ p["w_up"][e].T, xe @ p["w_gate"][e].T
        h = _silu(ag) * au
        ye = h @ p["w_down"][e].T
        a_u[tt, jj], a_g[tt, jj], y[tt, jj] = au, ag, ye
    out += np.einsum("tj,tjd->td", g, y)
    shared = None
    if p.get("ws_up") is not None:
        su, sgt = x @ p["ws_up"].T, x @ p["ws_gate"].T
        ys = (_silu(sgt) * su) @ p["ws_down"].T
        out = ys + out
        shared = (su, sgt)
    return {"out": out, "logits": logits, "idx": idx, "s": s, "S": S, "g": g, "a_u": a_u, "a_g": a_g, "y": y,
            "shared": shared}


def moe_bwd(p: dict, k: int, score: str, dO: np.ndarray, experts=None) -> dict:
    """dL/d(inputs) for L with dL/d out = dO, as listed in the module docstring.
    Keys: x, w_router, b_router, w_up, w_gate, w_down, ws_up, ws_gate, ws_down
    (None where the input is None).

    ``experts``: None, or a list of expert ids whose weight gradients are
    wanted; then w_up / w_gate / w_down only need ``.shape`` and ``[e]``
    (an object that converts one expert at a time will do) and the routed
    weight gradients are returned as {e: array} for those experts only.  The
    arithmetic is the same either way."""
    f = moe_fwd(p, k, score)
    x = p["x"]
    T, D = x.shape
    E = p["w_router"].shape[0]
    idx, g, s, S = f["idx"], f["g"], f["s"], f["S"]
    dx = np.zeros_like(x)
    if experts is None:
        dw_up, dw_gate, dw_down = np.zeros_like(p["w_up"]), np.zeros_like(p["w_gate"]), np.zeros_like(p["w_down"])
    else:
        I = p["w_up"].shape[1]
        dw_up = {e: np.zeros((I, D)) for e in experts}
        dw_gate = {e: np.zeros((I, D)) for e in experts}
        dw_down = {e: np.zeros((D, I)) for e in experts}
    dg = np.zeros((T, k))
    for e in range(E):
        tt, jj = np.nonzero(idx == e)
        if tt.size == 0:
            continue
        au, ag = f["a_u"][tt, jj], f["a_g"][tt, jj]
        h = _silu(ag) * au
        dOe = dO[tt]
        wdn = p["w_down"][e]
        dg[tt, jj] = np.einsum("nd,nd->n", dOe @ wdn, h)  # <W_down^T dO, h>
        dy = g[tt, jj][:, None] * dOe
        dh = dy @ wdn
        da_u = dh * _silu(ag)
        da_g = dh * au * _dsilu(ag)
        if experts is None or e in dw_up:
            dw_down[e] += dy.T @ h
            dw_up[e] += da_u.T @ x[tt]
            dw_gate[e] += da_g.T @ x[tt]
        np.add.at(dx, tt, da_u @ p["w_up"][e] + da_g @ p["w_gate"][e])
    # router: g = s_sel / S
    c = np.einsum("tj,tj->t", g, dg)
    ds = np.zeros((T, E))
    np.put_along_axis(ds, idx, (dg - c[:, None]) / S[:, None], axis=1)
    if score == "sigmoid":
        dl = ds * s * (1.0 - s)
    else:
        dl = s * (ds - np.einsum("te,te->t", s, ds)[:, None])
    dw_router = dl.T @ x
    db_router = dl.sum(axis=0) if p.get("b_router") is not None else None
    dx += dl @ p["w_router"]
    grads = {"x": dx, "w_router": dw_router, "b_router": db_router, "w_up": dw_up, "w_gate": dw_gate,
             "w_down": dw_down, "ws_up": None, "ws_gate": None, "ws_down": None}
    if f["shared"] is not None:
        su, sgt = f["shared"]
        hs = _silu(sgt) * su
        dhs = dO @ p["ws_down"]
        grads["ws_down"] = dO.T @ hs
        dsu = dhs * _silu(sgt)
        dsg = dhs * su * _dsilu(sgt)
        grads["ws_up"] = dsu.T @ x
        grads["ws_gate"] = dsg.T @ x
        dx += dsu @ p["ws_up"] + dsg @ p["ws_gate"]
    return grads
