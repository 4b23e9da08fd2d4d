"""Pins of the fp64 backward oracle (oracle/backward.py) against things other
than itself: its forward against the pinned C forward oracle, every gradient
against central finite differences of that forward, the dense special case
(E = k = 1, where the layer is a plain FFN) against torch autograd, and
linearity in the upstream gradient.  Sources: "Mixture-of-Kittens: MoE
Megakernel for NVL72s" Sec. 2.1 (Eq. MoE), Sec. 3.3 "Ring-Aware Forward
Replay" and Sec. 3.4 "Router Weight Gradient Computation".
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
from oracle import backward as bw

NAMES = ["x", "w_router", "b_router", "w_up", "w_gate", "w_down", "ws_up", "ws_gate", "ws_down"]


def f64(bits):
    return mi.bf16_bits_to_f32(bits).astype(np.float64)


def tiny_params(T=12, D=32, I=16, E=6, k=2, I_s=8, seed=3, bias=True):
    """bf16-representable fp64 inputs (so that the C oracle sees the same values)
    with the k-th and (k+1)-th logits of every token at least 1e-3 apart."""
    rng = np.random.default_rng(seed)

    def bf(a):
        return f64(mi.f32_to_bf16_bits(a.astype(np.float32)))

    for _ in range(100):
        p = {"x": bf(rng.normal(size=(T, D))),
             "w_router": bf(rng.normal(size=(E, D)) / np.sqrt(D)),
             "b_router": (0.3 * rng.normal(size=E)).astype(np.float32).astype(np.float64) if bias else None,
             "w_up": bf(rng.normal(size=(E, I, D)) / np.sqrt(D)),
             "w_gate": bf(rng.normal(size=(E, I, D)) / np.sqrt(D)),
             "w_down": bf(rng.normal(size=(E, D, I)) / np.sqrt(I)),
             "ws_up": bf(rng.normal(size=(I_s, D)) / np.sqrt(D)) if I_s else None,
             "ws_gate": bf(rng.normal(size=(I_s, D)) / np.sqrt(D)) if I_s else None,
             "ws_down": bf(rng.normal(size=(D, I_s)) / np.sqrt(I_s)) if I_s else None}
        l = p["x"] @ p["w_router"].T + (p["b_router"] if bias else 0.0)
        srt = -np.sort(-l, axis=1)
        if k == E or (srt[:, k - 1] - srt[:, k]).min() >= 1e-3:
            return p
    raise RuntimeError("no input with a clear top-k gap")


def bits(a):
    return mi.f32_to_bf16_bits(a.astype(np.float32))


@pytest.mark.parametrize("score", ["sigmoid", "softmax"])
@pytest.mark.parametrize("I_s", [8, 0])
def test_numpy_forward_matches_c_oracle(score, I_s):
    T, D, I, E, k = 12, 32, 16, 6, 2
    p = tiny_params(T, D, I, E, k, I_s, seed=5)
    f = bw.moe_fwd(p, k, score)
    shape = mi.custom_shape(T, D, I, E, k, I_s, score=score)
    out, idx, g = oracle.moe_fwd(shape, bits(p["x"]), bits(p["w_router"]), p["b_router"].astype(np.float32),
                                 bits(p["w_up"]), bits(p["w_gate"]), bits(p["w_down"]),
                                 bits(p["ws_up"]) if I_s else None, bits(p["ws_gate"]) if I_s else None,
                                 bits(p["ws_down"]) if I_s else None)
    assert np.array_equal(idx, f["idx"])
    np.testing.assert_allclose(g, f["g"], rtol=1e-12, atol=0)
    np.testing.assert_allclose(out, f["out"], rtol=1e-10, atol=1e-12)


def _loss(p, k, score, dO):
    return float(np.sum(bw.moe_fwd(p, k, score)["out"] * dO))


@pytest.mark.parametrize("score", ["sigmoid", "softmax"])
@pytest.mark.parametrize("I_s", [8, 0])
def test_gradients_match_central_differences(score, I_s):
    k = 2
    p = tiny_params(I_s=I_s, seed=11, k=k)
    rng = np.random.default_rng(7)
    dO = rng.normal(size=p["x"].shape)
    grads = bw.moe_bwd(p, k, score, dO)
    idx0 = bw.moe_fwd(p, k, score)["idx"]
    eps = 1e-6
    for name in NAMES:
        if p[name] is None:
            assert grads[name] is None
            continue
        a = p[name]
        assert grads[name].shape == a.shape
        flat = a.reshape(-1)
        for i in rng.choice(flat.size, size=min(12, flat.size), replace=False):
            orig = flat[i]
            flat[i] = orig + eps
            lp = _loss(p, k, score, dO)
            assert np.array_equal(bw.moe_fwd(p, k, score)["idx"], idx0)  # same selection
            flat[i] = orig - eps
            lm = _loss(p, k, score, dO)
            flat[i] = orig
            fd = (lp - lm) / (2 * eps)
            an = grads[name].reshape(-1)[i]
            assert abs(fd - an) <= 1e-6 * (1.0 + abs(an)), f"{name}[{i}]: fd {fd:.9g} vs {an:.9g}"


def test_dense_special_case_matches_torch_autograd():
    # E = k = 1: g = 1 and the routed expert is a plain FFN; the router gets no gradient
    T, D, I, I_s = 10, 24, 16, 8
    p = tiny_params(T, D, I, 1, 1, I_s, seed=2)
    dO = np.random.default_rng(4).normal(size=(T, D))
    grads = bw.moe_bwd(p, 1, "sigmoid", dO)
    t = {n: torch.tensor(p[n], dtype=torch.float64, requires_grad=True) for n in NAMES if p[n] is not None}

    def ffn(x, wu, wg, wd):
        return (torch.nn.functional.silu(x @ wg.T) * (x @ wu.T)) @ wd.T

    out = ffn(t["x"], t["w_up"][0], t["w_gate"][0], t["w_down"][0]) + ffn(t["x"], t["ws_up"], t["ws_gate"],
                                                                           t["ws_down"])
    out.backward(torch.tensor(dO))
    for n in t:
        ref = np.zeros_like(p[n]) if t[n].grad is None else t[n].grad.numpy()  # router: g = 1 is constant
        np.testing.assert_allclose(grads[n], ref, rtol=1e-10, atol=1e-12, err_msg=n)


def test_backward_is_linear_in_the_upstream_gradient():
    p = tiny_params(seed=13)
    rng = np.random.default_rng(8)
    d1, d2 = rng.normal(size=p["x"].shape), rng.normal(size=p["x"].shape)
    g1, g2 = bw.moe_bwd(p, 2, "sigmoid", d1), bw.moe_bwd(p, 2, "sigmoid", d2)
    g12 = bw.moe_bwd(p, 2, "sigmoid", d1 + 2.0 * d2)
    for n in NAMES:
        np.testing.assert_allclose(g12[n], g1[n] + 2.0 * g2[n], rtol=1e-10, atol=1e-12, err_msg=n)


def test_unrouted_expert_gets_no_gradient():
    # an expert no token selects has zero weight gradients
    p = tiny_params(seed=17)
    p["w_router"][5] = 0.0
    p["b_router"][5] = -50.0
    g = bw.moe_bwd(p, 2, "sigmoid", np.ones_like(p["x"]))
    assert not g["w_up"][5].any() and not g["w_gate"][5].any() and not g["w_down"][5].any()


def test_upstream_gradient_generator():
    # dL/d out of the backward workloads: N(0, 1) bf16, a prefix of the full draw for any T
    a, b = mi.grad_out("tiny"), mi.grad_out("tiny", T=100)
    assert a.shape == (256, 256) and a.dtype == np.uint16 and np.array_equal(a[:100], b)
    v = f64(a)
    assert abs(v.mean()) < 0.02 and abs(v.std() - 1.0) < 0.02
    assert not np.array_equal(a, mi.make_inputs("tiny").x)  # its own stream, not x's
