"""The CUDA backward pass (moe_bwd) against the fp64 backward oracle
(oracle/backward.py), through the C ABI.

Every gradient -- dx, dW_router, db, dW_up, dW_gate, dW_down and the shared
expert's -- within rel-L2 <= 1e-2 of the oracle (the GPU rounds h, the
activation gradients and the outputs to bf16, and the per-route dx to fp16);
two calls bitwise identical; an expert that no route reaches gets an exactly
zero weight gradient.  At the Kimi-K2 shape (T = 32768, E = 384, top-8, one
shared expert) the oracle runs on a token subset: every token routed to the
checked experts (so their weight gradients and router rows are complete) plus
sampled tokens for dx.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
from oracle import backward as ob

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from routing_grouped_expert_gemm_gb300 import build
    build.build()


def f64(bits):
    return mi.bf16_bits_to_f32(bits).astype(np.float64)


class LazyExperts:
    """[E, ...] bf16 weights converted to fp64 one expert at a time."""

    def __init__(self, bits):
        self.bits = bits
        self.shape = bits.shape

    def __getitem__(self, e):
        return f64(self.bits[e])


def run_bwd(inp, dO_bits, shared=True, plan_kw=None, layer=None):
    """Forward then backward on the GPU; returns (layer, gradients as device
    tensors, forward results)."""
    import gpu_util
    import routing_grouped_expert_gemm_gb300 as rg
    s = inp.shape
    if layer is None:
        layer = gpu_util.Layer(inp, shared=shared, **(plan_kw or dict(minibatch=1024, ring_slots=2, gather_ctas=2)))
    x = gpu_util.to_dev_bf16(inp.x)
    dO = gpu_util.to_dev_bf16(dO_bits)
    res = layer.run(x)
    assert res["status"] == 0
    T = inp.T
    g = {"dx": torch.empty((T, s.D), dtype=torch.bfloat16, device="cuda"),
         "dW_router": torch.empty((s.E, s.D), dtype=torch.float32, device="cuda"),
         "db_router": torch.empty(s.E, dtype=torch.float32, device="cuda") if inp.b_router is not None else None,
         "dW_up": torch.empty((s.E, s.I, s.D), dtype=torch.bfloat16, device="cuda"),
         "dW_gate": torch.empty((s.E, s.I, s.D), dtype=torch.bfloat16, device="cuda"),
         "dW_down": torch.empty((s.E, s.D, s.I), dtype=torch.bfloat16, device="cuda")}
    has_shared = shared and s.I_s > 0
    if has_shared:
        g.update(dWs_up=torch.empty((s.I_s, s.D), dtype=torch.bfloat16, device="cuda"),
                 dWs_gate=torch.empty((s.I_s, s.D), dtype=torch.bfloat16, device="cuda"),
                 dWs_down=torch.empty((s.D, s.I_s), dtype=torch.bfloat16, device="cuda"))
    for v in g.values():
        if v is not None:
            v.fill_(float("nan"))  # every element must be written
    wsb = rg.moe_bwd_workspace_bytes(layer.plan, T)
    assert wsb > 0
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    ws.fill_(0xFF)
    rg.moe_bwd(layer.plan, T, x, layer.w, dO, layer.ws, g, ws)
    assert rg.moe_get_status(layer.plan, ws) == 0
    return layer, g, res


def npy(t):
    return None if t is None else t.double().cpu().numpy()


def oracle_params(inp, shared=True, lazy=False):
    p = {"x": f64(inp.x), "w_router": f64(inp.w_router),
         "b_router": None if inp.b_router is None else inp.b_router.astype(np.float64)}
    for name in ("w_up", "w_gate", "w_down"):
        p[name] = LazyExperts(getattr(inp, name)) if lazy else f64(getattr(inp, name))
    if shared and inp.shape.I_s > 0:
        p.update(ws_up=f64(inp.ws_up), ws_gate=f64(inp.ws_gate), ws_down=f64(inp.ws_down))
    return p


def rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def check_all(gpu, ref, tol=1e-2):
    pairs = [("dx", "x"), ("dW_router", "w_router"), ("db_router", "b_router"), ("dW_up", "w_up"),
             ("dW_gate", "w_gate"), ("dW_down", "w_down"), ("dWs_up", "ws_up"), ("dWs_gate", "ws_gate"),
             ("dWs_down", "ws_down")]
    out = {}
    for gk, rk in pairs:
        if ref.get(rk) is None:
            assert gpu.get(gk) is None, gk
            continue
        got = npy(gpu[gk])
        assert np.isfinite(got).all(), f"{gk}: non-finite"
        r = rel(got, ref[rk])
        out[gk] = r
        assert r <= tol, f"{gk}: rel-L2 {r:.3g} > {tol}"
    return out


def small(T, D, I, E, k, I_s, score="sigmoid", cid=700, beta=0.3):
    shape = mi.custom_shape(T, D, I, E, k, I_s, score=score, config_id=cid)
    inp = mi.make_inputs(shape, calibration={"beta": None, "redraw": {}})
    if beta:
        inp.b_router = (beta * mi.normal_f64(shape.seed, 99, E)).astype(np.float32)
    return inp, mi.grad_out(shape)


ONE_CTA = dict(minibatch=1024, ring_slots=2, gather_ctas=2)
PAIRS = dict(minibatch=1024, ring_slots=2, gather_ctas=2, mma_pair=1)  # the backward's GEMMs as CTA pairs too


@pytest.mark.parametrize("kw", [ONE_CTA, PAIRS], ids=["one_cta", "pairs"])
@pytest.mark.parametrize("T", [1, 300])
def test_backward_small_sigmoid_shared(T, kw):
    inp, dO = small(300, 256, 256, 8, 3, 256)
    inp.x = inp.x[:T].copy()
    inp.T = T
    dO = dO[:T]
    _, gpu, _ = run_bwd(inp, dO, plan_kw=kw)
    ref = ob.moe_bwd(oracle_params(inp), inp.shape.k, inp.shape.score, f64(dO))
    check_all(gpu, ref)


@pytest.mark.parametrize("kw", [ONE_CTA, PAIRS], ids=["one_cta", "pairs"])
def test_backward_softmax_no_shared_ragged(kw):
    inp, dO = small(333, 512, 256, 16, 4, 0, score="softmax", cid=701, beta=0.0)
    _, gpu, _ = run_bwd(inp, dO, shared=False, plan_kw=kw)
    ref = ob.moe_bwd(oracle_params(inp, shared=False), inp.shape.k, inp.shape.score, f64(dO))
    check_all(gpu, ref)


@pytest.mark.parametrize("kw", [ONE_CTA, PAIRS], ids=["one_cta", "pairs"])
def test_backward_medium_several_tiles(kw):
    # ragged token tail, several 128-row M-tiles per expert (odd counts: empty
    # partners for pairs), D and I over many tiles
    inp, dO = small(1000, 512, 512, 32, 6, 256, cid=702)
    _, gpu, _ = run_bwd(inp, dO, plan_kw=kw)
    ref = ob.moe_bwd(oracle_params(inp), inp.shape.k, inp.shape.score, f64(dO))
    check_all(gpu, ref)


@pytest.mark.parametrize("kw", [ONE_CTA, PAIRS], ids=["one_cta", "pairs"])
def test_backward_unrouted_expert_has_zero_gradient(kw):
    inp, dO = small(256, 256, 256, 8, 2, 0, cid=703)
    inp.b_router[5] = -40.0  # no token selects expert 5
    _, gpu, res = run_bwd(inp, dO, shared=False, plan_kw=kw)
    assert res["expert_counts"].cpu().numpy()[5] == 0
    for key in ("dW_up", "dW_gate", "dW_down"):
        assert np.all(npy(gpu[key][5]) == 0.0), key
    assert np.all(npy(gpu["dW_router"][5]) == 0.0) and float(gpu["db_router"][5]) == 0.0
    ref = ob.moe_bwd(oracle_params(inp, shared=False), inp.shape.k, inp.shape.score, f64(dO))
    check_all(gpu, ref)


def test_backward_bitwise_deterministic():
    """Two calls give the same bits, and the CTA-pair GEMMs give the one-CTA
    GEMMs' bits (each output element keeps its K order)."""
    import gpu_util
    inp, dO = small(700, 512, 256, 16, 4, 256, cid=704)
    layer = gpu_util.Layer(inp, minibatch=512, ring_slots=2, gather_ctas=2)
    _, a, _ = run_bwd(inp, dO, layer=layer)
    _, b, _ = run_bwd(inp, dO, layer=layer)
    pl = gpu_util.Layer(inp, weights=layer.w, minibatch=512, ring_slots=2, gather_ctas=2, mma_pair=1)
    _, c, _ = run_bwd(inp, dO, layer=pl)
    for key in a:
        if a[key] is not None:
            assert torch.equal(a[key], b[key]), key
            assert torch.equal(a[key], c[key]), f"{key}: pairs differ from one CTA per tile"


def test_backward_kimi_k2_full_size_sampled():
    """Kimi-K2 shape: T = 32768, D = 7168, I = 2048, E = 384, top-8, one shared
    expert, uniform load, upstream gradient dO ~ N(0, 1)."""
    inp = mi.make_inputs("kimi_k2")
    s = inp.shape
    dO = mi.grad_out(s)
    _, gpu, res = run_bwd(inp, dO, plan_kw=dict(minibatch=8192, ring_slots=4, gather_ctas=8, mma_pair=1))
    counts = res["expert_counts"].cpu().numpy()
    idx = res["topk_idx"].cpu().numpy()
    live = np.nonzero(counts > 0)[0]
    experts = [int(live[np.argmin(counts[live])]), int(live[np.argmax(counts[live])])]
    rows = np.nonzero(np.isin(idx, experts).any(axis=1))[0]
    sample = np.unique(np.concatenate([rows, np.linspace(0, s.T - 1, 24).astype(np.int64)]))
    sub = mi.MoEInputs(s, len(sample), inp.x[sample], inp.w_router, inp.b_router, inp.w_up, inp.w_gate,
                       inp.w_down, inp.ws_up, inp.ws_gate, inp.ws_down)
    ref = ob.moe_bwd(oracle_params(sub, lazy=True), s.k, s.score, f64(dO[sample]), experts=experts)
    # dx of every sampled token (tokens are independent)
    assert rel(npy(gpu["dx"][torch.from_numpy(sample).cuda()]), ref["x"]) <= 1e-2
    # the checked experts' weight gradients and router rows: all their routes are in the subset
    for e in experts:
        for gk, rk in (("dW_up", "w_up"), ("dW_gate", "w_gate"), ("dW_down", "w_down")):
            r = rel(npy(gpu[gk][e]), ref[rk][e])
            assert r <= 1e-2, f"{gk}[{e}] rel-L2 {r:.3g}"
        assert rel(npy(gpu["dW_router"][e]), ref["w_router"][e]) <= 1e-2, f"dW_router[{e}]"
    for key in ("dWs_up", "dWs_gate", "dWs_down", "dW_up", "dW_gate", "dW_down", "dW_router"):
        assert bool(torch.isfinite(gpu[key].float()).all()), key
