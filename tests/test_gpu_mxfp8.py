"""MXFP8 routed experts (MoK Sec. 3.4 "MXFP8 Support"; OCP MX v1.0 E4M3 with
E8M0 scales per 32 elements along the contraction dimension) vs the fp64
oracle.  The oracle quantises x, the weights and h with its own quantiser;
the GPU quantiser must give the same codes and scales bit for bit.  Bar: top-k
and schedule bit-exact; rel-L2 <= 1e-2 against the oracle on the same
quantised values and <= 6e-2 against the unquantised oracle; bitwise
determinism across scheduling knobs."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from routing_grouped_expert_gemm_gb300 import build
    build.build()


def mx_inputs(T, D, I, E, k, I_s, cid, beta=0.3):
    shape = mi.custom_shape(T, D, I, E, k, I_s, config_id=cid, precision="mxfp8")
    inp = mi.make_inputs(shape, calibration={"beta": None, "redraw": {}})
    if beta:
        inp.b_router = (beta * mi.normal_f64(shape.seed, 99, E)).astype(np.float32)
    return inp


def oracle_mx_weights(inp):
    s = inp.shape
    mx = {}
    for name, w, rows, K in (("up", inp.w_up, s.E * s.I, s.D), ("gate", inp.w_gate, s.E * s.I, s.D),
                             ("down", inp.w_down, s.E * s.D, s.I)):
        q, sc = oracle.mx_quantize(w.reshape(rows, K))
        mx[name + "_q"], mx[name + "_s"] = q, sc
    return mx


def test_quantizer_matches_oracle_bitwise():
    import gpu_util
    import routing_grouped_expert_gemm_gb300 as rg
    rng = np.random.default_rng(21)
    rows, K = 384, 512
    v = rng.normal(size=(rows, K)) * np.exp(rng.normal(size=(rows, 1)) * 3)
    v[5, :32] = 0.0  # an all-zero block
    bits = mi.f32_to_bf16_bits(v.astype(np.float32))
    plan = rg.moe_plan_create(128, 256, 128, 8, 2, 0)
    q = torch.empty((rows, K), dtype=torch.uint8, device="cuda")
    sc = torch.empty(rg.moe_mxfp8_scale_bytes(rows, K), dtype=torch.uint8, device="cuda")
    rg.moe_quantize_mxfp8(plan, gpu_util.to_dev_bf16(bits), rows, K, q, sc)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.mx_quantize(bits)
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(gpu_util.scale_blocks_to_rows(sc.cpu().numpy(), rows, K), s_ref)


def run_mx(inp, **plan_kw):
    import gpu_util
    layer = gpu_util.Layer(inp, **plan_kw)
    res = layer.run(gpu_util.to_dev_bf16(inp.x), poison=True)
    assert res["status"] == 0
    return layer, res


def check_mx(inp, res, rows=None, bound_unquantised=6e-2):
    import gpu_util
    from test_gpu_parity import compare_routing
    T = inp.T
    rows = np.arange(T) if rows is None else rows
    mx = oracle_mx_weights(inp)
    ref_mx, idx_ref, g_ref = oracle.moe_fwd_inputs(inp, rows=rows, mx=mx)
    ref_bf, _, _ = oracle.moe_fwd_inputs(inp, rows=rows)
    if len(rows) == T:
        compare_routing(res, idx_ref, g_ref, inp.shape.E)
    got = gpu_util.bf16_dev_to_f64(res["out"])[rows]
    assert np.isfinite(got).all()
    rel_mx = gpu_util.rel_l2(got, ref_mx)
    rel_bf = gpu_util.rel_l2(got, ref_bf)
    assert rel_mx <= 1e-2, f"rel-L2 vs the MX oracle {rel_mx:.3g}"
    assert rel_bf <= bound_unquantised, f"rel-L2 vs the unquantised oracle {rel_bf:.3g}"
    return rel_mx, rel_bf


@pytest.mark.parametrize("dispatch", ["ring", "direct", "spread"])
def test_mx_layer_small_all_tokens(dispatch):
    inp = mx_inputs(600, 512, 256, 16, 4, 256, cid=500)
    _, res = run_mx(inp, minibatch=512, ring_slots=2, gather_ctas=3, dispatch=dispatch)
    check_mx(inp, res)


def test_mx_layer_ragged_no_shared():
    # No bf16 shared expert dilutes the format error here: four E4M3 roundings
    # (x, W_up/W_gate, h, W_down; 3 mantissa bits, ~2.5-3.5% rms each) put the
    # layer ~7% from the unquantised result, so the unquantised bound is 1e-1;
    # the 1e-2 bound against the oracle on the same quantised values is the
    # parity bar and is unchanged.
    inp = mx_inputs(333, 256, 128, 8, 3, 0, cid=501)
    _, res = run_mx(inp, minibatch=256, ring_slots=2, gather_ctas=2)
    check_mx(inp, res, bound_unquantised=1e-1)


def test_mx_bitwise_deterministic_across_knobs():
    inp = mx_inputs(700, 512, 256, 16, 4, 256, cid=502)
    outs = []
    for kw in (dict(minibatch=512, ring_slots=2, gather_ctas=3), dict(minibatch=512, ring_slots=2, gather_ctas=3),
               dict(minibatch=128, ring_slots=3, gather_ctas=1, lag=0), dict(minibatch=4096, ring_slots=1,
                                                                              gather_ctas=8, lag=0),
               dict(minibatch=512, ring_slots=2, dispatch="direct"),
               dict(minibatch=256, ring_slots=2, dispatch="spread"),
               dict(minibatch=128, ring_slots=1, lag=0, dispatch="direct")):
        _, res = run_mx(inp, **kw)
        outs.append(res["out"].view(torch.int16).cpu().numpy())
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


# Full-size DSV3 MXFP8 (every dispatch mode, CTA pairs, the minibatch sweep):
# tests/test_gpu_dsv3_full.py.


# CTA pairs (mma_pair = 1): one block-scaled tcgen05.mma.cta_group::2 per
# expert tile over two 128-row M-tiles; each CTA's scale blocks come in with
# the pair's tensor-map loads and the even CTA copies them into both CTAs'
# TMEM.  Same bars as the one-CTA kernel.
@pytest.mark.parametrize("dispatch", ["ring", "spread"])
def test_mx_pair_layer_small_all_tokens(dispatch):
    inp = mx_inputs(600, 512, 256, 16, 4, 256, cid=510)
    _, res = run_mx(inp, minibatch=512, ring_slots=2, gather_ctas=2, dispatch=dispatch, mma_pair=1)
    check_mx(inp, res)


@pytest.mark.parametrize("T", [1, 129, 333])
def test_mx_pair_ragged_no_shared(T):
    # T = 1: every expert tile is one token plus an empty partner
    import gpu_util
    inp = mx_inputs(333, 256, 128, 8, 3, 0, cid=511)
    layer = gpu_util.Layer(inp, minibatch=256, ring_slots=2, gather_ctas=2, mma_pair=1)
    res = layer.run(gpu_util.to_dev_bf16(inp.x[:T]), T, poison=True)
    assert res["status"] == 0
    check_mx(inp, res, rows=np.arange(T), bound_unquantised=1e-1)


def test_mx_pair_bitwise_deterministic_across_knobs():
    inp = mx_inputs(700, 512, 256, 16, 4, 256, cid=512)
    outs = []
    for kw in (dict(minibatch=512, ring_slots=2, gather_ctas=2), dict(minibatch=512, ring_slots=2, gather_ctas=2),
               dict(minibatch=128, ring_slots=3, gather_ctas=2, lag=0),
               dict(minibatch=4096, ring_slots=1, gather_ctas=8, lag=0, gemm_ctas=10),
               dict(minibatch=256, ring_slots=2, dispatch="spread"),
               dict(minibatch=512, ring_slots=3, dispatch="spread", raster=2)):
        _, res = run_mx(inp, mma_pair=1, **kw)
        outs.append((kw, res["out"].view(torch.int16).cpu().numpy()))
    for kw, o in outs[1:]:
        assert np.array_equal(o, outs[0][1]), f"output bits differ for {kw}"
