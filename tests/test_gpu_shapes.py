"""The pages' four evaluated MoE layer shapes ("Mixture-of-Kittens: MoE
Megakernel for NVL72s", Sec. 4.1: Kimi K2.7 Code, GLM-5.2, Qwen3.5-397B-A17B,
DeepSeek-V4-Pro, each with one shared expert) on one GPU, against the fp64
oracle, in the launch configuration the benchmark uses (CTA pairs; ring
dispatch for BF16, spread for MXFP8).  4096 of each workload's tokens; every
token's routing bit-exact, outputs compared on sampled tokens with the bars of
the other parity tests (BF16: rel-L2 <= 1e-2 and max-abs <= 3e-2 rms; MXFP8:
rel-L2 <= 1e-2 against the oracle on the same quantised values)."""
import dataclasses

import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle

pytestmark = pytest.mark.gpu

T_TEST = 4096


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from routing_grouped_expert_gemm_gb300 import build
    build.build()


def _routing(inp, res):
    from test_gpu_parity import compare_routing
    s = inp.shape
    logits = oracle.router_logits(inp.x, inp.w_router, inp.b_router)
    idx_ref, g_ref = oracle.topk(logits, s.k, s.score)
    compare_routing(res, idx_ref, g_ref, s.E)


@pytest.mark.parametrize("name", ["kimi_k27", "glm52", "qwen35", "dsv4pro"])
def test_page_shape_bf16_sampled(name):
    import gpu_util as g
    inp = mi.make_inputs(name, T=T_TEST)
    layer = g.Layer(inp, minibatch=8192, ring_slots=4, gather_ctas=8, mma_pair=1)
    res = layer.run(g.to_dev_bf16(inp.x), poison=True)
    assert res["status"] == 0
    _routing(inp, res)
    rows = np.unique(np.linspace(0, T_TEST - 1, 24).astype(np.int64))
    ref, _, _ = oracle.moe_fwd_inputs(inp, rows=rows)
    g.check_out(g.bf16_dev_to_f64(res["out"])[rows], ref)


@pytest.mark.parametrize("name", ["glm52", "qwen35", "kimi_k27", "dsv4pro"])
def test_page_shape_mxfp8_sampled(name):
    from test_gpu_mxfp8 import check_mx, run_mx
    base = mi.make_inputs(name, T=T_TEST)
    inp = dataclasses.replace(base, shape=mi.CONFIGS[name + "_mxfp8"])
    _, res = run_mx(inp, minibatch=8192, ring_slots=4, dispatch="spread", mma_pair=1)
    _routing(inp, res)
    rows = np.unique(np.linspace(0, T_TEST - 1, 16).astype(np.int64))
    check_mx(inp, res, rows=rows)
