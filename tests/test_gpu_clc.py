"""Cluster launch control scheduling (plan option clc = 1; "Mixture-of-Kittens:
MoE Megakernel for NVL72s", Sec. 3.4 "RDMA Overlap via Cluster Launch
Control") against the default persistent scheduling and the fp64 oracle.

With clc the persistent kernel is launched with one CTA per task; each running
CTA cancels the launch of a CTA that has not started and spends its token on
the next unit of the global task order.  The unit order is the same as with
the cooperative persistent grid, and each output element's arithmetic does
not depend on which CTA computes it, so the outputs must be bitwise equal."""
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


def _small(T, D, I, E, k, I_s, cid, precision="bf16"):
    shape = mi.custom_shape(T, D, I, E, k, I_s, config_id=cid, precision=precision)
    inp = mi.make_inputs(shape, calibration={"beta": None, "redraw": {}})
    inp.b_router = (0.3 * mi.normal_f64(shape.seed, 99, E)).astype(np.float32)
    return inp


@pytest.mark.parametrize("dispatch", ["ring", "spread", "direct"])
@pytest.mark.parametrize("precision", ["bf16", "mxfp8"])
def test_clc_matches_default_scheduling_bitwise(dispatch, precision):
    import gpu_util
    inp = _small(1000, 512, 256, 32, 6, 256, cid=800, precision=precision)
    x = gpu_util.to_dev_bf16(inp.x)
    kw = dict(minibatch=1024, ring_slots=3, gather_ctas=4, dispatch=dispatch)
    ref_layer = gpu_util.Layer(inp, **kw)
    ref = ref_layer.run(x, poison=True)
    assert ref["status"] == 0
    layer = gpu_util.Layer(inp, weights=ref_layer.w, clc=1, **kw)
    got = layer.run(x, poison=True)
    assert got["status"] == 0
    assert torch.equal(got["out"].view(torch.int16), ref["out"].view(torch.int16))
    for key in ("topk_idx", "sched", "route_row"):
        assert torch.equal(got[key], ref[key]), key


def test_clc_combine_over_several_chunks_per_cta():
    """Enough combine rounds (4096 tokens x 8 column tiles) that CTAs claim
    several chunks each: the chunked combine must still be bitwise the default."""
    import gpu_util
    inp = _small(4096, 2048, 256, 16, 4, 256, cid=802)
    x = gpu_util.to_dev_bf16(inp.x)
    ref_layer = gpu_util.Layer(inp, minibatch=4096, ring_slots=2, gather_ctas=4)
    ref = ref_layer.run(x)
    layer = gpu_util.Layer(inp, weights=ref_layer.w, minibatch=4096, ring_slots=2, gather_ctas=4, clc=1)
    got = layer.run(x, poison=True)
    assert ref["status"] == 0 and got["status"] == 0
    assert torch.equal(got["out"].view(torch.int16), ref["out"].view(torch.int16))


def test_clc_tiny_all_tokens_against_oracle():
    import gpu_util
    inp = mi.make_inputs("tiny")
    layer = gpu_util.Layer(inp, minibatch=512, ring_slots=2, gather_ctas=2, clc=1)
    res = layer.run(gpu_util.to_dev_bf16(inp.x), poison=True)
    assert res["status"] == 0
    ref, idx_ref, _ = oracle.moe_fwd_inputs(inp)
    assert np.array_equal(res["topk_idx"].cpu().numpy(), idx_ref)
    gpu_util.check_out(gpu_util.bf16_dev_to_f64(res["out"]), ref)


def test_clc_repeated_runs_and_knobs():
    import gpu_util
    inp = _small(700, 512, 256, 16, 4, 256, cid=801)
    x = gpu_util.to_dev_bf16(inp.x)
    outs = []
    for kw in (dict(minibatch=512, ring_slots=2, gather_ctas=3), dict(minibatch=512, ring_slots=2, gather_ctas=3),
               dict(minibatch=128, ring_slots=1, gather_ctas=1, lag=0), dict(minibatch=4096, ring_slots=2,
                                                                             dispatch="spread")):
        layer = gpu_util.Layer(inp, clc=1, **kw)
        res = layer.run(x, poison=True)
        assert res["status"] == 0
        outs.append(res["out"].view(torch.int16).cpu().numpy())
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


def test_clc_needs_the_one_cta_kernel():
    import routing_grouped_expert_gemm_gb300 as rg
    with pytest.raises(rg.MoEError) as ei:
        rg.moe_plan_create(256, 256, 128, 16, 4, 128, mma_pair=1, clc=1)
    assert ei.value.code == rg.MOE_ERR_INVALID_ARG
