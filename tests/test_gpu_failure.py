"""Failure detection of the persistent forward kernel, without a GPU fault.

Every device-side wait has a time limit; when one runs out the kernel records
MOE_STATUS_TIMEOUT in the workspace status word, every other wait sees the
word and gives up, and the kernel returns normally.  The test hook
``test_unfilled_minibatch`` makes the ring fill never mark one minibatch as
gathered (a flag that nothing sets), so the expert tiles that wait for it run
out of time: the forward must end, report MOE_STATUS_TIMEOUT, and leave the
stream and the workspace usable for a normal forward that then matches the
fp64 oracle.  The one-CTA kernel is used (ring and spread dispatch).

The fp16 staging rows saturate at +-65504: a layer whose expert outputs leave
that range must say so through MOE_STATUS_STAGING_OVERFLOW rather than return
MOE_STATUS_OK with a wrong result, with one CTA per tile and with CTA pairs.
"""
import time

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


@pytest.mark.parametrize("dispatch", ["ring", "spread"])
def test_wait_that_runs_out_reports_timeout_and_the_workspace_recovers(dispatch):
    import gpu_util
    import routing_grouped_expert_gemm_gb300 as rg

    inp = mi.make_inputs("tiny")
    s = inp.shape
    kw = dict(minibatch=512, ring_slots=2, gather_ctas=2, dispatch=dispatch)
    # minibatch 0 is never marked gathered; every wait gives up after 50 ms
    faulty = gpu_util.Layer(inp, timeout_ms=50, test_unfilled_minibatch=1, **kw)
    x = gpu_util.to_dev_bf16(inp.x)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    res = faulty.run(x)
    wall = time.perf_counter() - t0
    assert res["status"] == rg.MOE_STATUS_TIMEOUT
    assert wall < 5.0, f"the aborted forward took {wall:.2f} s"
    # the same workspace, a plan with the same layout and no hook: a normal forward
    good = gpu_util.Layer(inp, **kw)
    assert good.ws_bytes == faulty.ws_bytes
    good.ws = faulty.ws
    res = good.run(x)
    assert res["status"] == rg.MOE_STATUS_OK
    ref, idx_ref, _ = oracle.moe_fwd_inputs(inp)
    assert np.array_equal(res["topk_idx"].cpu().numpy(), idx_ref)
    gpu_util.check_out(gpu_util.bf16_dev_to_f64(res["out"]), ref)


@pytest.mark.parametrize("mma_pair", [0, 1])
def test_staging_overflow_is_reported(mma_pair):
    # one CTA per tile (staged epilogue stores) and CTA pairs (rows stored from registers)
    import gpu_util
    import routing_grouped_expert_gemm_gb300 as rg

    shape = mi.custom_shape(256, 256, 128, 16, 4, 128, config_id=320)
    inp = mi.make_inputs(shape, calibration={"beta": None, "redraw": {}})
    layer = gpu_util.Layer(inp, minibatch=512, ring_slots=2, gather_ctas=2, mma_pair=mma_pair)
    x = gpu_util.to_dev_bf16(inp.x)
    assert layer.run(x)["status"] == rg.MOE_STATUS_OK
    # expert outputs ~N(0, 1) scaled by 2^17: far outside the fp16 range of the staging rows
    big = mi.f32_to_bf16_bits(mi.bf16_bits_to_f32(inp.w_down) * np.float32(2.0 ** 17))
    layer.w["W_down"] = gpu_util.to_dev_bf16(big)
    res = layer.run(x)
    assert res["status"] == rg.MOE_STATUS_STAGING_OVERFLOW
    assert torch.isfinite(res["out"].float()).all()
    # the warning is cleared by the next forward
    layer.w["W_down"] = gpu_util.to_dev_bf16(inp.w_down)
    assert layer.run(x)["status"] == rg.MOE_STATUS_OK
