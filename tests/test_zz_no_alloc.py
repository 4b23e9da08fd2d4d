"""moe_route_static: the routing stage for callers that cannot allocate device
memory (a framework that owns every device byte, or a loop where cudaMalloc's
possible device synchronisation is not allowed).  Its scratch is a fixed array
inside the library, shared by every call.

Checked through the C ABI against what moe_fwd exports for the same inputs,
on two calls in a row with different token counts (the second call finds the
first call's leftovers in the shared array), and against the fp64 oracle's
routing; once more at the documented limits (T = 16384 tokens, E = 512
experts, k = 16), where the scratch is fullest.  The file sorts last so that
a run which stops at the first failure has run every other test before it.
"""
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


GAP = 1e-3  # the inputs' top-k gap rule: fp32 and fp64 logits then select alike


def _inputs(T, cid, D=1024, E=64, k=6):
    """Seeded inputs whose rows keep the k-th and (k+1)-th biased router logits
    at least GAP apart (a row that does not is redrawn, as the stored workloads'
    calibration does)."""
    shape = mi.custom_shape(T, D, 256 if D >= 256 else 128, E, k, 0, config_id=cid)
    inp = mi.make_inputs(shape, calibration={"beta": None, "redraw": {}})
    inp.b_router = (0.3 * mi.normal_f64(shape.seed, 99, shape.E)).astype(np.float32)
    beta = inp.b_router.astype(np.float64)
    attempt = np.zeros(T, dtype=np.int32)
    logits = oracle.router_logits(inp.x, inp.w_router, None) + beta
    for _ in range(50):
        part = -np.partition(-logits, k, axis=1)[:, :k + 1]
        part.sort(axis=1)
        bad = np.nonzero(part[:, 1] - part[:, 0] < GAP)[0]
        if bad.size == 0:
            return inp
        attempt[bad] += 1
        for t in bad:
            inp.x[t] = mi.x_rows(shape.seed, T, D, attempt, int(t), 1)[0]
        logits[bad] = oracle.router_logits(inp.x[bad], inp.w_router, None) + beta
    raise RuntimeError("gap rule did not converge")


def _check_oracle(inp, got):
    """Routing of route_static against the fp64 oracle: top-k and the schedule
    bit-exact, g within the parity tests' 5e-5 relative."""
    s = inp.shape
    logits = oracle.router_logits(inp.x, inp.w_router, inp.b_router)
    idx_ref, g_ref = oracle.topk(logits, s.k, s.score)
    assert np.array_equal(got["topk_idx"].cpu().numpy(), idx_ref)
    np.testing.assert_allclose(got["topk_w"].cpu().numpy(), g_ref, rtol=5e-5, atol=1e-7)
    M, S, sched, route_row = oracle.schedule(idx_ref, s.E)
    assert np.array_equal(got["expert_counts"].cpu().numpy(), M)
    assert np.array_equal(got["expert_offsets"].cpu().numpy(), S)
    assert np.array_equal(got["sched"].cpu().numpy(), sched)
    assert np.array_equal(got["route_row"].cpu().numpy(), route_row)


def _route_static(rg, layer, x, T):
    s = layer.shape
    R = T * s.k
    o = dict(topk_idx=torch.full((T, s.k), -1, dtype=torch.int32, device="cuda"),
             topk_w=torch.full((T, s.k), -1.0, dtype=torch.float32, device="cuda"),
             expert_counts=torch.full((s.E,), -1, dtype=torch.int32, device="cuda"),
             expert_offsets=torch.full((s.E + 1,), -1, dtype=torch.int32, device="cuda"),
             sched=torch.full((R, 3), -1, dtype=torch.int32, device="cuda"),
             route_row=torch.full((R,), -1, dtype=torch.int32, device="cuda"))
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    rg.moe_route_static(layer.plan, T, x, layer.w["W_router"], layer.w["b_router"], o["topk_idx"], o["topk_w"],
                        o["expert_counts"], o["expert_offsets"], o["sched"], o["route_row"], device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return o


def test_route_static_matches_moe_fwd_on_two_calls_in_a_row():
    import gpu_util
    import routing_grouped_expert_gemm_gb300 as rg

    refs, gots, inps = [], [], []
    for inp in (_inputs(3000, 401), _inputs(777, 402)):  # two calls in a row on the shared scratch
        inps.append(inp)
        layer = gpu_util.Layer(inp, minibatch=1024)
        x = gpu_util.to_dev_bf16(inp.x)
        gots.append(_route_static(rg, layer, x, inp.T))
        refs.append(layer.run(x, inp.T))
    for got, ref in zip(gots, refs):
        assert ref["status"] == 0
        for key in ("topk_idx", "expert_counts", "expert_offsets", "sched", "route_row"):
            assert torch.equal(got[key], ref[key]), key
        # same tolerance as the parity tests (the two paths run the same kernels)
        np.testing.assert_allclose(got["topk_w"].cpu().numpy(), ref["topk_w"].cpu().numpy(), rtol=5e-5, atol=1e-7)
    for inp, got in zip(inps, gots):
        _check_oracle(inp, got)


def test_route_static_at_its_documented_limits():
    """T = MOE_ROUTE_STATIC_MAX_TOKENS, E = 512, k = 16: the largest scratch
    layout; bit-exact against moe_fwd's routing exports and the oracle."""
    import gpu_util
    import routing_grouped_expert_gemm_gb300 as rg

    inp = _inputs(rg.MOE_ROUTE_STATIC_MAX_TOKENS, 403, D=256, E=512, k=16)
    layer = gpu_util.Layer(inp, minibatch=8192)
    x = gpu_util.to_dev_bf16(inp.x)
    got = _route_static(rg, layer, x, inp.T)
    ref = layer.run(x, inp.T)
    assert ref["status"] == 0
    for key in ("topk_idx", "topk_w", "expert_counts", "expert_offsets", "sched", "route_row"):
        assert torch.equal(got[key], ref[key]), key
    _check_oracle(inp, got)


def test_route_static_rejects_requests_beyond_its_scratch():
    import routing_grouped_expert_gemm_gb300 as rg

    T = rg.MOE_ROUTE_STATIC_MAX_TOKENS + 1
    plan = rg.moe_plan_create(T, 256, 128, 16, 4, 0)
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    with pytest.raises(rg.MoEError) as ei:
        rg.moe_route_static(plan, T, dummy, dummy, None, dummy, dummy, dummy, dummy, dummy, dummy)
    assert ei.value.code == rg.MOE_ERR_STATIC_SCRATCH_TOO_SMALL
    assert rg.moe_route_static_scratch_bytes() == 512 * 1024
