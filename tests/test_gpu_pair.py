"""The CTA-pair flavour of the persistent kernel (mma_pair = 1: each expert
tile is one tcgen05.mma.cta_group::2 over two 128-row M-tiles that share the
weight tile) against the fp64 oracle, with the same bars as the one-CTA
kernel: routing and schedule bit-exact, outputs within rel-L2 1e-2 and
max-abs 3e-2 rms, repeated runs and scheduling knobs bitwise identical.

The cases cover segments with an odd number of M-tiles (with bf16 the last
tile is split over the pair, 64 rows per CTA in one M = 128 MMA; with MXFP8,
or pad_odd_tiles = 1, the pair's second task is an empty partner), a single
token, a ragged token tail, no shared expert, one expert taking every token
and the full-size DSV3 workload."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from test_gpu_parity import _full_size, run_and_check, small

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from routing_grouped_expert_gemm_gb300 import build
    build.build()


def test_pair_tiny_workload_all_tokens():
    run_and_check(mi.make_inputs("tiny"), minibatch=512, ring_slots=2, gather_ctas=2, mma_pair=1)


def test_pair_medium_ragged_tokens_and_tiles():
    run_and_check(small(1000, 512, 256, 32, 6, 256), minibatch=1024, ring_slots=3, gather_ctas=4, mma_pair=1)


@pytest.mark.parametrize("T", [1, 129, 300])
def test_pair_edge_token_counts(T):
    inp = small(384, 256, 128, 16, 4, 128, cid=301)
    run_and_check(inp, T=T, minibatch=128, ring_slots=2, gather_ctas=2, mma_pair=1)


def test_pair_no_shared_expert_softmax():
    run_and_check(small(384, 512, 256, 24, 5, 0, score="softmax", cid=302, beta_scale=0.0), minibatch=512,
                  gather_ctas=2, mma_pair=1)


def test_pair_one_expert_takes_every_token():
    inp = small(640, 256, 128, 16, 3, 128, cid=304)
    inp.b_router[7] = 40.0
    _, _, res = run_and_check(inp, minibatch=256, ring_slots=2, gather_ctas=2, mma_pair=1)
    assert res["expert_counts"].cpu().numpy()[7] == 640


def test_pair_bitwise_deterministic_across_knobs():
    import gpu_util as g
    inp = small(1000, 512, 256, 32, 6, 256, cid=307)
    x = g.to_dev_bf16(inp.x)
    outs = []
    for kw in (dict(minibatch=1024, ring_slots=3, gather_ctas=4, lag=1),
               dict(minibatch=1024, ring_slots=3, gather_ctas=4, lag=1),
               dict(minibatch=128, ring_slots=2, gather_ctas=2, lag=1),
               dict(minibatch=256, ring_slots=1, gather_ctas=8, lag=0),
               dict(minibatch=8192, ring_slots=1, gather_ctas=2, lag=0, gemm_ctas=20),
               dict(minibatch=512, ring_slots=5, gather_ctas=16, lag=1, gemm_ctas=6),
               dict(minibatch=1024, ring_slots=3, gather_ctas=4, raster=2),
               dict(minibatch=256, ring_slots=2, gather_ctas=2, raster=3),
               dict(minibatch=512, ring_slots=3, dispatch="spread")):
        layer = g.Layer(inp, mma_pair=1, **kw)
        res = layer.run(x, poison=True)
        assert res["status"] == 0
        outs.append((kw, res["out"].view(torch.int16).cpu().numpy()))
    for kw, o in outs[1:]:
        assert np.array_equal(o, outs[0][1]), f"output bits differ for {kw}"


@pytest.mark.parametrize("precision", ["bf16", "mxfp8"])
def test_pair_plain_launch_is_bitwise_identical(precision):
    """The profiling launch (no cooperative attribute; the grid still fits the
    GPU) gives the bits of the cooperative launch."""
    import gpu_util as g
    inp = small(1000, 512, 256, 32, 6, 256, cid=313)
    if precision == "mxfp8":
        inp = mi.make_inputs(mi.custom_shape(1000, 512, 256, 32, 6, 256, config_id=313, precision="mxfp8"),
                             calibration={"beta": None, "redraw": {}})
    x = g.to_dev_bf16(inp.x)
    outs = []
    for plain in (0, 1):
        layer = g.Layer(inp, minibatch=512, ring_slots=3, dispatch="spread", mma_pair=1, plain_launch=plain)
        res = layer.run(x, poison=True)
        assert res["status"] == 0
        outs.append(res["out"].view(torch.int16).cpu().numpy())
    assert np.array_equal(outs[0], outs[1])


def test_pair_padded_odd_tiles_against_oracle():
    # the empty-partner form of an odd segment's last M-tile (bf16)
    run_and_check(small(1000, 512, 256, 32, 6, 256, cid=315), minibatch=1024, ring_slots=3, gather_ctas=4,
                  mma_pair=1, pad_odd_tiles=1)


@pytest.mark.parametrize("T", [1, 64, 65, 300])
def test_pair_split_tail_tiles_bitwise_equal_to_padded(T):
    """Splitting an odd segment's last M-tile over the pair (64 rows per CTA,
    one M = 128 MMA) gives the bits of the padded form (one M = 256 MMA with an
    empty partner); T = 64 / 65 put a tile edge at the split."""
    import gpu_util as g
    inp = small(1000, 512, 256, 32, 6, 256, cid=316)
    x = g.to_dev_bf16(inp.x[:T])
    for kw in (dict(minibatch=512, ring_slots=3, dispatch="spread"),
               dict(minibatch=256, ring_slots=2, gather_ctas=2, raster=2)):
        outs = []
        for pad in (1, 0):
            layer = g.Layer(inp, T_max=inp.T, mma_pair=1, pad_odd_tiles=pad, **kw)
            res = layer.run(x, T, poison=True)
            assert res["status"] == 0
            outs.append(res["out"].view(torch.int16).cpu().numpy())
        assert np.array_equal(outs[0], outs[1]), f"output bits differ for {kw}"


def test_pair_rejects_unsupported_modes():
    import routing_grouped_expert_gemm_gb300 as rg
    for kw in (dict(precision="mxfp8", dispatch="direct"), dict(dispatch="direct"), dict(gather_ctas=3)):
        with pytest.raises(rg.MoEError):
            rg.moe_plan_create(256, 256, 128, 16, 4, 128, mma_pair=1, **kw)


def test_pair_full_size_kimi_k2_sampled():
    # the largest configured shape: T = 32768, E = 384 (uniform load), one shared expert
    _full_size("kimi_k2", minibatch=8192, ring_slots=4, gather_ctas=8, mma_pair=1)
