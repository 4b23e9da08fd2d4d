"""The C ABI without a GPU: the library builds for sm_103a, loads, exports
every function include/moe.h declares, and validates arguments on the host."""
import ctypes
import subprocess

import pytest
import torch

import routing_grouped_expert_gemm_gb300 as rg
from routing_grouped_expert_gemm_gb300 import build as rgbuild


@pytest.fixture(scope="module")
def L():
    rgbuild.build()
    return rg.lib()


EXPECTED = {"moe_plan_create", "moe_plan_destroy", "moe_workspace_bytes", "moe_quantize_mxfp8",
            "moe_mxfp8_scale_bytes", "moe_fwd", "moe_get_status", "moe_error_string",
            "moe_plan_set_timing_events", "moe_get_phase_times", "moe_route_static", "moe_route_static_scratch_bytes",
            "moe_bwd", "moe_bwd_workspace_bytes", "moe_plan_set_bwd_timing_events"}


def test_header_declares_the_boundary():
    assert EXPECTED <= set(rg.declared_functions())


def _exported(path):
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
    return {line.split()[-1] for line in out.splitlines() if " T " in line}


def test_library_exports_every_declared_function(L):
    exported = _exported(rg.LIB_PATH)
    for name in rg.declared_functions():
        assert name in exported, name
        assert getattr(L, name) is not None


def test_test_hooks_live_in_their_own_library(L):
    """The one-tile probes (include/moe_testing.h) ship in the test-hook
    library only; the product library exports none of them."""
    hooks = rg.declared_functions(rg.TESTING_HEADER_PATH)
    assert hooks and all(h.startswith("moe_testing_") for h in hooks)
    exported = _exported(rg.TESTING_LIB_PATH)
    T = rg.testing_lib()
    for name in hooks:
        assert name in exported, name
        assert getattr(T, name) is not None
    assert not any(n.startswith("moe_testing_") for n in _exported(rg.LIB_PATH))


def test_error_strings(L):
    assert rg.moe_error_string(0) == "ok"
    assert "workspace" in rg.moe_error_string(rg.MOE_ERR_WORKSPACE_TOO_SMALL)
    assert rg.moe_error_string(123) == "unknown error"


@pytest.mark.parametrize("kw", [
    dict(D=100), dict(D=384), dict(I=96), dict(E=0), dict(E=513), dict(k=0), dict(k=17), dict(k=9, E=8),
    dict(I_s=100), dict(minibatch=100), dict(minibatch=65536), dict(ring_slots=1, lag=1),
])
def test_plan_rejects_unsupported_shapes(L, kw):
    base = dict(T_max=256, D=256, I=128, E=16, k=4, I_s=128)
    base.update(kw)
    with pytest.raises(rg.MoEError) as ei:
        rg.moe_plan_create(**base)
    assert ei.value.code == rg.MOE_ERR_UNSUPPORTED_SHAPE


def test_plan_rejects_bad_enums(L):
    for kw in (dict(score_fn=7), dict(precision=9), dict(lag=3)):
        with pytest.raises(rg.MoEError) as ei:
            rg.moe_plan_create(T_max=256, D=256, I=128, E=16, k=4, **kw)
        assert ei.value.code == rg.MOE_ERR_INVALID_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_plan_create_without_gpu_fails_cleanly(L):
    with pytest.raises(rg.MoEError) as ei:
        rg.moe_plan_create(T_max=256, D=256, I=128, E=16, k=4, I_s=128)
    assert ei.value.code in (rg.MOE_ERR_CUDA, rg.MOE_ERR_UNSUPPORTED_DEVICE)


def test_null_arguments(L):
    assert L.moe_plan_create(None, None) == rg.MOE_ERR_INVALID_ARG
    assert L.moe_workspace_bytes(None, 10) == 0
    assert L.moe_fwd(None, 1, None, None, None, None, 0, None) == rg.MOE_ERR_INVALID_ARG
    st = ctypes.c_int()
    assert L.moe_get_status(None, None, ctypes.byref(st), None) == rg.MOE_ERR_INVALID_ARG
    assert L.moe_plan_destroy(None) == 0
    assert L.moe_mxfp8_scale_bytes(128, 64) == 256


def test_plan_rejects_bad_knobs(L):
    # CTA pairs need ring or spread dispatch and even CTA counts; the knobs' ranges
    base = dict(T_max=256, D=256, I=128, E=16, k=4, I_s=128)
    for kw in (dict(mma_pair=1, dispatch="direct"), dict(mma_pair=1, gather_ctas=3), dict(mma_pair=1, gemm_ctas=5),
               dict(mma_pair=1, precision="mxfp8", dispatch="direct"), dict(mma_pair=2), dict(raster=-1),
               dict(l2_prefetch=65), dict(dispatch=7), dict(gemm_ctas=-1),
               dict(test_unfilled_minibatch=-1), dict(test_unfilled_minibatch=1, dispatch="direct"),
               dict(clc=2), dict(clc=1, mma_pair=1), dict(plain_launch=2), dict(plain_launch=-1),
               dict(pad_odd_tiles=2), dict(pad_odd_tiles=-1, mma_pair=1)):
        with pytest.raises(rg.MoEError) as ei:
            rg.moe_plan_create(**base, **kw)
        assert ei.value.code == rg.MOE_ERR_INVALID_ARG, kw


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_valid_knobs_pass_validation(L):
    # accepted configurations get as far as the device query (which fails without a GPU)
    base = dict(T_max=256, D=256, I=128, E=16, k=4, I_s=128)
    for kw in (dict(mma_pair=1), dict(mma_pair=1, precision="mxfp8", dispatch="spread"),
               dict(mma_pair=1, gather_ctas=3, dispatch="spread"), dict(dispatch="direct", precision="mxfp8"),
               dict(raster=3, mma_pair=1), dict(k=16, E=512, I_s=0), dict(test_unfilled_minibatch=1),
               dict(test_unfilled_minibatch=2, dispatch="spread"), dict(clc=1), dict(clc=1, dispatch="spread"),
               dict(plain_launch=1), dict(plain_launch=1, mma_pair=1), dict(pad_odd_tiles=1, mma_pair=1)):
        with pytest.raises(rg.MoEError) as ei:
            rg.moe_plan_create(**{**base, **kw})
        assert ei.value.code in (rg.MOE_ERR_CUDA, rg.MOE_ERR_UNSUPPORTED_DEVICE), kw
