"""Pins the CTA-pair tcgen05 MMA (cta_group::2) on one 256 x 256 x 64 tile
against a CPU matmul: TMEM allocated for both CTAs, each CTA's TMA loads
counted on the even CTA's mbarrier, the M = 256 instruction descriptor, A and
B each split 128 rows per CTA, the multicast commit, and D rows [128 r, 128 r
+ 128) landing in CTA r's TMEM lanes 0..127."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from routing_grouped_expert_gemm_gb300 import build
    build.build()


def test_pair_mma_tile():
    import routing_grouped_expert_gemm_gb300 as rg
    g = torch.Generator().manual_seed(11)
    A = torch.randn(256, 64, generator=g).to(torch.bfloat16)
    B = torch.randn(256, 64, generator=g).to(torch.bfloat16)
    want = A.double() @ B.double().T
    dA, dB = A.cuda(), B.cuda()
    dD = torch.full((256, 256), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(3, dtype=torch.int32, device="cuda")
    rc = rg.lib().moe_testing_pair_tile(dA.data_ptr(), dB.data_ptr(), dD.data_ptr(), st.data_ptr(),
                                        torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [0, 0, 0]
    got = dD.cpu().double()
    assert torch.isfinite(got).all()
    # 64 exact bf16 products summed in fp32
    torch.testing.assert_close(got, want, rtol=1e-5, atol=1e-5 * want.abs().max().item())
