"""Pins the MN-major operand encoding of the bf16 tcgen05 MMA on one tile
against a CPU matmul.  The backward pass contracts over tokens (weight
gradients) and over the forward weights' output dimension (input gradients),
so its operands arrive with the M or N index contiguous: the transpose bits of
the instruction descriptor and, in the shared-memory descriptor, the byte
offsets between 64-wide MN blocks (8192 B, the next TMA box) and between 8-row
K groups (1024 B) are what the backward kernels rely on."""
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


def _tile(N, a_mn, b_mn, lbo, sbo, seed):
    import routing_grouped_expert_gemm_gb300 as rg
    rng = np.random.default_rng(seed)
    A = torch.from_numpy(rng.normal(size=(128, 64)).astype(np.float32)).to(torch.bfloat16)
    B = torch.from_numpy(rng.normal(size=(N, 64)).astype(np.float32)).to(torch.bfloat16)
    ref = A.double().numpy() @ B.double().numpy().T
    dA, dB = A.cuda(), B.cuda()
    dD = torch.full((128, N), float("nan"), dtype=torch.float32, device="cuda")
    rc = rg.testing_lib().moe_testing_mn_tile(dA.data_ptr(), dB.data_ptr(), dD.data_ptr(), N, a_mn, b_mn, lbo, sbo,
                                              torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    return dD.double().cpu().numpy(), ref


@pytest.mark.parametrize("N", [128, 256])
@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_mn_major_operands(N, a_mn, b_mn):
    got, ref = _tile(N, a_mn, b_mn, 8192, 1024, seed=7 + N + 2 * a_mn + b_mn)
    # fp32 accumulation of 64 exact bf16 products
    np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-4)


def test_the_other_reading_of_the_offsets_differs():
    """With leading and stride offsets exchanged the MN-major tile is wrong:
    the pin above distinguishes the two readings."""
    got, ref = _tile(256, 1, 1, 1024, 8192, seed=99)
    assert not np.allclose(got, ref, rtol=1e-3, atol=1e-2)
