"""Pins the CTA-pair tcgen05 MMA (cta_group::2) on one tile against a CPU
matmul: TMEM allocated for both CTAs, each CTA's TMA loads counted on the even
CTA's mbarrier, the instruction descriptor, A and B each split over the two
CTAs, the multicast commit, and which TMEM lanes of which CTA receive which
rows of D.

M = 256: CTA r holds A rows [128 r, 128 r + 128) and its TMEM lanes 0..127
receive D rows [128 r, 128 r + 128).  M = 128 (64 A rows per CTA): each CTA's
64 rows come back split over its lane halves (columns 0..127 in lanes 0..63,
columns 128..255 in lanes 64..127), 128 TMEM columns wide."""
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


def run_tile(m, seed=11):
    import routing_grouped_expert_gemm_gb300 as rg
    g = torch.Generator().manual_seed(seed)
    A = torch.randn(m, 64, generator=g).to(torch.bfloat16)
    B = torch.randn(256, 64, generator=g).to(torch.bfloat16)
    want = (A.double() @ B.double().T).numpy()
    dA, dB = A.cuda(), B.cuda()
    dD = torch.full((2, 128, 256), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(3, dtype=torch.int32, device="cuda")
    rc = rg.lib().moe_testing_pair_tile(dA.data_ptr(), dB.data_ptr(), dD.data_ptr(), st.data_ptr(), m,
                                        torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [0, 0, 0]
    return dD.cpu().numpy().astype(np.float64), want


def test_pair_mma_tile_m256():
    got, want = run_tile(256)
    got = got.reshape(256, 256)
    assert np.isfinite(got).all()
    # 64 exact bf16 products summed in fp32
    np.testing.assert_allclose(got, want, rtol=1e-5, atol=1e-5 * np.abs(want).max())


def test_pair_mma_tile_m128_placement():
    """M = 128 over a pair: CTA r holds A rows [64 r, 64 r + 64); in its TMEM,
    lanes 0..63 hold those rows' output columns 0..127 and lanes 64..127 the
    same rows' columns 128..255, both in TMEM columns 0..127."""
    got, want = run_tile(128)
    tol = 1e-5 * np.abs(want).max()
    for r in range(2):
        rows = want[64 * r:64 * r + 64]
        np.testing.assert_allclose(got[r, :64, :128], rows[:, :128], rtol=1e-5, atol=tol)
        np.testing.assert_allclose(got[r, 64:, :128], rows[:, 128:], rtol=1e-5, atol=tol)
