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
    rc = rg.testing_lib().moe_testing_pair_tile(dA.data_ptr(), dB.data_ptr(), dD.data_ptr(), st.data_ptr(), m,
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


def run_mx_pair(mode, seed=23):
    import routing_grouped_expert_gemm_gb300 as rg
    from test_gpu_mx_probe import e4m3_values, random_codes, sf_block
    rng = np.random.default_rng(seed)
    A = random_codes(rng, (256, 128))
    B = random_codes(rng, (256, 128))
    sfa = rng.integers(118, 136, size=(256, 4)).astype(np.uint8)
    sfb = rng.integers(118, 136, size=(256, 4)).astype(np.uint8)
    a, b = e4m3_values(A), e4m3_values(B)
    want = np.zeros((256, 256))
    for kb in range(4):
        want += (a[:, 32 * kb:32 * kb + 32] @ b[:, 32 * kb:32 * kb + 32].T) * \
            np.exp2(sfa[:, kb].astype(np.float64) - 127)[:, None] * np.exp2(sfb[:, kb].astype(np.float64) - 127)[None, :]
    blocks = np.concatenate([sf_block(sfa[:128]), sf_block(sfa[128:]), sf_block(sfb[:128]), sf_block(sfb[128:])])
    dA, dB, dS = (torch.from_numpy(v).cuda() for v in (A, B, blocks))
    dD = torch.full((256, 256), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(3, dtype=torch.int32, device="cuda")
    rc = rg.testing_lib().moe_testing_pair_mx_tile(dA.data_ptr(), dB.data_ptr(), dS.data_ptr(), dD.data_ptr(), st.data_ptr(),
                                           mode, torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [0, 0, 0]
    return dD.cpu().numpy().astype(np.float64), want


def test_pair_mx_tile_scale_placement():
    """Block-scaled cta_group::2: each CTA's TMEM holds the A scales of its own
    128 rows and the B scales of all 256 N rows (two blocks, as for one CTA)
    -- the even CTA's tcgen05.cp.cta_group::2 fills both CTAs from their own
    shared memory.  (Holding only its own B half's block gives wrong columns in
    the other CTA's half.)"""
    got, want = run_mx_pair(1)
    assert np.isfinite(got).all()
    np.testing.assert_allclose(got, want, rtol=1e-5, atol=1e-6 * np.abs(want).max())
