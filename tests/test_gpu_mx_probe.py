"""Pins the block-scaled MXFP8 tcgen05 MMA (instruction descriptor, E8M0
scales in TMEM, scale-factor ids) on one 128 x 256 x 128 tile against a CPU
reference built from torch's float8_e4m3fn decoding and exact powers of two.

The probe takes the TMEM image of the scales from the caller, so the test can
state the placement the forward kernel relies on: A scales of row r at lane r,
B scales of column n at lane n % 128 in column n // 128, the four K-blocks of a
128-wide K step in the four bytes of that word (byte kb selected by the
scale-factor id of the kb-th MMA)."""
import ctypes

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


def e4m3_values(codes: np.ndarray) -> np.ndarray:
    return torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def reference(A, B, sfa, sfb):
    a, b = e4m3_values(A), e4m3_values(B)
    D = np.zeros((128, 256))
    for kb in range(4):
        blk = a[:, 32 * kb:32 * kb + 32] @ b[:, 32 * kb:32 * kb + 32].T
        D += blk * np.exp2(sfa[:, kb].astype(np.float64) - 127)[:, None] * \
            np.exp2(sfb[:, kb].astype(np.float64) - 127)[None, :]
    return D


def pack4(v):  # four scale bytes (kb = 0..3) -> one little-endian word
    v = v.astype(np.uint32)
    return v[..., 0] | (v[..., 1] << 8) | (v[..., 2] << 16) | (v[..., 3] << 24)


def image_lane_is_row(sfa, sfb):
    img = np.zeros((128, 12), dtype=np.uint32)
    img[:, 0] = pack4(sfa)
    img[:, 4] = pack4(sfb[:128])
    img[:, 5] = pack4(sfb[128:])
    return img


def run_probe(A, B, img):
    import routing_grouped_expert_gemm_gb300 as rg
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dI = torch.from_numpy(img.view(np.int32)).cuda()
    dD = torch.full((128, 256), float("nan"), dtype=torch.float32, device="cuda")
    rc = rg.lib().moe_testing_mx_tile(dA.data_ptr(), dB.data_ptr(), dI.data_ptr(), dD.data_ptr(),
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    return dD.cpu().numpy().astype(np.float64)


def random_codes(rng, shape):
    c = rng.integers(0, 256, size=shape).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x38  # no NaN codes
    return c


def test_block_scaled_mma_scale_placement():
    rng = np.random.default_rng(5)
    A = random_codes(rng, (128, 128))
    B = random_codes(rng, (256, 128))
    sfa = rng.integers(118, 136, size=(128, 4)).astype(np.uint8)
    sfb = rng.integers(118, 136, size=(256, 4)).astype(np.uint8)
    want = reference(A, B, sfa, sfb)
    got = run_probe(A, B, image_lane_is_row(sfa, sfb))
    assert np.isfinite(got).all()
    np.testing.assert_allclose(got, want, rtol=1e-5, atol=1e-6 * np.abs(want).max())
