"""Pins the block-scaled MXFP8 tcgen05 MMA (instruction descriptor, E8M0
scales in TMEM, scale-factor ids) on one 128 x 256 x 128 tile against a CPU
reference built from torch's float8_e4m3fn decoding and exact powers of two.

The placement the forward kernel relies on: the scales of a 128-row operand
block form a 512-byte block with byte offset (r % 32) * 16 + (r // 32) * 4 + kb
(kb = 32-wide K block inside a 128-wide K step); tcgen05.cp.32x128b.warpx4
puts its 32 x 16-byte rows into TMEM lanes r % 32 of every lane quarter, so row
r's word sits in column base + r // 32 and the kb-th MMA picks byte kb through
its scale-factor id.  A 256-row B operand uses two such blocks (columns
base..base+3 for rows 0-127, base+4..base+7 for rows 128-255)."""
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


def sf_block(sf128):
    """[128 rows, 4 K-blocks] scale codes -> the 512-byte block layout."""
    blk = np.zeros(512, dtype=np.uint8)
    for r in range(128):
        for kb in range(4):
            blk[(r % 32) * 16 + (r // 32) * 4 + kb] = sf128[r, kb]
    return blk


def tmem_image(sfa, sfb):
    """What tcgen05.cp.32x128b.warpx4 of the three blocks leaves in TMEM
    columns 256..267 (mode 0 writes this image directly)."""
    img = np.zeros((128, 12), dtype=np.uint32)
    for col0, sf in ((0, sfa), (4, sfb[:128]), (8, sfb[128:])):
        words = sf_block(sf).view(np.uint32).reshape(32, 4)  # lane l: 4 words
        for q in range(4):
            img[32 * q:32 * q + 32, col0:col0 + 4] = words
    return img


def run_probe(A, B, img, mode=0):
    import routing_grouped_expert_gemm_gb300 as rg
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dI = torch.from_numpy(np.ascontiguousarray(img).view(np.uint8)).cuda()
    dD = torch.full((128, 256), float("nan"), dtype=torch.float32, device="cuda")
    rc = rg.testing_lib().moe_testing_mx_tile(dA.data_ptr(), dB.data_ptr(), dI.data_ptr(), dD.data_ptr(), mode,
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    return dD.cpu().numpy().astype(np.float64)


def random_codes(rng, shape):
    c = rng.integers(0, 256, size=shape).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x38  # no NaN codes
    return c


@pytest.mark.parametrize("mode", [0, 1])
def test_block_scaled_mma_scale_placement(mode):
    rng = np.random.default_rng(5 + mode)
    A = random_codes(rng, (128, 128))
    B = random_codes(rng, (256, 128))
    sfa = rng.integers(118, 136, size=(128, 4)).astype(np.uint8)
    sfb = rng.integers(118, 136, size=(256, 4)).astype(np.uint8)
    want = reference(A, B, sfa, sfb)
    if mode == 0:
        got = run_probe(A, B, tmem_image(sfa, sfb), 0)
    else:
        blocks = np.concatenate([sf_block(sfa), sf_block(sfb[:128]), sf_block(sfb[128:])])
        got = run_probe(A, B, blocks, 1)
    assert np.isfinite(got).all()
    np.testing.assert_allclose(got, want, rtol=1e-5, atol=1e-6 * np.abs(want).max())
