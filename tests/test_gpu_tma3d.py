"""Pins the 3-D tensor-map view the backward uses to load two 64-wide blocks of
an MN-major operand in one TMA instruction: dimensions (64 columns, row,
64-column block) of a row-major bf16 matrix, the block dimension's stride (128
bytes) below the row stride.  The encoder must accept it, and a {64, 64, 2}
box must land as two 8 KB tiles, block j at j * 8192, row r at r * 128, its
16-byte chunk c at chunk c ^ (r % 8) (128-byte swizzle) -- the layout of two
{64, 64} boxes of the 2-D view side by side."""
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


def expected_tiles(src: np.ndarray, r0: int, b0: int) -> np.ndarray:
    """The 16384 bytes as uint16 words: two swizzled 64 x 64 tiles."""
    out = np.zeros(8192, dtype=np.uint16)
    for j in range(2):
        for r in range(64):
            for c in range(8):
                chunk = src[r0 + r, (b0 + j) * 64 + 8 * c:(b0 + j) * 64 + 8 * c + 8]
                off = (j * 8192 + r * 128 + ((c ^ (r % 8)) * 16)) // 2
                out[off:off + 8] = chunk
    return out


@pytest.mark.parametrize("rows,cols,r0,b0", [(256, 512, 64, 3), (128, 7168, 0, 110), (200, 256, 136, 2)])
def test_tma3d_two_column_blocks(rows, cols, r0, b0):
    import routing_grouped_expert_gemm_gb300 as rg
    rng = np.random.default_rng(rows + cols)
    src = rng.integers(0, 65536, size=(rows, cols), dtype=np.uint32).astype(np.uint16)
    dsrc = torch.from_numpy(src.view(np.int16)).cuda()
    out = torch.zeros(8192, dtype=torch.int16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = rg.testing_lib().moe_testing_tma3d_load(dsrc.data_ptr(), rows, cols, r0, b0, out.data_ptr(),
                                                 status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc != -5, "the tensor-map encoder rejected the 3-D view"
    assert rc == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    got = out.cpu().numpy().view(np.uint16)
    np.testing.assert_array_equal(got, expected_tiles(src, r0, b0))
