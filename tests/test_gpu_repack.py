"""GPU scale repack: bit-exact against the oracle's closed form, padding included."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import nvfp4_block_scaled_gemv_gb300 as nv  # noqa: E402
import oracle  # noqa: E402
from nvfp4_block_scaled_gemv_gb300 import build as libbuild  # noqa: E402
from nvfp4_block_scaled_gemv_gb300 import synthetic  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    libbuild.build()
    nv.library()


def gpu_repack(src, rows, K, L, src_offset=0):
    """Repack on the GPU; src_offset > 0 places the source that many bytes past a
    256-byte boundary (4 forces the shared-memory kernel, 0 allows the register one)."""
    n = nv.nvfp4_permuted_scale_bytes(rows, K, L)
    pad = 512
    buf = torch.full((n + 2 * pad,), 0xA5, dtype=torch.uint8, device=DEV)
    dst = buf[pad:pad + n]
    flat = torch.from_numpy(np.ascontiguousarray(src).reshape(-1))
    sbuf = torch.empty(flat.numel() + src_offset, dtype=torch.uint8, device=DEV)
    s = sbuf[src_offset:]
    s.copy_(flat)
    nv.nvfp4_repack_scales(s.data_ptr(), dst.data_ptr(), rows, K, L,
                           torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    whole = buf.cpu().numpy()
    assert np.all(whole[:pad] == 0xA5) and np.all(whole[pad + n:] == 0xA5), "write outside dst"
    return whole[pad:pad + n]


@pytest.mark.parametrize("rows,K,L", [
    (1, 64, 1), (1, 16384, 4), (31, 128, 2), (128, 64, 1), (129, 1088, 3), (200, 7168, 2),
    (1000, 2048, 1), (4096, 64, 2), (7168, 2048, 4), (7168, 16384, 1), (333, 4160, 5),
    # K % 256 == 0 with 1, 3, 5 and 13 16-byte columns per plain row (partial column groups)
    (1, 256, 3), (129, 768, 3), (333, 1280, 2), (300, 3328, 3), (4096, 7168, 8),
    # K % 64 != 0: the byte kernel, last atom column padded with 0x00
    (1, 16, 1), (33, 48, 2), (130, 80, 3), (5, 1040, 1), (7168, 2064, 2), (300, 208, 1),
])
@pytest.mark.parametrize("src_offset", [0, 4])
def test_repack_bit_exact(rows, K, L, src_offset):
    rng = np.random.default_rng(rows + K)
    src = rng.integers(0, 256, (L, rows, K // 16), dtype=np.uint8)
    got = gpu_repack(src, rows, K, L, src_offset)
    assert np.array_equal(got, oracle.repack_scales(src, rows, K, L))


def test_repack_full_size_scales():
    # sfa of the largest benchmark workload: 16 batches of 16384 x 512 scale bytes
    M, K, L = 16384, 8192, 16
    src = synthetic.scale_bytes(2, L * M * (K // 16)).reshape(L, M, K // 16)
    assert np.array_equal(gpu_repack(src, M, K, L), oracle.repack_scales(src, M, K, L))


def test_repack_overwrites_stale_padding():
    for rows, K, L, off in [(5, 256, 2, 0), (5, 256, 2, 4), (5, 192, 2, 0), (5, 80, 2, 4),
                            (130, 16, 1, 0)]:
        src = np.full((L, rows, K // 16), 0x38, dtype=np.uint8)
        got = gpu_repack(src, rows, K, L, off)  # dst pre-filled with 0xA5 by gpu_repack
        assert np.array_equal(got, oracle.repack_scales(src, rows, K, L))
        assert np.count_nonzero(got) == src.size
