"""Pins for the oracle's scale repack (CPU only).

The 128x4-atom layout is stated three ways on the pages; each is restated
here with torch/numpy reshapes and compared with the oracle's closed form:

* submission 69953, ``to_blocked_batch``: per batch,
  view(rest_m, 128, rest_k, 4).permute(0, 2, 1, 3).reshape(-1, 4, 32, 4)
  .transpose(1, 2).reshape(-1, 32, 16);
* submission 69575, ``blocked_transform_kernel``: the perm / chunk / d1 d2 d3
  index arithmetic;
* submission 103289, ``permuted_to_blocked``: the [32, 4, rest_m, 4, rest_k, L]
  tensor permuted by (2, 4, 0, 1, 3) and reshaped to [-1, 32, 16] is the
  blocked order, i.e. a view.
"""
import numpy as np
import pytest
import torch

import oracle


def blocked_per_batch_torch(src):
    """Restatement of submission 69953's to_blocked_batch for one [rows, cols] slice."""
    rows, cols = src.shape
    n_row_blocks, n_col_blocks = (rows + 127) // 128, (cols + 3) // 4
    blocks = src.view(n_row_blocks, 128, n_col_blocks, 4).permute(0, 2, 1, 3)
    return blocks.reshape(-1, 4, 32, 4).transpose(1, 2).reshape(-1, 32, 16).flatten()


def blocked_per_batch_padded_torch(src):
    """to_blocked_batch on a slice first padded with zero rows/columns up to the
    ceil_div sizes it computes (its view needs whole 128x4 atoms)."""
    rows, cols = src.shape
    padded = torch.zeros((rows + 127) // 128 * 128, (cols + 3) // 4 * 4, dtype=src.dtype)
    padded[:rows, :cols] = src
    return blocked_per_batch_torch(padded)


def blocked_index_math_numpy(src_l, rows, cols):
    """Restatement of submission 69575's scatter indices (output sized for padding)."""
    ncb = (cols + 3) // 4
    nrb = (rows + 127) // 128
    offs = np.arange(rows * cols)
    i, j = offs // cols, offs % cols
    rb, ri, cb, ci = i // 128, i % 128, j // 4, j % 4
    perm = rb * ncb * 128 * 4 + cb * 128 * 4 + ri * 4 + ci
    chunk, in_chunk = perm // 512, perm % 512
    d1, rest = in_chunk // 128, in_chunk % 128
    d2, d3 = rest // 4, rest % 4
    out_idx = chunk * 512 + d2 * 16 + d1 * 4 + d3
    out = np.zeros(nrb * ncb * 512, dtype=np.uint8)
    out[out_idx] = src_l.reshape(-1)
    return out


@pytest.mark.parametrize("rows,K,L", [(128, 64, 1), (256, 192, 2), (384, 1024, 3), (128, 2048, 1)])
def test_repack_equals_to_blocked_batch(rows, K, L):
    rng = np.random.default_rng(rows + K + L)
    src = rng.integers(0, 256, (L, rows, K // 16), dtype=np.uint8)
    got = oracle.repack_scales(src, rows, K, L).reshape(L, -1)
    for l in range(L):
        want = blocked_per_batch_torch(torch.from_numpy(src[l].copy())).numpy()
        assert np.array_equal(got[l], want)


@pytest.mark.parametrize("rows,K,L", [(130, 80, 2), (1, 16, 1), (300, 1072, 1), (128, 112, 3)])
def test_repack_equals_padded_to_blocked_batch(rows, K, L):
    rng = np.random.default_rng(rows + 3 * K)
    src = rng.integers(0, 256, (L, rows, K // 16), dtype=np.uint8)
    got = oracle.repack_scales(src, rows, K, L).reshape(L, -1)
    for l in range(L):
        want = blocked_per_batch_padded_torch(torch.from_numpy(src[l].copy())).numpy()
        assert np.array_equal(got[l], want)


@pytest.mark.parametrize("rows,K,L", [(1, 64, 1), (1, 256, 3), (31, 128, 2), (129, 64, 1),
                                      (200, 320, 2), (128, 64, 2), (7, 1024, 1),
                                      # K % 64 != 0: a partly padded last atom column
                                      (1, 16, 2), (33, 48, 1), (130, 80, 2), (5, 1040, 1),
                                      (256, 208, 1)])
def test_repack_equals_index_math_with_zero_padding(rows, K, L):
    rng = np.random.default_rng(rows * 7 + K)
    src = rng.integers(1, 256, (L, rows, K // 16), dtype=np.uint8)  # no zero source bytes
    got = oracle.repack_scales(src, rows, K, L).reshape(L, -1)
    for l in range(L):
        want = blocked_index_math_numpy(src[l], rows, K // 16)
        assert np.array_equal(got[l], want)
    # every source byte appears once; everything else is 0x00 padding
    assert np.count_nonzero(got) == src.size
    assert oracle.permuted_scale_bytes(rows, K, L) == \
        L * ((rows + 127) // 128) * ((K + 63) // 64) * 512


@pytest.mark.parametrize("rows,K,L", [(256, 256, 2), (130, 128, 3)])
def test_permuted_tensor_view_semantics(rows, K, L):
    """[32, 4, rest_m, 4, rest_k, L] indexing, and the permute(2,4,0,1,3) view."""
    rng = np.random.default_rng(3)
    src = rng.integers(0, 256, (L, rows, K // 16), dtype=np.uint8)
    flat = torch.from_numpy(oracle.repack_scales(src, rows, K, L))
    rest_m, rest_k = (rows + 127) // 128, K // 64
    t = flat.as_strided((32, 4, rest_m, 4, rest_k, L),
                        (16, 4, 512 * rest_k, 1, 512, 512 * rest_k * rest_m))
    for l in range(L):
        for m in range(0, rows, 7):
            for kb in range(K // 16):
                assert int(t[m % 32, (m // 32) % 4, m // 128, kb % 4, kb // 4, l]) == src[l, m, kb]
        view = t[:, :, :, :, :, l].permute(2, 4, 0, 1, 3).reshape(-1, 32, 16).flatten()
        assert np.array_equal(view.numpy(), flat.numpy().reshape(L, -1)[l])
