"""C ABI on the host (CPU only, no kernel launches).

The library loads and exports every function the header declares; argument
validation rejects bad calls before touching the GPU; the launch planner
and the kernel's row partition are checked as host arithmetic.
"""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import nvfp4_block_scaled_gemv_gb300 as nv
from nvfp4_block_scaled_gemv_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4_gemv.h")


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return nv.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4_[a-z_0-9]+)\s*\(", text)))


def test_header_declarations_match_binding_and_exports(lib):
    declared = declared_functions()
    assert declared == sorted(nv.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", nv.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(nvfp4_\w+)", out))
    assert set(declared) <= exported


def test_wait_selftest_rejects_null_outputs_before_any_launch(lib):
    import ctypes
    i = ctypes.c_int(0)
    w = ctypes.c_int64(0)
    r = ctypes.byref
    assert lib.nvfp4_selftest_bounded_wait(None, r(i), r(i), r(w), None) == nv.ERR_INVALID_VALUE
    assert lib.nvfp4_selftest_bounded_wait(r(i), None, r(i), r(w), None) == nv.ERR_INVALID_VALUE
    assert lib.nvfp4_selftest_bounded_wait(r(i), r(i), None, r(w), None) == nv.ERR_INVALID_VALUE
    assert lib.nvfp4_selftest_bounded_wait(r(i), r(i), r(i), None, None) == nv.ERR_INVALID_VALUE


def test_header_compiles_as_c(tmp_path):
    src = tmp_path / "t.c"
    src.write_text('#include "nvfp4_gemv.h"\nint main(void){return (int)NVFP4_OK;}\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER), "-c",
                    str(src), "-o", str(tmp_path / "t.o")], check=True)


def _call(lib, a=64, b=64, sfa=64, sfb=64, c=64, M=8, K=64, L=1, layout=0):
    return lib.nvfp4_gemv(a, b, sfa, sfb, c, M, K, L, layout, None)


def test_validation_before_any_cuda_call(lib):
    # the pointers below are never dereferenced: every case fails validation
    assert _call(lib, M=-1) == nv.ERR_INVALID_VALUE
    assert _call(lib, K=-64) == nv.ERR_INVALID_VALUE
    assert _call(lib, L=-2) == nv.ERR_INVALID_VALUE
    assert _call(lib, layout=2) == nv.ERR_INVALID_VALUE
    assert _call(lib, K=88) == nv.ERR_UNSUPPORTED_SHAPE  # whole 16-element blocks only
    assert _call(lib, K=(1 << 30) + 64) == nv.ERR_UNSUPPORTED_SHAPE
    assert _call(lib, M=1 << 31) == nv.ERR_UNSUPPORTED_SHAPE
    assert _call(lib, M=1 << 30, L=1 << 11) == nv.ERR_UNSUPPORTED_SHAPE
    assert _call(lib, a=None) == nv.ERR_INVALID_VALUE
    assert _call(lib, c=None) == nv.ERR_INVALID_VALUE
    assert _call(lib, sfb=None) == nv.ERR_INVALID_VALUE
    # a and b: 16 bytes (the pages' assumed_align=16); scales: 32; c: 2
    assert _call(lib, a=64 + 8) == nv.ERR_MISALIGNED
    assert _call(lib, b=64 + 8) == nv.ERR_MISALIGNED
    assert _call(lib, sfa=64 + 16) == nv.ERR_MISALIGNED
    assert _call(lib, sfb=64 + 1) == nv.ERR_MISALIGNED
    assert _call(lib, c=64 + 1) == nv.ERR_MISALIGNED


def test_empty_problems_are_noops(lib):
    assert _call(lib, a=None, b=None, sfa=None, sfb=None, c=None, M=0) == nv.OK
    assert _call(lib, a=None, b=None, sfa=None, sfb=None, c=None, L=0) == nv.OK
    assert lib.nvfp4_repack_scales(None, None, 0, 64, 1, None) == nv.OK
    assert lib.nvfp4_repack_scales(None, None, 5, 0, 1, None) == nv.OK


def test_explicit_schedule_validation(lib):
    args = (64, 64, 64, 64, 64, 8, 64, 1, 0)
    for kernel in (nv.KERNEL_DIRECT, nv.KERNEL_PIPELINED):
        assert lib.nvfp4_gemv_explicit(*args, kernel, 12, 1, 1, None) == nv.ERR_INVALID_VALUE
        assert lib.nvfp4_gemv_explicit(*args, kernel, 32, 3, 1, None) == nv.ERR_INVALID_VALUE
        assert lib.nvfp4_gemv_explicit(*args, kernel, 32, 1, 0, None) == nv.ERR_INVALID_VALUE
        assert lib.nvfp4_gemv_explicit(*args, kernel, 32, 1, 1 << 31, None) == nv.ERR_INVALID_VALUE
    assert lib.nvfp4_gemv_explicit(*args, 7, 32, 1, 1, None) == nv.ERR_INVALID_VALUE
    # the pipelined kernel needs K > 0 and a K step for every K-split warp (K=64: one step)
    assert lib.nvfp4_gemv_explicit(*args, nv.KERNEL_PIPELINED, 32, 2, 1, None) == nv.ERR_INVALID_VALUE
    zero_k = (64, 64, 64, 64, 64, 8, 0, 1, 0)
    assert lib.nvfp4_gemv_explicit(*zero_k, nv.KERNEL_PIPELINED, 32, 1, 1, None) == nv.ERR_INVALID_VALUE


def test_k_not_multiple_of_64(lib):
    """K % 16 == 0 with K % 64 != 0: the blockwise kernel's shapes."""
    args = (64, 64, 64, 64, 64, 8, 80, 1, 0)
    for kernel, lpr in ((nv.KERNEL_DIRECT, 32), (nv.KERNEL_PIPELINED, 32), (nv.KERNEL_TENSOR, 4),
                        (nv.KERNEL_BLOCKDOT, 0)):
        for layout in (nv.SF_PLAIN, nv.SF_PERMUTED_128x4):
            assert lib.nvfp4_gemv_explicit(*args[:-1], layout, kernel, lpr, 1, 1, None) == \
                nv.ERR_UNSUPPORTED_SHAPE
    B = nv.KERNEL_BLOCKWISE
    assert lib.nvfp4_gemv_explicit(*args, B, 16, 1, 1, None) == nv.ERR_INVALID_VALUE
    assert lib.nvfp4_gemv_explicit(*args, B, 32, 2, 1, None) == nv.ERR_INVALID_VALUE
    assert lib.nvfp4_gemv_explicit(*args, B, 32, 1, 0, None) == nv.ERR_INVALID_VALUE
    assert lib.nvfp4_gemv_explicit(*(args[:5] + (0,) + args[6:]), B, 32, 1, 1, None) == nv.OK
    assert lib.nvfp4_gemv_explicit(*(args[:3] + (64 + 16,) + args[4:]), B, 32, 1, 1, None) == \
        nv.ERR_MISALIGNED
    for layout in (nv.SF_PLAIN, nv.SF_PERMUTED_128x4):
        for K in (16, 48, 80, 1040):
            plan = nv.nvfp4_gemv_plan(4096, K, 8, layout, 152, 2)
            assert plan["kernel"] == B
            assert (plan["lanes_per_row"], plan["k_split"], plan["threads_per_cta"]) == (32, 1, 256)
            assert plan["rows_per_pass"] == 32 and plan["steps"] == (K // 16 + 31) // 32
            # one warp per 4-row group, at most 2 CTAs per SM
            assert plan["ctas"] == min(152 * 2, 8 * 1024 // 8)
        with pytest.raises(nv.Nvfp4Error):
            nv.nvfp4_gemv_plan(4096, 80, 8, layout, 152, 2, kernel=nv.KERNEL_PIPELINED)
    # small problems: one warp per group
    assert nv.nvfp4_gemv_plan(5, 48, 1, 0, 152, 2)["ctas"] == 1
    assert nv.nvfp4_gemv_plan(100, 48, 3, 0, 152, 2)["ctas"] == (3 * 25 + 7) // 8
    # K % 64 == 0 keeps its schedule; the blockwise kernel is there on request
    assert nv.nvfp4_gemv_plan(4096, 1024, 8, 0, 152, 2)["kernel"] == nv.KERNEL_PIPELINED
    assert nv.nvfp4_gemv_plan(4096, 1024, 8, 0, 152, 2, kernel=B)["kernel"] == B


def test_tensor_kernel_schedule_validation(lib):
    # (a, b, sfa, sfb, c, M, K, L, layout): checked before any CUDA call
    perm = (64, 64, 64, 64, 64, 300, 1024, 2, nv.SF_PERMUTED_128x4)
    plain = perm[:-1] + (nv.SF_PLAIN,)
    T = nv.KERNEL_TENSOR
    # plain scales need whole 256-element stages of 16-byte scale rows
    plain320 = plain[:6] + (320,) + plain[7:]
    assert lib.nvfp4_gemv_explicit(*plain320, T, 4, 1, 1, None) == nv.ERR_UNSUPPORTED_SHAPE
    assert lib.nvfp4_gemv_explicit(*plain, T, 4, 8, 8, None) == nv.ERR_INVALID_VALUE
    plain_zero_k = plain[:6] + (0,) + plain[7:]
    assert lib.nvfp4_gemv_explicit(*plain_zero_k, T, 4, 1, 1, None) == nv.ERR_INVALID_VALUE
    # every CTA of a cluster needs a 256-element K stage: K = 1024 has 4
    assert lib.nvfp4_gemv_explicit(*perm, T, 4, 8, 8, None) == nv.ERR_INVALID_VALUE
    # whole clusters only
    assert lib.nvfp4_gemv_explicit(*perm, T, 4, 2, 3, None) == nv.ERR_INVALID_VALUE
    assert lib.nvfp4_gemv_explicit(*perm, T, 4, 3, 3, None) == nv.ERR_INVALID_VALUE
    zero_k = perm[:6] + (0,) + perm[7:]
    assert lib.nvfp4_gemv_explicit(*zero_k, T, 4, 1, 1, None) == nv.ERR_INVALID_VALUE
    # empty problems are no-ops
    assert lib.nvfp4_gemv_explicit(*(perm[:5] + (0,) + perm[6:]), T, 4, 1, 1, None) == nv.OK


def test_repack_validation(lib):
    assert lib.nvfp4_repack_scales(64, 64, -1, 64, 1, None) == nv.ERR_INVALID_VALUE
    assert lib.nvfp4_repack_scales(64, 64, 4, 72, 1, None) == nv.ERR_UNSUPPORTED_SHAPE
    assert lib.nvfp4_repack_scales(None, 64, 4, 64, 1, None) == nv.ERR_INVALID_VALUE
    assert lib.nvfp4_repack_scales(66, 64, 4, 64, 1, None) == nv.ERR_MISALIGNED
    assert lib.nvfp4_repack_scales(64, 72, 4, 64, 1, None) == nv.ERR_MISALIGNED


def test_permuted_scale_bytes_and_status_strings(lib):
    assert nv.nvfp4_permuted_scale_bytes(7168, 2048, 4) == 4 * 56 * 32 * 512
    assert nv.nvfp4_permuted_scale_bytes(1, 16384, 1) == 256 * 512
    assert nv.nvfp4_permuted_scale_bytes(129, 64, 2) == 2 * 2 * 1 * 512
    # K % 64 != 0: a last, partly padded atom column
    assert nv.nvfp4_permuted_scale_bytes(5, 80, 1) == 2 * 512
    assert nv.nvfp4_permuted_scale_bytes(130, 16, 3) == 3 * 2 * 1 * 512
    assert nv.nvfp4_permuted_scale_bytes(5, 72, 1) == 0
    assert nv.status_string(nv.OK) == "NVFP4_OK"
    assert nv.status_string(nv.ERR_MISALIGNED) == "NVFP4_ERR_MISALIGNED"
    assert nv.status_string(99) == "NVFP4_ERR_UNKNOWN"
    assert nv.nvfp4_last_cuda_error() == 0


BENCH_SHAPES = [(128, 256, 1), (7168, 2048, 4), (4096, 7168, 8), (7168, 16384, 1),
                (16384, 8192, 16)]


@pytest.mark.parametrize("shape,layout,kernel,want", [
    (BENCH_SHAPES[0], 0, -1, (0, 4, 1, 2, 8)),  # tiny: direct kernel, one CTA per 8 KB of A
    (BENCH_SHAPES[1], 0, -1, (1, 16, 1, 304, 16)),
    (BENCH_SHAPES[2], 0, -1, (1, 16, 1, 304, 16)),
    (BENCH_SHAPES[3], 0, -1, (1, 32, 4, 304, 16)),
    # >= 512 MB of A with K <= 8192 (plain scales: K % 256 == 0): the
    # tensor-core kernel, 4 stages, clusters of 2 (32 K stages), on every
    # resident 4-stage CTA
    (BENCH_SHAPES[4], 0, -1, (2, 4, 2, 304, 128)),
    (BENCH_SHAPES[0], 1, -1, (1, 4, 1, 64, 32)),  # permuted: the general schedule
    (BENCH_SHAPES[1], 1, -1, (1, 4, 4, 304, 64)),
    # 256 tiles fill 84% of one wave of 4-stage tensor-core CTAs, K >= 6144:
    # the tensor-core kernel, one 4-stage CTA per tile, no K split
    (BENCH_SHAPES[2], 1, -1, (2, 4, 1, 256, 128)),
    (BENCH_SHAPES[3], 1, -1, (1, 16, 8, 304, 32)),
    (BENCH_SHAPES[4], 1, -1, (2, 4, 2, 304, 128)),
    (BENCH_SHAPES[4], 1, 1, (1, 4, 8, 304, 64)),
    (BENCH_SHAPES[1], 0, 3, (3, 5, 1, 152, 128)),  # block-dot: one CTA per SM, 5 ring slots
    (BENCH_SHAPES[3], 1, 3, (3, 11, 1, 152, 128)),
    (BENCH_SHAPES[0], 0, 0, (0, 4, 1, 64, 8)),
    (BENCH_SHAPES[1], 0, 0, (0, 32, 1, 304, 8)),
    (BENCH_SHAPES[2], 0, 0, (0, 16, 1, 304, 8)),
    (BENCH_SHAPES[3], 0, 0, (0, 32, 4, 304, 8)),
    (BENCH_SHAPES[4], 0, 0, (0, 32, 1, 304, 8)),
])
def test_plan_for_the_benchmark_shapes(lib, shape, layout, kernel, want):
    M, K, L = shape
    plan = nv.nvfp4_gemv_plan(M, K, L, layout, num_sms=152, ctas_per_sm=2, kernel=kernel)
    got = tuple(plan[k] for k in ("kernel", "lanes_per_row", "k_split", "ctas", "rows_per_pass"))
    assert got == want
    if plan["kernel"] == nv.KERNEL_TENSOR:  # lanes_per_row = stages; steps = 256-element K stages
        assert plan["steps"] == -(-K // 256) and plan["threads_per_cta"] == 224
    elif plan["kernel"] == nv.KERNEL_BLOCKDOT:  # lanes_per_row = ring slots; 512-element stages
        assert plan["steps"] == -(-K // 512) and plan["threads_per_cta"] == 192
    else:
        assert plan["steps"] == -(-(K // 64) // plan["lanes_per_row"])


def test_tensor_kernel_plans(lib):
    """The tensor-core kernel: plain scales need K % 256 == 0; its schedule
    follows the measured rule: tiles that fit one wave of 4-stage
    CTAs (2 per SM) get 4 stages and the largest cluster that still fits, one
    CTA per tile and rank; tiles that fit one wave of 2-stage CTAs (4 per SM)
    4 stages on every resident 4-stage CTA, clusters of 2 only when that
    leaves each rank fewer K stages over the waves of tiles; larger problems 4
    stages on every resident 4-stage CTA, clusters of 2 from 32 K stages."""
    with pytest.raises(nv.Nvfp4Error):
        nv.nvfp4_gemv_plan(4096, 7232, 8, 0, 152, 2, kernel=nv.KERNEL_TENSOR)
    assert nv.nvfp4_gemv_plan(4096, 7168, 8, 0, 152, 2, kernel=nv.KERNEL_TENSOR) == \
        nv.nvfp4_gemv_plan(4096, 7168, 8, 1, 152, 2, kernel=nv.KERNEL_TENSOR)
    # nvfp4_gemv takes it (M >= 1024) from 512 MB of A with K <= 8192 (plain
    # scales: K % 256 == 0), and for pre-permuted scales when the tiles fill
    # 80-100% of one wave of 4-stage CTAs (2 per SM) with K >= 6144, or more
    # than one wave from 128 MB of A with any K (measured faster there)
    T, P = nv.KERNEL_TENSOR, nv.KERNEL_PIPELINED
    for shape, perm, plain in (((16384, 8192, 16), T, T), ((28672, 8192, 8), T, T),
                               ((16384, 8192, 8), T, T), ((16383, 8192, 8), T, P),
                               ((16384, 16384, 8), T, P), ((16384, 8192, 2), T, P),
                               ((512, 8192, 512), P, P), ((4096, 7168, 8), T, P),
                               ((31232, 8192, 1), T, P), ((4864, 7680, 8), T, P),
                               ((28672, 8192, 1), P, P), ((4096, 4096, 8), P, P),
                               ((4096, 16384, 8), T, P), ((39040, 8192, 1), T, P),
                               ((7168, 65536, 1), P, P), ((32768, 1024, 6), P, P),
                               ((16384, 1024, 16), T, P), ((16384, 1024, 15), P, P),
                               ((65536, 1024, 16), T, T), ((65536, 1088, 16), T, P),
                               ((1, 1024, 1 << 31), P, P), ((1, 1024, (1 << 31) - 1), P, P)):
        assert nv.nvfp4_gemv_plan(*shape, 1, 152, 2)["kernel"] == perm, shape
        assert nv.nvfp4_gemv_plan(*shape, 0, 152, 2)["kernel"] == plain, shape
    rng = np.random.default_rng(1)
    for _ in range(200):
        M, K, L = int(rng.integers(1, 30000)), 64 * int(rng.integers(1, 400)), int(rng.integers(1, 9))
        sms = int(rng.integers(1, 200))
        plan = nv.nvfp4_gemv_plan(M, K, L, 1, sms, 2, kernel=nv.KERNEL_TENSOR)
        tiles, kst = L * -(-M // 128), -(-K // 256)
        ks = plan["k_split"]
        assert ks in (1, 2, 4, 8) and (ks == 1 or ks <= kst)
        assert plan["ctas"] % ks == 0 and plan["ctas"] // ks <= tiles
        if tiles <= 2 * sms:  # one wave of 4-stage CTAs
            assert plan["lanes_per_row"] == 4 and plan["ctas"] == tiles * ks
            assert plan["ctas"] <= 2 * sms and (ks == 1 or 2 * ks <= kst)
            assert ks == 8 or 2 * tiles * ks > 2 * sms or 4 * ks > kst
        elif tiles <= 4 * sms:  # one wave of 2-stage CTAs, not of 4-stage ones
            slots4, pairs = 2 * sms, sms
            w1 = -(-tiles // slots4) * kst
            w2 = -(-tiles // pairs) * -(-kst // 2)
            assert plan["lanes_per_row"] == 4 and ks == (2 if kst >= 2 and w2 < w1 else 1)
            assert plan["ctas"] == min(tiles, slots4 // ks) * ks
        else:  # 4 stages on every resident 4-stage CTA, clusters of 2 from 32 K stages
            assert plan["lanes_per_row"] == 4 and ks == (2 if kst >= 32 else 1)
            assert plan["ctas"] == max(1, 2 * sms // ks) * ks


def test_block_dot_plans_and_validation(lib):
    """The block-dot kernel, selected explicitly: one CTA per SM (no more than
    the 8-row units), the deepest ring that fits; plain scales need K % 256 == 0."""
    for M, K, L, layout in ((7168, 2048, 4, 0), (7168, 16384, 1, 1), (1, 64, 1, 1), (9, 512, 3, 0),
                            (100000, 64, 1, 1)):
        plan = nv.nvfp4_gemv_plan(M, K, L, layout, 152, 2, kernel=nv.KERNEL_BLOCKDOT)
        units = L * -(-M // 8)
        cb = 2 if K % 256 == 0 else 1
        assert plan["kernel"] == nv.KERNEL_BLOCKDOT and plan["k_split"] == 1
        assert plan["ctas"] == min(152, units) and 2 <= plan["lanes_per_row"] <= 32
        assert plan["steps"] == -(-(K // 64) // (4 * cb)) and plan["threads_per_cta"] == 192
    with pytest.raises(nv.Nvfp4Error):  # plain scales, K % 256 != 0
        nv.nvfp4_gemv_plan(128, 320, 1, 0, 152, 2, kernel=nv.KERNEL_BLOCKDOT)
    args = (64, 64, 64, 64, 64, 300, 1024, 2, nv.SF_PLAIN)
    B = nv.KERNEL_BLOCKDOT
    assert lib.nvfp4_gemv_explicit(*args, B, 4, 2, 8, None) == nv.ERR_INVALID_VALUE   # k_split
    assert lib.nvfp4_gemv_explicit(*args, B, 1, 1, 8, None) == nv.ERR_INVALID_VALUE   # 1 slot
    assert lib.nvfp4_gemv_explicit(*args, B, 33, 1, 8, None) == nv.ERR_INVALID_VALUE  # > 32 slots
    assert lib.nvfp4_gemv_explicit(*args, B, 4, 1, 0, None) == nv.ERR_INVALID_VALUE   # no CTA
    plain320 = args[:6] + (320,) + args[7:]
    assert lib.nvfp4_gemv_explicit(*plain320, B, 4, 1, 8, None) == nv.ERR_UNSUPPORTED_SHAPE
    empty = args[:5] + (0,) + args[6:]
    assert lib.nvfp4_gemv_explicit(*empty, B, 4, 1, 8, None) == nv.OK


def max_rows_per_row_lane(M, L, perm, lpr, ks, ctas):
    """Longest row-lane range of the pipelined kernel's partition."""
    nr = 4 * (32 // lpr)
    unit = nr if perm else 1
    rows_per_l = -(-M // 128) * 128 if perm else M
    t = rows_per_l * L // unit
    per_cta = -(-t // ctas)
    return -(-per_cta // (8 // ks)) * unit


def test_pipelined_rows_per_pass_cover_the_longest_range(lib):
    """rows_per_pass = groups * 4 * (32 / lanes_per_row), with the fewest of
    1, 2 or 4 groups that hold the longest row-lane range, or 2 when it needs
    more than 4."""
    rng = np.random.default_rng(1)
    for _ in range(300):
        M, L = int(rng.integers(1, 30000)), int(rng.integers(1, 17))
        K = 64 * int(rng.integers(1, 300))
        layout = int(rng.integers(0, 2))
        plan = nv.nvfp4_gemv_plan(M, K, L, layout, 152, 2, kernel=nv.KERNEL_PIPELINED)
        nr = 4 * (32 // plan["lanes_per_row"])
        rows = max_rows_per_row_lane(M, L, layout == 1, plan["lanes_per_row"], plan["k_split"],
                                     plan["ctas"])
        need = -(-rows // nr)
        groups = 1 if need <= 1 else 2 if need <= 2 else 4 if need <= 4 else 2
        assert plan["rows_per_pass"] == groups * nr


def test_permuted_plans_avoid_half_sector_scale_reads(lib):
    rng = np.random.default_rng(2)
    for _ in range(200):
        M, L = int(rng.integers(1, 30000)), int(rng.integers(1, 17))
        K = 64 * int(rng.integers(1, 300))
        assert nv.nvfp4_gemv_plan(M, K, L, nv.SF_PERMUTED_128x4, 152, 2,
                                  kernel=nv.KERNEL_PIPELINED)["lanes_per_row"] != 32


def test_permuted_plans_with_plenty_of_rows_use_narrow_rows(lib):
    """Permuted scales, at least 24 rows per row lane and an even K split to at
    most 4 steps per warp: 4 lanes per row."""
    assert nv.nvfp4_gemv_plan(7168, 2048, 4, nv.SF_PERMUTED_128x4, 152, 2)["lanes_per_row"] == 4
    assert nv.nvfp4_gemv_plan(28672, 4096, 1, nv.SF_PERMUTED_128x4, 152, 2)["k_split"] == 8
    # scarce rows: the cost model decides
    assert nv.nvfp4_gemv_plan(2048, 4096, 1, nv.SF_PERMUTED_128x4, 152, 2)["lanes_per_row"] != 4
    # uneven K split (28 steps over 8 warps): the cost model decides
    plan = nv.nvfp4_gemv_plan(4096, 7168, 8, nv.SF_PERMUTED_128x4, 152, 2, kernel=nv.KERNEL_PIPELINED)
    assert plan["lanes_per_row"] != 4


def test_gemv_ex_option_validation(lib):
    """Option errors come back before any launch (no GPU needed)."""
    base = dict(a=64, b=64, sfa=64, sfb=64, c=64, M=8, K=2048, L=2)

    def status(layout=nv.SF_PLAIN, **kw):
        try:
            nv.nvfp4_gemv_ex(*base.values(), layout, **kw)
        except nv.Nvfp4Error as e:
            return e.status
        return nv.OK

    assert status(b_batch_stride=-32) == nv.ERR_INVALID_VALUE
    assert status(b_batch_stride=512) == nv.ERR_INVALID_VALUE           # below K/2
    assert status(b_batch_stride=1024 + 8) == nv.ERR_MISALIGNED          # not a multiple of 16
    assert status(sfb_batch_stride=64) == nv.ERR_INVALID_VALUE          # below K/16
    assert status(sfb_batch_stride=130) == nv.ERR_MISALIGNED
    assert status(nv.SF_PERMUTED_128x4, sfb_batch_stride=512) == nv.ERR_INVALID_VALUE  # below 32*512
    assert status(nv.SF_PERMUTED_128x4, sfb_batch_stride=32 * 512 + 4) == nv.ERR_MISALIGNED
    assert status(bias=3) == nv.ERR_MISALIGNED
    # valid options on an empty problem: nothing to do
    nv.nvfp4_gemv_ex(0, 0, 0, 0, 0, 0, 2048, 2, 0, alpha=2.0, b_batch_stride=4096,
                     sfb_batch_stride=256)


def test_kernel_choice(lib):
    assert nv.nvfp4_gemv_plan(100, 0, 3, 0, 152, 2)["kernel"] == nv.KERNEL_DIRECT
    # up to 512 KB of A the direct kernel; above it the pipelined kernel
    assert nv.nvfp4_gemv_plan(100, 64, 3, 0, 152, 2)["kernel"] == nv.KERNEL_DIRECT
    assert nv.nvfp4_gemv_plan(1024, 1024, 1, 0, 152, 2)["kernel"] == nv.KERNEL_DIRECT
    assert nv.nvfp4_gemv_plan(1025, 1024, 1, 0, 152, 2)["kernel"] == nv.KERNEL_PIPELINED
    with pytest.raises(nv.Nvfp4Error) as e:
        nv.nvfp4_gemv_plan(100, 0, 3, 0, 152, 2, kernel=nv.KERNEL_PIPELINED)
    assert e.value.status == nv.ERR_UNSUPPORTED_SHAPE
    with pytest.raises(nv.Nvfp4Error):
        nv.nvfp4_gemv_plan(100, 64, 3, 0, 152, 2, kernel=5)


def test_plan_invariants_on_random_shapes(lib):
    rng = np.random.default_rng(0)
    for _ in range(300):
        M = int(rng.integers(1, 20000))
        K = 64 * int(rng.integers(0, 300))
        L = int(rng.integers(1, 20))
        sms = int(rng.integers(1, 200))
        plan = nv.nvfp4_gemv_plan(M, K, L, 0, sms, 2)
        kch = K // 64
        tiny = M * L * (K // 2) <= 512 << 10
        tensor = M >= 1024 and 0 < K <= 8192 and K % 256 == 0 and M * L * (K // 2) >= 512 << 20
        if tensor:  # large plain streams: the tensor-core kernel (checked elsewhere)
            assert plan["kernel"] == nv.KERNEL_TENSOR
            continue
        assert plan["kernel"] == (nv.KERNEL_PIPELINED if kch and not tiny else nv.KERNEL_DIRECT)
        if kch and tiny:  # narrow rows, at most 4 K steps split over warps, 8 KB of A per CTA
            assert plan["steps"] <= 4 or plan["lanes_per_row"] == 32
            assert plan["ctas"] <= max(1, M * L * (K // 2) // 8192)
        if kch and not tiny and M * L * (K // 2) <= 2 << 20:
            assert plan["ctas"] <= 64
        assert plan["lanes_per_row"] in (4, 8, 16, 32) and plan["k_split"] in (1, 2, 4, 8)
        assert plan["steps"] * plan["lanes_per_row"] >= kch
        assert (plan["steps"] - 1) * plan["lanes_per_row"] < max(kch, 1)
        assert 1 <= plan["ctas"] <= 2 * sms
        assert plan["k_split"] == 1 or plan["k_split"] <= plan["steps"]


# --- a model of the kernel's row partition (same integer arithmetic) ---------

def visited_row(rp, perm):
    if not perm:
        return rp
    q = rp & 127
    j, t = q >> 3, q & 7
    return (rp & ~127) + 32 * (t >> 1) + 2 * j + (t & 1)


def cta_units(T, ctas, cta):
    """Units [c0, c1) of one CTA: floor(T*b/ctas), as q*b + floor(r*b/ctas)."""
    q, r = divmod(T, ctas)
    first = lambda b: q * b + (r * b) // ctas
    assert first(cta) == T * cta // ctas
    return first(cta), first(cta + 1)


def partition(M, L, ctas, ks, perm, nr=8):
    """Rows each (cta, row lane, pass of nr rows) handles, as (l, m) pairs."""
    rows_per_l = ((M + 127) // 128) * 128 if perm else M
    T = rows_per_l * L
    wr_count = 8 // ks
    seen = []
    for cta in range(ctas):
        c0, c1 = cta_units(T, ctas, cta)
        for wr in range(wr_count):
            r, r_end = c0 + (c1 - c0) * wr // wr_count, c0 + (c1 - c0) * (wr + 1) // wr_count
            while r < r_end:
                l = r // rows_per_l
                pass_end = min(r_end, r + nr, (l + 1) * rows_per_l)
                for rho in range(pass_end - r):
                    m = visited_row(r + rho - l * rows_per_l, perm)
                    if m < M:
                        seen.append((l, m))
                r = pass_end
    return seen


@pytest.mark.parametrize("nr", [4, 8, 16, 32])
@pytest.mark.parametrize("perm", [False, True])
@pytest.mark.parametrize("M,L,ctas,ks", [(1, 1, 1, 1), (7, 3, 2, 2), (128, 1, 16, 1),
                                         (200, 3, 37, 4), (129, 2, 304, 8), (1000, 5, 13, 1)])
def test_row_partition_covers_every_row_once(M, L, ctas, ks, perm, nr):
    seen = partition(M, L, ctas, ks, perm, nr)
    assert sorted(seen) == [(l, m) for l in range(L) for m in range(M)]


def test_permuted_visit_order_groups_scale_sectors():
    for blk in range(3):
        order = [visited_row(blk * 128 + q, True) for q in range(128)]
        assert sorted(order) == list(range(blk * 128, blk * 128 + 128))
        for g in range(16):
            rows = order[8 * g: 8 * g + 8]
            # offsets of the rows' scale words in the 512-byte atom share one 32-byte sector
            offs = {((m % 32) * 16 + ((m // 32) % 4) * 4) // 32 for m in rows}
            assert len(offs) == 1


def async_row(rp, perm, ri):
    """Row order of the pipelined kernel (model of its integer arithmetic)."""
    if not perm:
        return rp
    nr = 4 * ri
    q = rp & 127
    chunk, t = q // nr, q % nr
    return (rp & ~127) + 32 * (t // ri) + chunk * ri + (t % ri)


@pytest.mark.parametrize("ri", [1, 2, 4, 8])
def test_pipelined_permuted_order_shares_scale_runs(ri):
    nr = 4 * ri
    for blk in range(2):
        order = [async_row(blk * 128 + q, True, ri) for q in range(128)]
        assert sorted(order) == list(range(blk * 128, blk * 128 + 128))
        for c in range(128 // nr):
            for sub in range(ri):
                rows = [order[c * nr + g * ri + sub] for g in range(4)]  # a lane's 4 items
                offs = [(m % 32) * 16 + ((m // 32) % 4) * 4 for m in rows]
                assert offs == [offs[0] + 4 * g for g in range(4)] and offs[0] % 16 == 0


@pytest.mark.parametrize("groups", [1, 2, 4])
@pytest.mark.parametrize("perm", [False, True])
@pytest.mark.parametrize("M,L,ctas,ks,ri", [(1, 1, 1, 1, 1), (129, 2, 37, 2, 2), (7168, 4, 304, 1, 1),
                                            (1000, 3, 13, 4, 8), (200, 1, 600, 8, 4),
                                            (333, 5, 7, 1, 2)])
def test_pipelined_tasks_cover_every_row_once(M, L, ctas, ks, ri, perm, groups):
    """Model of the pipelined kernel's work split: row-lane ranges, passes of
    up to groups*nr rows inside one batch, and in each group the items
    i*ri + sub of every lane group sub."""
    nr = 4 * ri
    unit = nr if perm else 1
    rows_per_l = ((M + 127) // 128) * 128 if perm else M
    T = rows_per_l * L // unit
    wr_count = 8 // ks
    seen = []
    for cta in range(ctas):
        c0, c1 = cta_units(T, ctas, cta)
        for wr in range(wr_count):
            r = (c0 + (c1 - c0) * wr // wr_count) * unit
            r_end = (c0 + (c1 - c0) * (wr + 1) // wr_count) * unit
            while r < r_end:
                l = r // rows_per_l
                cnt = min(r_end, r + groups * nr, (l + 1) * rows_per_l) - r
                if perm:
                    assert cnt % nr == 0  # aligned chunks: whole groups only
                ng = -(-cnt // nr)
                for g in range(ng):
                    for sub in range(ri):
                        m0 = async_row(r - l * rows_per_l + g * nr + sub, perm, ri)
                        for i in range(4):
                            if g * nr + i * ri + sub >= cnt:
                                continue
                            m = m0 + (32 * i if perm else i * ri)
                            if m < M:
                                seen.append((l, m))
                r += cnt
    assert sorted(seen) == [(l, m) for l in range(L) for m in range(M)]


def test_gemm_small_n_validation(lib):
    G = lib.nvfp4_gemm_small_n
    E = lib.nvfp4_gemm_small_n_explicit
    ptrs = (64, 64, 64, 64, 64)
    # (M, N, K, L): checked before any CUDA call
    assert G(*ptrs, 300, 17, 1024, 2, None, None) == nv.ERR_UNSUPPORTED_SHAPE
    assert G(*ptrs, 300, -1, 1024, 2, None, None) == nv.ERR_INVALID_VALUE
    assert G(*ptrs, 300, 4, 1000, 2, None, None) == nv.ERR_UNSUPPORTED_SHAPE
    assert G(*ptrs, 0, 4, 1024, 2, None, None) == nv.OK
    assert G(*ptrs, 300, 0, 1024, 2, None, None) == nv.OK
    assert G(*ptrs, 300, 4, 1024, 0, None, None) == nv.OK
    assert G(None, 64, 64, 64, 64, 300, 4, 1024, 2, None, None) == nv.ERR_INVALID_VALUE
    assert G(64, 64, 64, 64, None, 300, 4, 1024, 2, None, None) == nv.ERR_INVALID_VALUE
    assert G(64, 72, 64, 64, 64, 300, 4, 1024, 2, None, None) == nv.ERR_MISALIGNED
    assert G(64, 64, 80, 64, 64, 300, 4, 1024, 2, None, None) == nv.ERR_MISALIGNED
    assert G(64, 64, 64, 64, 65, 300, 4, 1024, 2, None, None) == nv.ERR_MISALIGNED
    # b batch stride below N*K/2, or not a multiple of 16
    opt = nv._Options(1.0, None, 4 * 512 - 32, 0)
    assert G(*ptrs, 300, 4, 1024, 2, ctypes.byref(opt), None) == nv.ERR_INVALID_VALUE
    opt = nv._Options(1.0, None, 4 * 512 + 8, 0)
    assert G(*ptrs, 300, 4, 1024, 2, ctypes.byref(opt), None) == nv.ERR_MISALIGNED
    # sfb batch stride below (K/64)*512, or not a multiple of 16
    opt = nv._Options(1.0, None, 0, 16 * 512 - 16)
    assert G(*ptrs, 300, 4, 1024, 2, ctypes.byref(opt), None) == nv.ERR_INVALID_VALUE
    opt = nv._Options(1.0, None, 0, 16 * 512 + 8)
    assert G(*ptrs, 300, 4, 1024, 2, ctypes.byref(opt), None) == nv.ERR_MISALIGNED
    # explicit schedules: stages 2 or 4; cluster sizes 1/2/4/8 within the K stages; whole clusters
    args = ptrs + (300, 4, 1024, 2)
    assert E(*args, 3, 1, 1, None) == nv.ERR_INVALID_VALUE
    assert E(*args, 2, 3, 3, None) == nv.ERR_INVALID_VALUE
    assert E(*args, 2, 8, 8, None) == nv.ERR_INVALID_VALUE  # K = 1024: 4 stages
    assert E(*args, 4, 2, 3, None) == nv.ERR_INVALID_VALUE
    assert E(*args, 2, 1, 0, None) == nv.ERR_INVALID_VALUE
    assert E(*(ptrs + (300, 4, 0, 2)), 2, 2, 2, None) == nv.ERR_INVALID_VALUE  # K = 0: no split
    assert E(*(ptrs + (0, 4, 1024, 2)), 2, 1, 1, None) == nv.OK


def test_gemm_small_n_plan_validation(lib):
    st, ks, ctas, res = ctypes.c_int(), ctypes.c_int(), ctypes.c_int64(), ctypes.c_int()
    args = (ctypes.byref(st), ctypes.byref(ks), ctypes.byref(ctas), ctypes.byref(res))
    assert lib.nvfp4_gemm_small_n_plan(300, 17, 1024, 2, *args) == nv.ERR_UNSUPPORTED_SHAPE
    assert lib.nvfp4_gemm_small_n_plan(300, 4, 1000, 2, *args) == nv.ERR_UNSUPPORTED_SHAPE
    assert lib.nvfp4_gemm_small_n_plan(-1, 4, 1024, 2, *args) == nv.ERR_UNSUPPORTED_SHAPE
    assert lib.nvfp4_gemm_small_n_plan(300, 4, 1024, 2, None, None, None, None) == \
        nv.ERR_INVALID_VALUE


def test_options_validation(lib):
    """nvfp4_gemv_ex / nvfp4_gemm_small_n options, checked before any CUDA call."""
    import ctypes

    def opt(**kw):
        o = nv._Options(1.0, None, 0, 0, 0)
        for k, v in kw.items():
            setattr(o, k, v)
        return ctypes.byref(o)

    args = (64, 64, 64, 64, 64, 8, 256, 2, 0)
    for act in (-1, 5, 99):
        assert lib.nvfp4_gemv_ex(*args, opt(activation=act), None) == nv.ERR_INVALID_VALUE
        assert lib.nvfp4_gemm_small_n(64, 64, 64, 64, 64, 8, 4, 256, 2, opt(activation=act),
                                      None) == nv.ERR_INVALID_VALUE
    assert lib.nvfp4_gemv_ex(*args, opt(b_batch_stride=-16), None) == nv.ERR_INVALID_VALUE
    assert lib.nvfp4_gemv_ex(*args, opt(b_batch_stride=64), None) == nv.ERR_INVALID_VALUE  # < K/2
    assert lib.nvfp4_gemv_ex(*args, opt(b_batch_stride=136), None) == nv.ERR_MISALIGNED
    assert lib.nvfp4_gemv_ex(*args, opt(bias=65), None) == nv.ERR_MISALIGNED
    # empty problems with a valid activation are no-ops
    for act in range(5):
        assert lib.nvfp4_gemv_ex(None, None, None, None, None, 0, 256, 2, 0, opt(activation=act),
                                 None) == nv.OK


def test_huge_shapes_plan_without_overflow(lib):
    # M*L*K/2 beyond 2^63: the byte count saturates instead of wrapping into
    # the tiny-problem schedule
    M, K, L = (1 << 31) - 1, 1 << 30, 500
    plan = nv.nvfp4_gemv_plan(M, K, L, nv.SF_PLAIN, 152, 2)
    assert plan["kernel"] == nv.KERNEL_PIPELINED and plan["ctas"] == 304
    # the small-N GEMM's 128-row tiles must number below 2^31
    st, ks, ctas = ctypes.c_int(), ctypes.c_int(), ctypes.c_int64()
    assert lib.nvfp4_gemm_small_n_plan(M, 4, 1024, 200, ctypes.byref(st), ctypes.byref(ks),
                                       ctypes.byref(ctas), None) == nv.ERR_UNSUPPORTED_SHAPE
