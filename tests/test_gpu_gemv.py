"""GPU parity of nvfp4_gemv against the CPU oracle, called through the C ABI.

Small and ragged shapes are compared element by element; the full-size
benchmark workloads, in the launch schedule the benchmark times, are
compared on sampled outputs the oracle computes one by one.  Tolerance:
|gpu - oracle| <= 1e-3 * sum|terms| + 1 fp16 ulp of the oracle value.
"""
import json
import math
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import nvfp4_block_scaled_gemv_gb300 as nv  # noqa: E402
import oracle  # noqa: E402
from nvfp4_block_scaled_gemv_gb300 import build as libbuild  # noqa: E402
from nvfp4_block_scaled_gemv_gb300 import synthetic  # noqa: E402
from oracle import parity  # noqa: E402

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
SENTINEL = -4096.0
SENTINEL_BITS = int(np.array([SENTINEL], dtype=np.float16).view(np.uint16)[0])


@pytest.fixture(scope="module", autouse=True)
def _lib():
    libbuild.build()
    nv.library()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def to_dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(DEV)


def bits(c):
    return c.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def device_problem(p, M, K, L, layout, via_gpu_repack=False):
    a, b = to_dev(p["a"]), to_dev(p["b"])
    if layout == nv.SF_PLAIN:
        sfa, sfb = to_dev(p["sfa"]), to_dev(p["sfb"])
    elif via_gpu_repack:
        sfa = nv.repack_scales(to_dev(p["sfa"]))
        sfb = nv.repack_scales(to_dev(p["sfb"].reshape(L, 1, K // 16)))
    else:
        sfa = to_dev(oracle.repack_scales(p["sfa"], M, K, L))
        sfb = to_dev(oracle.repack_scales(p["sfb"].reshape(L, 1, K // 16), 1, K, L))
    return a, b, sfa, sfb


def run(p, M, K, L, layout=nv.SF_PLAIN, schedule=None, via_gpu_repack=False):
    a, b, sfa, sfb = device_problem(p, M, K, L, layout, via_gpu_repack)
    # sentinel-filled c with slack on both sides: nothing outside [0, L*M) may change
    pad = 64
    buf = torch.full((L * M + 2 * pad,), SENTINEL, dtype=torch.float16, device=DEV)
    c = buf[pad:pad + L * M]
    if schedule is None:
        nv.nvfp4_gemv(a.data_ptr(), b.data_ptr(), sfa.data_ptr(), sfb.data_ptr(), c.data_ptr(),
                      M, K, L, layout, torch.cuda.current_stream().cuda_stream)
    else:
        kernel, lpr, ks, ctas = schedule
        nv.nvfp4_gemv_explicit(a.data_ptr(), b.data_ptr(), sfa.data_ptr(), sfb.data_ptr(),
                               c.data_ptr(), M, K, L, layout, kernel, lpr, ks, ctas,
                               torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    whole = bits(buf)
    assert np.all(whole[:pad] == SENTINEL_BITS) and np.all(whole[pad + L * M:] == SENTINEL_BITS), \
        "write outside c"
    return whole[pad:pad + L * M].reshape(L, M)


SMALL_SHAPES = [
    (128, 256, 1),   # the smallest benchmark workload
    (1, 64, 1), (7, 64, 2), (8, 128, 1), (9, 192, 3), (31, 320, 1), (33, 1024, 2),
    (127, 2048, 1), (129, 448, 2), (200, 7168, 1), (256, 4096, 3), (1000, 64, 4),
    (37, 16384, 1), (513, 1152, 2),
]


@pytest.mark.parametrize("layout", [nv.SF_PLAIN, nv.SF_PERMUTED_128x4])
@pytest.mark.parametrize("M,K,L", SMALL_SHAPES)
def test_parity_all_outputs(M, K, L, layout):
    p = synthetic.make_problem(M, K, L, seed=M + K + L)
    ref, sums, sumabs = oracle.gemv(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L)
    got = run(p, M, K, L, layout)
    parity.assert_parity(got, ref, sums, sumabs, f"M={M} K={K} L={L} layout={layout}")


@pytest.mark.parametrize("kernel", [nv.KERNEL_DIRECT, nv.KERNEL_PIPELINED])
@pytest.mark.parametrize("lpr", [4, 8, 16, 32])
@pytest.mark.parametrize("ks", [1, 2, 4, 8])
def test_every_schedule(kernel, lpr, ks):
    M, K, L = 150, 2560, 3
    if kernel == nv.KERNEL_PIPELINED and ks > -(-(K // 64) // lpr):
        pytest.skip("the pipelined kernel needs a K step for every K-split warp")
    p = synthetic.make_problem(M, K, L, seed=lpr * 10 + ks)
    ref, sums, sumabs = oracle.gemv(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L)
    outs = []
    # grid sizes that give the pipelined kernel 1, 2 and 4 row groups per pass
    # and several passes per row lane
    for ctas in (1, 5, 13, 40, 150, 600):
        for layout in (nv.SF_PLAIN, nv.SF_PERMUTED_128x4):
            got = run(p, M, K, L, layout, schedule=(kernel, lpr, ks, ctas))
            parity.assert_parity(got, ref, sums, sumabs,
                                 f"kernel={kernel} lpr={lpr} ks={ks} ctas={ctas}")
            outs.append(got)
    # the summation order depends only on (kernel, lpr, ks): grid and layout change no bit
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


def _sample_indices(M, L, n, rng):
    m = [0, M - 1, min(127, M - 1), min(128, M - 1), M // 2]
    mi = np.concatenate([rng.integers(0, M, n), np.tile(m, L)])
    li = np.concatenate([rng.integers(0, L, n), np.repeat(np.arange(L), len(m))])
    return mi, li


@pytest.mark.parametrize("name,M,K,L", synthetic.WORKLOADS[1:])
def test_full_size_workloads_sampled(name, M, K, L):
    p = synthetic.make_problem(M, K, L, seed=0)
    rng = np.random.default_rng(1)
    mi, li = _sample_indices(M, L, 3000, rng)
    ref, sums, sumabs = oracle.gemv_at(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L, mi, li)
    results = {}
    for layout in (nv.SF_PLAIN, nv.SF_PERMUTED_128x4):
        got = run(p, M, K, L, layout, via_gpu_repack=(layout == nv.SF_PERMUTED_128x4))
        parity.assert_parity(got[li, mi], ref, sums, sumabs, f"{name} layout={layout}")
        assert np.isfinite(parity.half_values(got)).all()
        results[layout] = got
    # the benchmark's scale codes keep every partial sum exact in fp32, so even
    # different kernels (M16384_K8192_L16 permuted runs on the tensor cores)
    # give the same bits in both layouts
    assert np.array_equal(results[nv.SF_PLAIN], results[nv.SF_PERMUTED_128x4])


def test_default_route_takes_the_tensor_cores_for_multi_wave_permuted_streams():
    # pre-permuted scales, more than one wave of 128-row tiles, 128 MB of A:
    # nvfp4_gemv picks the tensor-core kernel; scales over 0x01..0x50 so that
    # the fp32 sums round
    M, K, L = 16384, 2048, 8
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert nv.nvfp4_gemv_plan(M, K, L, nv.SF_PERMUTED_128x4, sms, 0)["kernel"] == nv.KERNEL_TENSOR
    p = synthetic.make_problem(M, K, L, seed=12, scale_codes=(0x01, 0x50))
    mi, li = _sample_indices(M, L, 3000, np.random.default_rng(6))
    ref, sums, sumabs = oracle.gemv_at(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L, mi, li)
    got = run(p, M, K, L, nv.SF_PERMUTED_128x4, via_gpu_repack=True)
    assert nv.nvfp4_tensor_wait_timeouts(reset=True) == 0
    parity.assert_parity(got[li, mi], ref, sums, sumabs, "M16384_K2048_L8 permuted, default route")


def test_hand_worked_golden_values(golden_dir):
    with open(os.path.join(golden_dir, "hand_dots.json")) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        p = {"a": np.frombuffer(bytes.fromhex(case["a"]), np.uint8).reshape(1, 1, 32),
             "b": np.frombuffer(bytes.fromhex(case["b"]), np.uint8).reshape(1, 32),
             "sfa": np.frombuffer(bytes.fromhex(case["sfa"]), np.uint8).reshape(1, 1, 4),
             "sfb": np.frombuffer(bytes.fromhex(case["sfb"]), np.uint8).reshape(1, 4)}
        for layout in (nv.SF_PLAIN, nv.SF_PERMUTED_128x4):
            got = float(parity.half_values(run(p, 1, 64, 1, layout))[0, 0])
            want = float(case["expected"])
            if math.isnan(want):
                assert math.isnan(got), case["name"]
            else:
                assert got == want, (case["name"], layout, got, want)


def test_sign_flip_and_scale_doubling_are_exact():
    M, K, L = 300, 4096, 2
    p = synthetic.make_problem(M, K, L, seed=21)
    base = parity.half_values(run(p, M, K, L))
    flipped = dict(p, b=p["b"] ^ 0x88)
    assert np.array_equal(parity.half_values(run(flipped, M, K, L)), -base)
    doubled = dict(p, sfb=p["sfb"] + 8)
    assert np.array_equal(parity.half_values(run(doubled, M, K, L)), 2 * base)


def test_extreme_codes_and_nan():
    rng = np.random.default_rng(5)
    M, K, L = 64, 512, 2
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    p = {"a": rng.integers(0, 256, (L, M, K // 2), dtype=np.uint8),
         "b": rng.integers(0, 256, (L, K // 2), dtype=np.uint8),
         "sfa": rng.choice(finite, (L, M, K // 16)),
         "sfb": rng.choice(finite, (L, K // 16))}
    p["sfa"][0, 3, 5] = 0x7F           # NaN scale on one row
    p["sfb"][1, 2] = 0xFF              # NaN scale on every row of batch 1
    p["a"][0, 10] = 0x77               # +6 everywhere
    p["sfa"][0, 10] = 0x7E             # 448: overflows to +inf
    ref, sums, sumabs = oracle.gemv(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L)
    for layout in (nv.SF_PLAIN, nv.SF_PERMUTED_128x4):
        got = run(p, M, K, L, layout)
        parity.assert_parity(got, ref, sums, sumabs, f"extreme layout={layout}")
        v = parity.half_values(got)
        assert np.isnan(v[0, 3]) and np.isnan(v[1]).all()


def test_zero_k_writes_zeros_and_empty_is_noop():
    M, L = 100, 3
    c = torch.full((L, M), 7.0, dtype=torch.float16, device=DEV)
    nv.nvfp4_gemv(0, 0, 0, 0, c.data_ptr(), M, 0, L, nv.SF_PLAIN,
                  torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert np.all(bits(c) == 0)
    nv.nvfp4_gemv(0, 0, 0, 0, 0, 0, 128, L, nv.SF_PLAIN, 0)
    nv.nvfp4_gemv(0, 0, 0, 0, 0, M, 128, 0, nv.SF_PLAIN, 0)


def test_deterministic_run_to_run():
    M, K, L = 7168, 2048, 4
    p = synthetic.make_problem(M, K, L, seed=3)
    a, b, sfa, sfb = device_problem(p, M, K, L, nv.SF_PLAIN)
    outs = []
    for _ in range(3):
        c = nv.gemv(a.view(L, M, K // 2), b, sfa.view(L, M, K // 16), sfb)
        torch.cuda.synchronize()
        outs.append(bits(c))
    assert all(np.array_equal(outs[0], o) for o in outs[1:])


def test_misaligned_device_pointers_rejected_without_launch():
    M, K, L = 16, 128, 1
    buf = torch.zeros(4096, dtype=torch.uint8, device=DEV)
    c = torch.full((M,), 3.0, dtype=torch.float16, device=DEV)
    base = buf.data_ptr()
    for ptrs in ((base + 8, base + 1024, base + 2048, base + 3072),
                 (base, base + 1032, base + 2048, base + 3072),
                 (base, base + 1024, base + 2064, base + 3072)):
        with pytest.raises(nv.Nvfp4Error) as e:
            nv.nvfp4_gemv(*ptrs, c.data_ptr(), M, K, L)
        assert e.value.status == nv.ERR_MISALIGNED
    # a direct-kernel schedule needs a 32-byte aligned a
    with pytest.raises(nv.Nvfp4Error) as e:
        nv.nvfp4_gemv_explicit(base + 16, base + 1024, base + 2048, base + 3072, c.data_ptr(),
                               M, K, L, nv.SF_PLAIN, nv.KERNEL_DIRECT, 4, 1, 1)
    assert e.value.status == nv.ERR_MISALIGNED
    torch.cuda.synchronize()
    assert np.all(parity.half_values(bits(c)) == 3.0)


@pytest.mark.parametrize("layout", [nv.SF_PLAIN, nv.SF_PERMUTED_128x4])
@pytest.mark.parametrize("M,K,L", [(128, 256, 1), (7, 1024, 3), (1000, 2048, 2), (4096, 4096, 4)])
def test_sixteen_byte_aligned_a_and_b(M, K, L, layout):
    """a and b 16 bytes past a 32-byte boundary (the pages' assumed_align=16):
    the library's own schedule (never the direct kernel for such an a), and
    every other kernel that runs the shape, against the oracle."""
    p = synthetic.make_problem(M, K, L, seed=M + 3 * K)
    ref, sums, sumabs = oracle.gemv(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L)
    abuf = torch.empty(p["a"].size + 64, dtype=torch.uint8, device=DEV)
    bbuf = torch.empty(p["b"].size + 64, dtype=torch.uint8, device=DEV)
    a_off, b_off = (16 - abuf.data_ptr()) % 32, (16 - bbuf.data_ptr()) % 32
    a = abuf[a_off:a_off + p["a"].size]
    b = bbuf[b_off:b_off + p["b"].size]
    assert a.data_ptr() % 32 == 16 and b.data_ptr() % 32 == 16
    a.copy_(torch.from_numpy(p["a"].reshape(-1)))
    b.copy_(torch.from_numpy(p["b"].reshape(-1)))
    _, _, sfa, sfb = device_problem(p, M, K, L, layout)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    runs = [None]
    for kern in (nv.KERNEL_PIPELINED, nv.KERNEL_BLOCKDOT):
        if kern == nv.KERNEL_BLOCKDOT and layout == nv.SF_PLAIN and K % 256:
            continue
        plan = nv.nvfp4_gemv_plan(M, K, L, layout, sms, 0, kernel=kern)
        runs.append((kern, plan["lanes_per_row"], plan["k_split"], plan["ctas"]))
    for sched in runs:
        c = torch.full((L * M,), SENTINEL, dtype=torch.float16, device=DEV)
        if sched is None:
            nv.nvfp4_gemv(a.data_ptr(), b.data_ptr(), sfa.data_ptr(), sfb.data_ptr(), c.data_ptr(),
                          M, K, L, layout, torch.cuda.current_stream().cuda_stream)
        else:
            nv.nvfp4_gemv_explicit(a.data_ptr(), b.data_ptr(), sfa.data_ptr(), sfb.data_ptr(),
                                   c.data_ptr(), M, K, L, layout, *sched,
                                   stream=torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        parity.assert_parity(bits(c).reshape(L, M), ref, sums, sumabs,
                             f"16-byte aligned a, b M={M} K={K} L={L} layout={layout} {sched}")


def test_graph_capture_and_replay():
    M, K, L = 512, 1024, 2
    p = synthetic.make_problem(M, K, L, seed=8)
    a, b, sfa, sfb = device_problem(p, M, K, L, nv.SF_PLAIN)
    a, sfa = a.view(L, M, K // 2), sfa.view(L, M, K // 16)
    c = torch.zeros((L, M), dtype=torch.float16, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        nv.gemv(a, b, sfa, sfb, c)  # warm-up outside capture
    torch.cuda.synchronize()
    want = bits(c)
    c.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        nv.gemv(a, b, sfa, sfb, c, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(bits(c), want)


def test_random_shapes_default_schedule():
    """Random shapes through the library's own plans (row groups per pass,
    ragged batches, narrow permuted rows, K splits) against the oracle."""
    rng = np.random.default_rng(2024)
    for case in range(24):
        M = int(rng.integers(1, 3000))
        K = 64 * int(rng.integers(1, 129))
        L = int(rng.integers(1, 6))
        layout = int(rng.integers(0, 2))
        p = synthetic.make_problem(M, K, L, seed=1000 + case)
        ref, sums, sumabs = oracle.gemv(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L)
        got = run(p, M, K, L, layout)
        plan = nv.nvfp4_gemv_plan(M, K, L, layout, torch.cuda.get_device_properties(0).multi_processor_count, 0)
        parity.assert_parity(got, ref, sums, sumabs, f"case {case}: M={M} K={K} L={L} layout={layout} plan={plan}")


# --- nvfp4_gemv_ex: output scale, bias, batch strides of b and sfb -----------

def _ex_call(a, b, sfa, sfb, c, M, K, L, layout, **kw):
    nv.nvfp4_gemv_ex(a.data_ptr(), b.data_ptr(), sfa.data_ptr(), sfb.data_ptr(), c.data_ptr(),
                     M, K, L, layout, stream=torch.cuda.current_stream().cuda_stream, **kw)
    torch.cuda.synchronize()
    return bits(c).reshape(L, M)


@pytest.mark.parametrize("layout", [nv.SF_PLAIN, nv.SF_PERMUTED_128x4])
def test_gemv_ex_defaults_are_nvfp4_gemv(layout):
    M, K, L = 700, 2048, 3
    p = synthetic.make_problem(M, K, L, seed=41)
    base = run(p, M, K, L, layout)
    a, b, sfa, sfb = device_problem(p, M, K, L, layout)
    c = torch.empty(L * M, dtype=torch.float16, device=DEV)
    assert np.array_equal(_ex_call(a, b, sfa, sfb, c, M, K, L, layout), base)


@pytest.mark.parametrize("layout", [nv.SF_PLAIN, nv.SF_PERMUTED_128x4])
@pytest.mark.parametrize("M,K,L,alpha", [(700, 2048, 3, 0.375), (129, 7168, 2, -1.5e-3),
                                         (4096, 1024, 2, 37.0), (130, 80, 3, -0.75),
                                         (300, 1040, 2, 3.0)])
def test_gemv_ex_alpha_bias_and_padded_b(layout, M, K, L, alpha):
    """b as row 0 of an [L][8][K/2] buffer and sfb in a padded per-batch
    stride, the other rows random: only row 0 may reach c."""
    p = synthetic.make_problem(M, K, L, seed=M + K)
    rng = np.random.default_rng(M)
    bias = (rng.standard_normal((L, M)) * 8).astype(np.float16).view(np.uint16)
    ref, vals, sumabs = oracle.gemv_ex(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L,
                                       alpha=alpha, bias=bias)
    a, b, sfa, sfb = device_problem(p, M, K, L, layout)
    N = 8
    b_pad = torch.from_numpy(rng.integers(0, 256, (L, N, K // 2), dtype=np.uint8)).to(DEV)
    b_pad[:, 0, :] = b.view(L, K // 2)
    sfb_dense = sfb.numel() // L
    sfb_stride = -(-2 * sfb_dense // 16) * 16  # a multiple of 16 (of 4 for plain scales)
    sfb_pad = torch.from_numpy(rng.integers(0, 256, (L, sfb_stride), dtype=np.uint8)).to(DEV)
    sfb_pad[:, :sfb_dense] = sfb.view(L, sfb_dense)
    c = torch.full((L * M,), SENTINEL, dtype=torch.float16, device=DEV)
    bias_d = torch.from_numpy(bias.reshape(-1).copy()).to(DEV)
    got = _ex_call(a, b_pad, sfa, sfb_pad, c, M, K, L, layout, alpha=alpha,
                   bias=bias_d.data_ptr(), b_batch_stride=N * (K // 2),
                   sfb_batch_stride=sfb_stride)
    parity.assert_parity(got, ref, vals, sumabs, f"ex M={M} K={K} L={L} alpha={alpha} layout={layout}")


@pytest.mark.parametrize("activation", [nv.ACT_RELU, nv.ACT_SILU, nv.ACT_GELU_TANH,
                                        nv.ACT_GELU_ERF])
@pytest.mark.parametrize("layout", [nv.SF_PLAIN, nv.SF_PERMUTED_128x4])
@pytest.mark.parametrize("M,K,L", [(128, 256, 1), (700, 2048, 3), (130, 80, 3)])
def test_gemv_ex_activation(activation, layout, M, K, L):
    """Each kernel nvfp4_gemv_ex picks (direct, pipelined, blockwise) with an
    output scale, a bias and each activation, against the oracle."""
    p = synthetic.make_problem(M, K, L, seed=M + K + activation)
    rng = np.random.default_rng(activation)
    bias = (rng.standard_normal((L, M)) * 2).astype(np.float16).view(np.uint16)
    _, s, _ = oracle.gemv(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L)
    alpha = float(2.0 / max(np.std(s), 1e-3))
    ref, vals, tol = oracle.gemv_ex(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L, alpha=alpha,
                                    bias=bias, activation=activation)
    a, b, sfa, sfb = device_problem(p, M, K, L, layout)
    c = torch.full((L * M,), SENTINEL, dtype=torch.float16, device=DEV)
    bias_d = torch.from_numpy(bias.reshape(-1).copy()).to(DEV)
    got = _ex_call(a, b, sfa, sfb, c, M, K, L, layout, alpha=alpha, bias=bias_d.data_ptr(),
                   activation=activation)
    parity.assert_parity(got, ref, vals, tol,
                         f"act={activation} M={M} K={K} L={L} layout={layout}")
    v = got.view(np.float16).astype(np.float64)
    assert (v > 0).any() and ((v < 0).any() or activation == nv.ACT_RELU)


def test_gemv_ex_zero_k_gives_the_bias():
    M, L = 37, 2
    bias = (np.arange(L * M, dtype=np.float32) - 20).astype(np.float16)
    bias_d = torch.from_numpy(bias).to(DEV)
    c = torch.full((L * M,), SENTINEL, dtype=torch.float16, device=DEV)
    nv.nvfp4_gemv_ex(0, 0, 0, 0, c.data_ptr(), M, 0, L, nv.SF_PLAIN, alpha=3.0,
                     bias=bias_d.data_ptr(), stream=torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert np.array_equal(c.cpu().numpy().astype(np.float64), bias.astype(np.float64))


@pytest.mark.parametrize("layout", [nv.SF_PLAIN, nv.SF_PERMUTED_128x4])
@pytest.mark.parametrize("M,K,L", [(1, 64, 1000), (100000, 64, 1), (3, 16384, 7), (129, 128, 33),
                                   (2, 2048, 300)])
def test_extreme_shapes(M, K, L, layout):
    """One-row batches by the thousand, 100k rows of one chunk, long K over
    tiny batches, one row past an atom block: every output against the oracle."""
    p = synthetic.make_problem(M, K, L, seed=M * 7 + K + L)
    ref, sums, sumabs = oracle.gemv(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L)
    got = run(p, M, K, L, layout, via_gpu_repack=(layout == nv.SF_PERMUTED_128x4))
    parity.assert_parity(got, ref, sums, sumabs, f"M={M} K={K} L={L} layout={layout}")


# --- K % 16 == 0 with K % 64 != 0: the blockwise kernel --------------------

K16_SHAPES = [(1, 16, 1), (7, 48, 2), (130, 80, 3), (33, 1040, 2), (513, 208, 1),
              (1000, 4112, 2), (4, 16, 300)]


@pytest.mark.parametrize("M,K,L", K16_SHAPES)
def test_k_multiple_of_16(M, K, L):
    """Every output against the oracle, both layouts (permuted scales through
    the oracle's and through the GPU's repack, with the padded last atom
    column), the default plan and explicit grids: one set of bits, since the
    blockwise kernel's summation order depends on K alone."""
    p = synthetic.make_problem(M, K, L, seed=M + 3 * K + L)
    ref, sums, sumabs = oracle.gemv(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    outs = []
    for layout in (nv.SF_PLAIN, nv.SF_PERMUTED_128x4):
        assert nv.nvfp4_gemv_plan(M, K, L, layout, sms, 0)["kernel"] == nv.KERNEL_BLOCKWISE
        runs = [run(p, M, K, L, layout)]
        if layout == nv.SF_PERMUTED_128x4:
            runs.append(run(p, M, K, L, layout, via_gpu_repack=True))
        for ctas in (1, 3, 40, 1000):
            runs.append(run(p, M, K, L, layout, schedule=(nv.KERNEL_BLOCKWISE, 32, 1, ctas)))
        for got in runs:
            parity.assert_parity(got, ref, sums, sumabs, f"M={M} K={K} L={L} layout={layout}")
        outs += runs
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


@pytest.mark.parametrize("M,K,L", [(150, 2560, 3), (128, 256, 1), (37, 16384, 1)])
def test_blockwise_kernel_on_k_multiple_of_64(M, K, L):
    p = synthetic.make_problem(M, K, L, seed=K + L)
    ref, sums, sumabs = oracle.gemv(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L)
    outs = []
    for layout in (nv.SF_PLAIN, nv.SF_PERMUTED_128x4):
        got = run(p, M, K, L, layout, schedule=(nv.KERNEL_BLOCKWISE, 32, 1, 64))
        parity.assert_parity(got, ref, sums, sumabs, f"blockwise M={M} K={K} L={L}")
        outs.append(got)
    assert np.array_equal(outs[0], outs[1])


def test_random_k16_shapes_default_schedule():
    rng = np.random.default_rng(77)
    for case in range(16):
        M = int(rng.integers(1, 2000))
        K = 16 * int(rng.integers(1, 400))
        L = int(rng.integers(1, 5))
        layout = int(rng.integers(0, 2))
        p = synthetic.make_problem(M, K, L, seed=2000 + case)
        ref, sums, sumabs = oracle.gemv(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L)
        got = run(p, M, K, L, layout, via_gpu_repack=bool(case % 2))
        parity.assert_parity(got, ref, sums, sumabs, f"case {case}: M={M} K={K} L={L} layout={layout}")


def test_k16_large_sampled():
    """A 59 MB A with K % 64 == 16, above nothing but the blockwise kernel's
    own schedule: sampled outputs against the oracle."""
    M, K, L = 7168, 16400, 1
    p = synthetic.make_problem(M, K, L, seed=5)
    mi, li = _sample_indices(M, L, 2000, np.random.default_rng(8))
    ref, sums, sumabs = oracle.gemv_at(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L, mi, li)
    for layout in (nv.SF_PLAIN, nv.SF_PERMUTED_128x4):
        got = run(p, M, K, L, layout, via_gpu_repack=(layout == nv.SF_PERMUTED_128x4))
        parity.assert_parity(got[li, mi], ref, sums, sumabs, f"M={M} K={K} layout={layout}")


@pytest.mark.parametrize("layout", [nv.SF_PLAIN, nv.SF_PERMUTED_128x4])
def test_large_stream_runs_on_tensor_cores_with_options(layout):
    """>= 512 MB of A with K <= 8192 (nvfp4_gemv's tensor-core route, plain
    scales laid out as atoms in shared memory): alpha, an fp16 bias, SiLU and
    b / sfb in padded buffers, sampled outputs against the oracle; the plain
    call's bits equal the pipelined kernel's (exact sums on the benchmark's
    scale codes).  With plain scales, a sfb batch stride that is not a
    multiple of 16 bytes takes the pipelined kernel, with the same bits."""
    M, K, L = 16384, 8192, 12
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert nv.nvfp4_gemv_plan(M, K, L, layout, sms, 0)["kernel"] == nv.KERNEL_TENSOR
    p = synthetic.make_problem(M, K, L, seed=31)
    rng = np.random.default_rng(5)
    mi, li = _sample_indices(M, L, 4000, rng)
    bias = (rng.standard_normal((L, M)) * 2).astype(np.float16).view(np.uint16)
    _, s_all, _ = oracle.gemv_at(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L, mi, li)
    alpha = float(2.0 / max(np.std(s_all), 1e-3))
    ref, sums, sumabs = oracle.gemv_at(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L, mi, li)
    y = oracle.activate(alpha * sums + bias.view(np.float16).astype(np.float64)[li, mi], oracle.ACT_SILU)
    ref_ex = oracle.fp16_rne(y)
    tol_ex = oracle.LIPSCHITZ[oracle.ACT_SILU] * abs(alpha) * sumabs
    a, b, sfa, sfb = device_problem(p, M, K, L, layout, via_gpu_repack=True)
    # plain call: tensor cores, against the oracle and against the pipelined kernel
    c = torch.empty(L * M, dtype=torch.float16, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream
    nv.nvfp4_gemv(a.data_ptr(), b.data_ptr(), sfa.data_ptr(), sfb.data_ptr(), c.data_ptr(), M, K, L,
                  layout, stream)
    torch.cuda.synchronize()
    assert nv.nvfp4_tensor_wait_timeouts(reset=True) == 0
    got = bits(c).reshape(L, M)
    parity.assert_parity(got[li, mi], ref, sums, sumabs, "tensor route, plain call")
    plan = nv.nvfp4_gemv_plan(M, K, L, layout, sms, 0, kernel=nv.KERNEL_PIPELINED)
    c2 = torch.empty_like(c)
    nv.nvfp4_gemv_explicit(a.data_ptr(), b.data_ptr(), sfa.data_ptr(), sfb.data_ptr(), c2.data_ptr(),
                           M, K, L, layout, nv.KERNEL_PIPELINED, plan["lanes_per_row"],
                           plan["k_split"], plan["ctas"], stream=stream)
    torch.cuda.synchronize()
    assert np.array_equal(bits(c2).reshape(L, M), got)
    # with options: b as row 0 of an [L][2][K/2] buffer, sfb at twice its dense stride
    b_pad = torch.zeros((L, 2, K // 2), dtype=torch.uint8, device=DEV)
    b_pad[:, 0, :] = b.view(L, K // 2)
    dense = sfb.numel() // L
    sfb_pad = torch.full((L, 2 * dense), 0x7F, dtype=torch.uint8, device=DEV)  # NaN if misread
    sfb_pad[:, :dense] = sfb.view(L, dense)
    bias_d = torch.from_numpy(bias.reshape(-1).copy()).to(DEV)
    c3 = torch.full((L * M,), SENTINEL, dtype=torch.float16, device=DEV)
    nv.nvfp4_gemv_ex(a.data_ptr(), b_pad.data_ptr(), sfa.data_ptr(), sfb_pad.data_ptr(), c3.data_ptr(),
                     M, K, L, layout, alpha=alpha, bias=bias_d.data_ptr(),
                     b_batch_stride=K, sfb_batch_stride=2 * dense, stream=stream,
                     activation=nv.ACT_SILU)
    torch.cuda.synchronize()
    assert nv.nvfp4_tensor_wait_timeouts(reset=True) == 0
    got3 = bits(c3).reshape(L, M)
    parity.assert_parity(got3[li, mi], ref_ex, y, tol_ex, "tensor route with options")
    if layout == nv.SF_PLAIN:
        # sfb rows 4 bytes apart from 16-byte alignment: the pipelined kernel
        odd = dense + 4
        sfb_odd = torch.full((L, odd), 0x7F, dtype=torch.uint8, device=DEV)
        sfb_odd[:, :dense] = sfb.view(L, dense)
        c4 = torch.full((L * M,), SENTINEL, dtype=torch.float16, device=DEV)
        nv.nvfp4_gemv_ex(a.data_ptr(), b_pad.data_ptr(), sfa.data_ptr(), sfb_odd.data_ptr(),
                         c4.data_ptr(), M, K, L, layout, alpha=alpha, bias=bias_d.data_ptr(),
                         b_batch_stride=K, sfb_batch_stride=odd, stream=stream,
                         activation=nv.ACT_SILU)
        torch.cuda.synchronize()
        assert np.array_equal(bits(c4).reshape(L, M), got3)
