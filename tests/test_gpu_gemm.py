"""GPU parity of the small-N NVFP4 GEMM (nvfp4_gemm_small_n) against the CPU oracle.

c [L][N][M] is compared element by element with oracle.gemm_small_n (N GEMVs
sharing A), tolerance |gpu - oracle| <= 1e-3 * |alpha| * sum|terms| + 1 fp16
ulp of the oracle value.  Scales reach the GPU in the pre-permuted layout
made by the library's own repack (sfa with rows = M, sfb with rows = N).
Every launch is checked for writes outside c and for pipeline waits that ran
out.
"""
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
    nv.nvfp4_tensor_wait_timeouts(reset=True)


def to_dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(DEV)


def run_gemm(p, M, N, K, L, schedule=None, alpha=1.0, bias=None, b_pad_rows=0, activation=0):
    """c bits [L, N, M]; schedule = (stages, k_split, ctas) for the explicit call.
    b_pad_rows > 0 puts b in an [L][N + b_pad_rows][K/2] buffer (batch stride)."""
    a = to_dev(p["a"])
    if b_pad_rows:
        bb = np.zeros((L, N + b_pad_rows, K // 2), dtype=np.uint8)
        bb[:, :N] = p["b"]
        b = to_dev(bb)
        b_stride = (N + b_pad_rows) * (K // 2)
    else:
        b = to_dev(p["b"]) if K else torch.zeros(32, dtype=torch.uint8, device=DEV)
        b_stride = 0
    if K:
        sfa = nv.repack_scales(to_dev(p["sfa"]))
        sfb = nv.repack_scales(to_dev(p["sfb"]))
    else:
        sfa = sfb = torch.zeros(32, dtype=torch.uint8, device=DEV)
    pad = 64
    n_out = L * N * M
    buf = torch.full((n_out + 2 * pad,), SENTINEL, dtype=torch.float16, device=DEV)
    c = buf[pad:pad + n_out]
    stream = torch.cuda.current_stream().cuda_stream
    bias_t = to_dev(bias) if bias is not None else None
    if schedule is None:
        nv.nvfp4_gemm_small_n(a.data_ptr(), b.data_ptr(), sfa.data_ptr(), sfb.data_ptr(),
                              c.data_ptr(), M, N, K, L, alpha=alpha,
                              bias=bias_t.data_ptr() if bias_t is not None else 0,
                              b_batch_stride=b_stride, stream=stream, activation=activation)
    else:
        assert alpha == 1.0 and bias is None and not b_pad_rows and not activation
        nv.nvfp4_gemm_small_n_explicit(a.data_ptr(), b.data_ptr(), sfa.data_ptr(),
                                       sfb.data_ptr(), c.data_ptr(), M, N, K, L, *schedule,
                                       stream=stream)
    torch.cuda.synchronize()
    assert nv.nvfp4_tensor_wait_timeouts(reset=True) == 0, "a pipeline wait ran out"
    whole = buf.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.all(whole[:pad] == SENTINEL_BITS) and np.all(whole[pad + n_out:] == SENTINEL_BITS), \
        "write outside c"
    return whole[pad:pad + n_out].reshape(L, N, M)


def check(M, N, K, L, seed, schedule=None, alpha=1.0, with_bias=False, b_pad_rows=0,
          activation=0):
    p = synthetic.make_gemm_problem(M, N, K, L, seed=seed)
    bias = None
    if with_bias:
        rng = np.random.default_rng(seed)
        bias = (rng.standard_normal((L, N, M)) * 4).astype(np.float16).view(np.uint16)
    ref, vals, tol = oracle.gemm_small_n(p["a"], p["b"], p["sfa"], p["sfb"], M, N, K, L,
                                         alpha=alpha, bias=bias, activation=activation)
    got = run_gemm(p, M, N, K, L, schedule, alpha, bias, b_pad_rows, activation)
    parity.assert_parity(got, ref, vals, tol, f"gemm M={M} N={N} K={K} L={L} {schedule}")
    return got


# (M, N, K, L): every column count the kernel instantiates (1, 2, 4, 8, 16
# read back), N not a power of two, ragged M, a partial last K stage
GEMM_SHAPES = [
    (128, 2, 256, 1), (200, 3, 1088, 2), (1, 5, 64, 1), (333, 8, 2304, 2), (129, 16, 512, 3),
    (1000, 7, 4096, 2), (640, 12, 768, 5), (64, 16, 16384, 1),
]


@pytest.mark.parametrize("M,N,K,L", GEMM_SHAPES)
def test_gemm_default_schedule(M, N, K, L):
    check(M, N, K, L, seed=M + N + K)


@pytest.mark.parametrize("stages", [2, 4])
@pytest.mark.parametrize("ks", [1, 2, 4, 8])
@pytest.mark.parametrize("N", [1, 3, 16])
def test_gemm_every_schedule(stages, ks, N):
    M, K, L = 300, 2560, 3  # 10 K stages: uneven splits rotate between tiles
    outs = []
    for ctas in (ks, 3 * ks, 64 * ks):  # 1 and 3 persistent clusters, more clusters than tiles
        outs.append(check(M, N, K, L, seed=7 * N + ks, schedule=(stages, ks, ctas)))
    # the summation order depends only on the cluster size, not on the grid
    assert all(np.array_equal(outs[0], o) for o in outs[1:])


def test_gemm_with_one_vector_uses_the_gemv():
    # N = 1 through the automatic entry is the CUDA-core GEMV on permuted scales
    M, K, L = 7168, 2048, 4
    p = synthetic.make_gemm_problem(M, 1, K, L, seed=0)
    got = check(M, 1, K, L, seed=0)
    ref = torch.full((L * M,), SENTINEL, dtype=torch.float16, device=DEV)
    # keep every input referenced until the call has run
    a, b = to_dev(p["a"]), to_dev(p["b"])
    sfa, sfb = nv.repack_scales(to_dev(p["sfa"])), nv.repack_scales(to_dev(p["sfb"]))
    nv.nvfp4_gemv(a.data_ptr(), b.data_ptr(), sfa.data_ptr(), sfb.data_ptr(), ref.data_ptr(),
                  M, K, L, nv.SF_PERMUTED_128x4, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert np.array_equal(got[:, 0, :], ref.cpu().view(torch.int16).numpy().view(np.uint16)
                          .reshape(L, M))


def test_gemm_alpha_bias_and_padded_b():
    check(517, 6, 1344, 3, seed=11, alpha=-0.75, with_bias=True, b_pad_rows=5)
    check(517, 1, 1344, 3, seed=12, alpha=2.0, with_bias=True, b_pad_rows=3)


@pytest.mark.parametrize("activation", [nv.ACT_RELU, nv.ACT_SILU, nv.ACT_GELU_TANH,
                                        nv.ACT_GELU_ERF])
@pytest.mark.parametrize("N", [1, 5, 16])
def test_gemm_activation(activation, N):
    """alpha scales the sums to about unit spread and the bias (4 sigma)
    shifts them, so outputs fall on both sides of each activation's knee."""
    M, K, L = 300, 1024, 2
    got = check(M, N, K, L, seed=N + 10 * activation, alpha=0.0625, with_bias=True,
                activation=activation)
    vals = got.view(np.float16).astype(np.float64)
    assert (vals > 0).any() and ((vals < 0).any() or activation == nv.ACT_RELU)


def test_gemm_zero_k_gives_bias_or_zeros():
    M, N, L = 70, 4, 2
    got = check(M, N, 0, L, seed=1, with_bias=True)
    assert got.shape == (L, N, M)
    zeros = run_gemm(synthetic.make_gemm_problem(M, N, 0, L), M, N, 0, L)
    assert np.all((zeros == 0) | (zeros == 0x8000))


def test_gemm_is_deterministic():
    first = check(1000, 8, 4096, 2, seed=5)
    again = run_gemm(synthetic.make_gemm_problem(1000, 8, 4096, 2, seed=5), 1000, 8, 4096, 2)
    assert np.array_equal(first, again)


@pytest.mark.parametrize("name", ["M7168_N8_K2048_L4", "M7168_N16_K16384_L1"])
def test_gemm_full_size(name):
    _, M, N, K, L = next(w for w in synthetic.GEMM_WORKLOADS if w[0] == name)
    check(M, N, K, L, seed=0)


FINITE_E4M3 = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)


@pytest.mark.parametrize("M,N,K,L,schedule", [(300, 2, 1024, 3, None), (257, 16, 2304, 2, None),
                                              (129, 5, 4096, 1, (4, 4, 8))])
def test_gemm_every_e4m3_scale_code(M, N, K, L, schedule):
    """sfa and every vector's sfb from all 254 finite E4M3 codes (negative,
    -0, subnormal, 448), plus NaN codes on one row and one vector: negative
    codes are folded into the operands' sign bits before the MMA."""
    rng = np.random.default_rng(M * N)
    p = {"a": rng.integers(0, 256, (L, M, K // 2), dtype=np.uint8),
         "b": rng.integers(0, 256, (L, N, K // 2), dtype=np.uint8),
         "sfa": rng.choice(FINITE_E4M3, (L, M, K // 16)),
         "sfb": rng.choice(FINITE_E4M3, (L, N, K // 16))}
    p["sfa"][0, 9, 3] = 0x7F       # one row NaN for every vector
    p["sfb"][L - 1, 1, 20] = 0xFF  # one vector NaN for every row
    ref, vals, tol = oracle.gemm_small_n(p["a"], p["b"], p["sfa"], p["sfb"], M, N, K, L)
    got = run_gemm(p, M, N, K, L, schedule)
    parity.assert_parity(got, ref, vals, tol, f"gemm all E4M3 codes M={M} N={N} K={K} L={L}")
    v = parity.half_values(got)
    assert np.isnan(v[0, :, 9]).all() and np.isnan(v[L - 1, 1, :]).all()
    # a negative scale on one vector only: that vector's outputs change sign
    q = dict(p, sfb=p["sfb"].copy())
    q["sfb"][:, 0, :] ^= 0x80
    flipped = parity.half_values(run_gemm(q, M, N, K, L, schedule))
    assert np.array_equal(flipped[:, 1:, :], v[:, 1:, :], equal_nan=True)
    base, neg = v[:, 0, :], flipped[:, 0, :]
    fin = np.isfinite(base)
    assert np.array_equal(np.isnan(neg), np.isnan(base)) and np.array_equal(neg[fin], -base[fin])
