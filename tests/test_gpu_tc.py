"""GPU parity of the tensor-core kernel (NVFP4_KERNEL_TENSOR) against the CPU oracle.

Pre-permuted scales, and plain scales when K % 256 == 0 (the kernel lays a
stage's plain scale rows out as atoms in shared memory).  Every launch is checked for
writes outside c (sentinel slack) and for bounded pipeline waits that ran out
(nvfp4_tensor_wait_timeouts must stay 0).  Tolerance as for the CUDA-core
kernels: |gpu - oracle| <= 1e-3 * sum|terms| + 1 fp16 ulp of the oracle value.
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


PERM, PLAIN = nv.SF_PERMUTED_128x4, nv.SF_PLAIN


def run_tc(a, b, sfa_plain, sfb_plain, M, K, L, ks, ctas, stages=4, layout=PERM):
    """One tensor-core launch (stages per CTA, clusters of ks) on oracle-repacked
    scales, or on the plain ones; returns c's fp16 bits [L, M]."""
    if layout == PERM:
        sfa = to_dev(oracle.repack_scales(sfa_plain, M, K, L))
        sfb = to_dev(oracle.repack_scales(np.asarray(sfb_plain).reshape(L, 1, K // 16), 1, K, L))
    else:
        sfa, sfb = to_dev(sfa_plain), to_dev(sfb_plain)
    ad, bd = to_dev(a), to_dev(b)
    pad = 64
    buf = torch.full((L * M + 2 * pad,), SENTINEL, dtype=torch.float16, device=DEV)
    c = buf[pad:pad + L * M]
    nv.nvfp4_gemv_explicit(ad.data_ptr(), bd.data_ptr(), sfa.data_ptr(), sfb.data_ptr(),
                           c.data_ptr(), M, K, L, layout, nv.KERNEL_TENSOR, stages, ks,
                           ctas, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert nv.nvfp4_tensor_wait_timeouts(reset=True) == 0, "a pipeline wait ran out"
    whole = buf.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.all(whole[:pad] == SENTINEL_BITS) and np.all(whole[pad + L * M:] == SENTINEL_BITS), \
        "write outside c"
    return whole[pad:pad + L * M].reshape(L, M)


def check(p, M, K, L, ks, ctas, stages=4, layout=PERM):
    ref, sums, sumabs = oracle.gemv(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L)
    got = run_tc(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L, ks, ctas, stages, layout)
    parity.assert_parity(got, ref, sums, sumabs,
                         f"tensor M={M} K={K} L={L} ks={ks} ctas={ctas} layout={layout}")
    return got


def test_all_ones():
    # a = b = 1.0 (E2M1 code 2), every scale 1.0 (E4M3 0x38): c = K exactly
    M, K, L = 128, 256, 1
    a = np.full((L, M, K // 2), 0x22, np.uint8)
    b = np.full((L, K // 2), 0x22, np.uint8)
    s = np.full((L, M, K // 16), 0x38, np.uint8)
    got = run_tc(a, b, s, s[:, 0, :], M, K, L, 1, 1)
    assert np.all(got.view(np.float16) == K)


def test_row_sums():
    # b = 1.0 and unit scales: c[m] is the plain sum of row m's E2M1 values
    M, K, L = 200, 1088, 2
    rng = np.random.default_rng(7)
    p = {"a": rng.integers(0, 256, (L, M, K // 2), dtype=np.uint8),
         "b": np.full((L, K // 2), 0x22, np.uint8),
         "sfa": np.full((L, M, K // 16), 0x38, np.uint8),
         "sfb": np.full((L, K // 16), 0x38, np.uint8)}
    check(p, M, K, L, 2, 4)


# (M, K, L, k_split, ctas): one CTA; ragged M; a last K stage of 1..3 MMAs;
# clusters of 2, 4 and 8 (split K summed through distributed shared memory);
# fewer clusters than tiles (persistent clusters); a 128-row block per batch
TC_CASES = [
    (128, 256, 1, 1, 1), (1, 64, 1, 1, 1), (7, 192, 3, 1, 2), (256, 512, 2, 1, 2),
    (200, 1088, 3, 1, 3), (129, 320, 2, 2, 2), (256, 2048, 2, 2, 2), (200, 1088, 3, 2, 4),
    (1000, 4096, 2, 4, 8), (333, 16384, 1, 8, 16), (513, 2304, 2, 8, 8), (640, 768, 5, 2, 6),
    (4096, 1024, 1, 4, 152), (128, 16384, 4, 8, 32),
]


@pytest.mark.parametrize("stages", [2, 4])
@pytest.mark.parametrize("M,K,L,ks,ctas", TC_CASES)
def test_parity_tensor_kernel(M, K, L, ks, ctas, stages):
    p = synthetic.make_problem(M, K, L, seed=M + K + ks)
    got = check(p, M, K, L, ks, ctas, stages)
    if K % 256 == 0:
        # plain scales: the same MMAs on the same atoms, so the same bits
        assert np.array_equal(got, check(p, M, K, L, ks, ctas, stages, PLAIN))


def test_plain_scales_ragged_rows_and_stage_counts():
    # plain scale boxes of 128 rows x 16 bytes: rows past M arrive as zeros,
    # and every K % 256 == 0 gives whole stages (odd stage counts included)
    for M, K, L in ((1, 256, 3), (7, 768, 2), (129, 1280, 2), (333, 2816, 1)):
        p = synthetic.make_problem(M, K, L, seed=M * K)
        check(p, M, K, L, 1, 4, 4, PLAIN)
        ks = min(2, K // 256)  # every rank of a cluster needs a K stage
        check(p, M, K, L, ks, 2 * ks, 2, PLAIN)


def test_tensor_kernel_is_deterministic():
    M, K, L = 1000, 4096, 2
    p = synthetic.make_problem(M, K, L, seed=5)
    first = check(p, M, K, L, 4, 8)
    again = run_tc(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L, 4, 8)
    assert np.array_equal(first, again)
    # the rounding depends on the cluster size only: other grids and stage counts agree
    for ctas, stages in ((4, 2), (32, 4), (64, 2)):
        assert np.array_equal(first, run_tc(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L, 4,
                                            ctas, stages))


@pytest.mark.parametrize("name,ks,ctas,stages", [("M7168_K2048_L4", 2, 152, 4),
                                                 ("M7168_K16384_L1", 8, 152, 2),
                                                 ("M4096_K7168_L8", 1, 512, 2)])
def test_tensor_kernel_full_size(name, ks, ctas, stages):
    _, M, K, L = next(w for w in synthetic.WORKLOADS if w[0] == name)
    p = synthetic.make_problem(M, K, L, seed=0)
    got = check(p, M, K, L, ks, ctas, stages)
    assert np.array_equal(got, check(p, M, K, L, ks, ctas, stages, PLAIN))


FINITE_E4M3 = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)


@pytest.mark.parametrize("layout", [PERM, PLAIN])
@pytest.mark.parametrize("M,K,L,ks,ctas,stages", [(300, 1024, 3, 1, 3, 2), (200, 2304, 2, 2, 4, 4),
                                                  (129, 4096, 1, 4, 8, 2)])
def test_every_e4m3_scale_code(M, K, L, ks, ctas, stages, layout):
    """sfa and sfb from all 254 finite E4M3 codes (negative, -0, subnormal,
    448) and NaN codes: the MMA reads codes as unsigned magnitudes, and the
    kernel folds negative codes into the operands' sign bits."""
    rng = np.random.default_rng(M + K)
    p = {"a": rng.integers(0, 256, (L, M, K // 2), dtype=np.uint8),
         "b": rng.integers(0, 256, (L, K // 2), dtype=np.uint8),
         "sfa": rng.choice(FINITE_E4M3, (L, M, K // 16)),
         "sfb": rng.choice(FINITE_E4M3, (L, K // 16))}
    p["sfa"][0, 5, 7] = 0x7F
    p["sfa"][L - 1, 77, 60] = 0xFF
    if L > 1:
        p["sfb"][0, 33] = 0xFF  # every output of batch 0 NaN
    got = check(p, M, K, L, ks, ctas, stages, layout)
    v = parity.half_values(got)
    assert np.isnan(v[0, 5]) and np.isnan(v[L - 1, 77]) and (L == 1 or np.isnan(v[0]).all())
    assert np.signbit(v[np.isfinite(v)]).any()


@pytest.mark.parametrize("layout", [PERM, PLAIN])
def test_each_scale_code_alone(layout):
    """Row m: a = b = 1.0, sfb = 1.0, sfa code m on block 0 and 0 elsewhere:
    c[m] = 16 * E4M3(m) exactly; then every sfb code across batches."""
    K = 256
    table = oracle.e4m3_table()
    want = 16.0 * table
    nan = np.isnan(want)
    M, L = 256, 1
    a = np.full((L, M, K // 2), 0x22, np.uint8)
    b = np.full((L, K // 2), 0x22, np.uint8)
    sfa = np.zeros((L, M, K // 16), np.uint8)
    sfa[0, :, 0] = np.arange(256, dtype=np.uint8)
    sfb = np.full((L, K // 16), 0x38, np.uint8)
    got = parity.half_values(run_tc(a, b, sfa, sfb, M, K, L, 1, 2, 2, layout))[0]
    assert np.array_equal(np.isnan(got), nan) and np.array_equal(got[~nan], want[~nan])
    M, L = 8, 256
    a = np.full((L, M, K // 2), 0x22, np.uint8)
    b = np.full((L, K // 2), 0x22, np.uint8)
    sfa = np.zeros((L, M, K // 16), np.uint8)
    sfa[:, :, 0] = 0x38
    sfb = np.zeros((L, K // 16), np.uint8)
    sfb[:, 0] = np.arange(256, dtype=np.uint8)
    got = parity.half_values(run_tc(a, b, sfa, sfb, M, K, L, 1, 64, 4, layout))[:, 3]
    assert np.array_equal(np.isnan(got), nan) and np.array_equal(got[~nan], want[~nan])


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    # The pipeline barriers' bounded wait, made to run out on purpose in a
    # one-warp kernel (a barrier phase that nothing completes): it must give
    # up after its 2 s limit, count the give-up and return; the next launches
    # then run normally.
    r = nv.nvfp4_selftest_bounded_wait(torch.cuda.current_stream().cuda_stream)
    assert r["completed"] == 1, r
    assert r["gave_up"] == 1, r
    assert r["timeouts"] == 1, r
    assert 1.9e9 <= r["waited_ns"] <= 20e9, r
    assert nv.nvfp4_tensor_wait_timeouts(reset=False) == 0  # its own counter
    p = synthetic.make_problem(300, 512, 2, seed=11)
    check(p, 300, 512, 2, ks=2, ctas=8)
    check(p, 300, 512, 2, ks=1, ctas=3, layout=PLAIN)
