"""GPU parity of the block-dot kernel (NVFP4_KERNEL_BLOCKDOT) against the CPU oracle.

The kernel computes every 16-element block dot on the tensor cores (an MMA
whose A scales are 1.0 and whose B scales select one block per accumulator
column) and applies the E4M3 scales on the CUDA cores, so signed, subnormal,
maximal and NaN scale codes must all follow the oracle's signed E4M3 reading.  Every launch is checked for writes
outside c (sentinel slack) and for bounded pipeline waits that ran out.
Tolerance: |gpu - oracle| <= 1e-3 * sum|terms| + 1 fp16 ulp of the oracle value.
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
LAYOUTS = [nv.SF_PLAIN, nv.SF_PERMUTED_128x4]
FINITE_E4M3 = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    libbuild.build()
    nv.library()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    nv.nvfp4_tensor_wait_timeouts(reset=True)


def to_dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(DEV)


def device_inputs(p, M, K, L, layout):
    a, b = to_dev(p["a"]), to_dev(p["b"])
    if layout == nv.SF_PLAIN:
        return a, b, to_dev(p["sfa"]), to_dev(p["sfb"])
    return (a, b, to_dev(oracle.repack_scales(p["sfa"], M, K, L)),
            to_dev(oracle.repack_scales(np.asarray(p["sfb"]).reshape(L, 1, K // 16), 1, K, L)))


def run_bd(p, M, K, L, layout, stages=0, ctas=None):
    """One block-dot launch (ring slots `stages`, 0 = the most that fit; `ctas`
    CTAs, default one per 8-row unit up to 152); returns c's fp16 bits [L, M]."""
    a, b, sfa, sfb = device_inputs(p, M, K, L, layout)
    pad = 64
    buf = torch.full((L * M + 2 * pad,), SENTINEL, dtype=torch.float16, device=DEV)
    c = buf[pad:pad + L * M]
    stream = torch.cuda.current_stream().cuda_stream
    if ctas is None:
        ctas = min(152, L * -(-M // 8))
    nv.nvfp4_gemv_explicit(a.data_ptr(), b.data_ptr(), sfa.data_ptr(), sfb.data_ptr(),
                           c.data_ptr(), M, K, L, layout, nv.KERNEL_BLOCKDOT, stages, 1, ctas,
                           stream)
    torch.cuda.synchronize()
    assert nv.nvfp4_tensor_wait_timeouts(reset=True) == 0, "a pipeline wait ran out"
    whole = buf.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.all(whole[:pad] == SENTINEL_BITS) and np.all(whole[pad + L * M:] == SENTINEL_BITS), \
        "write outside c"
    return whole[pad:pad + L * M].reshape(L, M)


def check(p, M, K, L, layout, **kw):
    ref, sums, sumabs = oracle.gemv(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L)
    got = run_bd(p, M, K, L, layout, **kw)
    parity.assert_parity(got, ref, sums, sumabs, f"blockdot M={M} K={K} L={L} layout={layout} {kw}")
    return got


def test_all_ones():
    # a = b = 1.0 (E2M1 code 2), every scale 1.0 (E4M3 0x38): c = K exactly
    M, K, L = 128, 256, 1
    p = {"a": np.full((L, M, K // 2), 0x22, np.uint8), "b": np.full((L, K // 2), 0x22, np.uint8),
         "sfa": np.full((L, M, K // 16), 0x38, np.uint8),
         "sfb": np.full((L, K // 16), 0x38, np.uint8)}
    for layout in LAYOUTS:
        got = run_bd(p, M, K, L, layout, stages=2, ctas=1)
        assert np.all(got.view(np.float16) == K)


def test_one_block_at_a_time():
    """Row m carries a nonzero scale on block m % 16 only: c names that block,
    so a block routed to the wrong accumulator column shows up at once."""
    M, K, L = 256, 256, 1
    rng = np.random.default_rng(3)
    p = {"a": rng.integers(0, 256, (L, M, K // 2), dtype=np.uint8),
         "b": rng.integers(0, 256, (L, K // 2), dtype=np.uint8),
         "sfa": np.zeros((L, M, K // 16), np.uint8), "sfb": np.full((L, K // 16), 0x38, np.uint8)}
    p["sfa"][0, np.arange(M), np.arange(M) % 16] = 0x38
    for layout in LAYOUTS:
        check(p, M, K, L, layout, stages=3, ctas=2)


# (M, K, L): ragged M and batches, one 8-row unit, partial last K stage of
# 1..3 chunks (pre-permuted only: plain scales need K % 256 == 0), long K,
# many batches, tiles cut at batch and atom-block ends
BD_SHAPES = [
    (1, 256, 1), (7, 512, 3), (8, 256, 1), (9, 768, 2), (127, 2048, 1), (128, 256, 1),
    (129, 1024, 2), (200, 7168, 1), (333, 16384, 1), (1000, 4096, 3), (513, 2304, 2),
    (2, 2048, 300), (4096, 1024, 2), (37, 8192, 5), (1, 64, 1), (7, 192, 3), (129, 320, 2),
    (200, 1088, 3), (640, 448, 5),
]


@pytest.mark.parametrize("M,K,L", BD_SHAPES)
def test_parity_block_dot_kernel(M, K, L):
    p = synthetic.make_problem(M, K, L, seed=M + K + L)
    outs = []
    for layout in LAYOUTS:
        if layout == nv.SF_PLAIN and K % 256:
            continue
        for stages, ctas in ((0, None), (2, 1), (3, 5), (5, 37)):
            units = L * -(-M // 8)
            if ctas is not None and ctas > units:
                continue
            outs.append(check(p, M, K, L, layout, stages=stages, ctas=ctas))
    # every row is summed block by block in K order: grid, ring depth and
    # scale layout change no bit
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


@pytest.mark.parametrize("layout", LAYOUTS)
def test_every_e4m3_scale_code(layout):
    """sfa and sfb drawn from all 254 finite E4M3 codes (negative, -0,
    subnormal, 448), plus NaN codes 0x7F and 0xFF on some rows and batches."""
    M, K, L = 300, 1024, 3
    rng = np.random.default_rng(11)
    p = {"a": rng.integers(0, 256, (L, M, K // 2), dtype=np.uint8),
         "b": rng.integers(0, 256, (L, K // 2), dtype=np.uint8),
         "sfa": rng.choice(FINITE_E4M3, (L, M, K // 16)),
         "sfb": rng.choice(FINITE_E4M3, (L, K // 16))}
    p["sfa"][0, 5, 7] = 0x7F
    p["sfa"][2, 77, 60] = 0xFF
    p["sfb"][1, 33] = 0xFF
    ref, sums, sumabs = oracle.gemv(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L)
    got = run_bd(p, M, K, L, layout, stages=4, ctas=19)
    parity.assert_parity(got, ref, sums, sumabs, f"all E4M3 codes layout={layout}")
    v = parity.half_values(got)
    assert np.isnan(v[0, 5]) and np.isnan(v[2, 77]) and np.isnan(v[1]).all()
    assert (np.signbit(v[np.isfinite(v)])).any()  # negative scales do reach c


@pytest.mark.parametrize("layout", LAYOUTS)
def test_each_scale_code_alone(layout):
    """Row m: a = b = 1.0, sfb = 1.0, sfa code m on block 0 and zero elsewhere,
    so c[m] = 16 * E4M3(m) exactly; then the same for sfb codes across batches."""
    K = 256
    M, L = 256, 1
    p = {"a": np.full((L, M, K // 2), 0x22, np.uint8), "b": np.full((L, K // 2), 0x22, np.uint8),
         "sfa": np.zeros((L, M, K // 16), np.uint8), "sfb": np.full((L, K // 16), 0x38, np.uint8)}
    p["sfa"][0, :, 0] = np.arange(256, dtype=np.uint8)
    table = oracle.e4m3_table()
    got = parity.half_values(run_bd(p, M, K, L, layout, stages=2, ctas=4))[0]
    want = 16.0 * table
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan) and np.array_equal(got[~nan], want[~nan])
    M, L = 8, 256
    p = {"a": np.full((L, M, K // 2), 0x22, np.uint8), "b": np.full((L, K // 2), 0x22, np.uint8),
         "sfa": np.zeros((L, M, K // 16), np.uint8), "sfb": np.zeros((L, K // 16), np.uint8)}
    p["sfa"][:, :, 0] = 0x38
    p["sfb"][:, 0] = np.arange(256, dtype=np.uint8)
    got = parity.half_values(run_bd(p, M, K, L, layout, stages=3, ctas=50))[:, 3]
    assert np.array_equal(np.isnan(got), nan) and np.array_equal(got[~nan], want[~nan])


def test_sign_flip_and_scale_doubling_are_exact():
    M, K, L = 300, 4096, 2
    p = synthetic.make_problem(M, K, L, seed=21)
    base = parity.half_values(run_bd(p, M, K, L, nv.SF_PLAIN))
    flipped = dict(p, b=p["b"] ^ 0x88)
    assert np.array_equal(parity.half_values(run_bd(flipped, M, K, L, nv.SF_PLAIN)), -base)
    doubled = dict(p, sfb=p["sfb"] + 8)
    assert np.array_equal(parity.half_values(run_bd(doubled, M, K, L, nv.SF_PLAIN)), 2 * base)
    # a negative sfb code (sign bit set) negates every block it scales
    negated = dict(p, sfb=p["sfb"] | 0x80)
    assert np.array_equal(parity.half_values(run_bd(negated, M, K, L, nv.SF_PERMUTED_128x4)), -base)


def _sample_indices(M, L, n, rng):
    m = [0, M - 1, min(127, M - 1), min(128, M - 1), M // 2, min(7, M - 1), min(8, M - 1)]
    mi = np.concatenate([rng.integers(0, M, n), np.tile(m, L)])
    li = np.concatenate([rng.integers(0, L, n), np.repeat(np.arange(L), len(m))])
    return mi, li


@pytest.mark.parametrize("name,M,K,L", synthetic.WORKLOADS[1:])
def test_full_size_workloads_sampled(name, M, K, L):
    """The benchmark workloads on the block-dot kernel's own plan (one CTA
    per SM, the deepest ring), run twice: identical bits."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    p = synthetic.make_problem(M, K, L, seed=0)
    rng = np.random.default_rng(1)
    mi, li = _sample_indices(M, L, 3000, rng)
    ref, sums, sumabs = oracle.gemv_at(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L, mi, li)
    outs = []
    for layout in LAYOUTS:
        plan = nv.nvfp4_gemv_plan(M, K, L, layout, sms, 0, kernel=nv.KERNEL_BLOCKDOT)
        got = run_bd(p, M, K, L, layout, stages=plan["lanes_per_row"], ctas=plan["ctas"])
        assert np.array_equal(run_bd(p, M, K, L, layout, stages=plan["lanes_per_row"],
                                     ctas=plan["ctas"]), got)
        parity.assert_parity(got[li, mi], ref, sums, sumabs, f"{name} layout={layout}")
        assert np.isfinite(parity.half_values(got)).all()
        outs.append(got)
    assert np.array_equal(outs[0], outs[1])


def test_deterministic_run_to_run():
    M, K, L = 7168, 2048, 4
    p = synthetic.make_problem(M, K, L, seed=3)
    first = run_bd(p, M, K, L, nv.SF_PLAIN)
    for _ in range(2):
        assert np.array_equal(run_bd(p, M, K, L, nv.SF_PLAIN), first)
