"""Full-size parity where fp32 accumulation rounds.

With the benchmark's scale codes (values in [1/16, 1/2]) every partial sum
is a multiple of 2^-16 below 2^8, so fp32 accumulation is exact in any order
and full-size comparisons never exercise the tolerance.  Here the scale codes
run over 0x01..0x50 (values 2^-9, subnormal, up to 8): a block term is a
multiple of 2^-20 and partial sums reach 10^4, so they need about 34
significant bits and each kernel's fp32 summation order rounds differently.
(Codes up to 448 would overflow fp16 in nearly every output: |c| ~ 10^7.)
Every kernel and layout is compared on sampled outputs (random rows plus the
first, last and atom-boundary rows of every batch) against the oracle,
|gpu - oracle| <= 1e-3 * sum|terms| + 1 fp16 ulp; the largest
|gpu - oracle| / tolerance is printed, and reported in the assertion message.
A second launch of each must repeat every output bit for bit.
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
WIDE_SCALES = (0x01, 0x50)  # E4M3 codes 0x01..0x50: 2^-9 .. 8


@pytest.fixture(scope="module", autouse=True)
def _lib():
    libbuild.build()
    nv.library()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    nv.nvfp4_tensor_wait_timeouts(reset=True)


def _samples(M, L, n, rng):
    rows = [0, 1, 31, 32, 127, 128, 129, M // 2, M - 129, M - 128, M - 1]
    mi = np.concatenate([rng.integers(0, M, n), np.tile(rows, L)])
    li = np.concatenate([rng.integers(0, L, n), np.repeat(np.arange(L), len(rows))])
    return mi, li


def _runs(M, K, L, layout):
    """(label, kernel, lanes_per_row, k_split, ctas) of every kernel that runs
    the shape and layout: the library's own choice, then each kernel's plan."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    out = [("default", None)]
    kernels = [nv.KERNEL_PIPELINED, nv.KERNEL_BLOCKDOT, nv.KERNEL_BLOCKWISE]
    if layout == nv.SF_PERMUTED_128x4 or K % 256 == 0:
        kernels.append(nv.KERNEL_TENSOR)
    for k in kernels:
        plan = nv.nvfp4_gemv_plan(M, K, L, layout, sms, 0, kernel=k)
        out.append((["direct", "pipelined", "tensor", "blockdot", "blockwise"][k],
                    (k, plan["lanes_per_row"], plan["k_split"], plan["ctas"])))
    return out


@pytest.mark.parametrize("name,M,K,L,layout", [
    ("M7168_K16384_L1", 7168, 16384, 1, nv.SF_PLAIN),
    ("M7168_K16384_L1", 7168, 16384, 1, nv.SF_PERMUTED_128x4),
    ("M16384_K8192_L16", 16384, 8192, 16, nv.SF_PLAIN),
    ("M16384_K8192_L16", 16384, 8192, 16, nv.SF_PERMUTED_128x4),
])
def test_full_size_with_rounding(name, M, K, L, layout):
    p = synthetic.make_problem(M, K, L, seed=9, scale_codes=WIDE_SCALES)
    mi, li = _samples(M, L, 3000, np.random.default_rng(4))
    ref, sums, sumabs = oracle.gemv_at(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L, mi, li)
    a, b = torch.from_numpy(p["a"]).to(DEV), torch.from_numpy(p["b"]).to(DEV)
    sfa, sfb = torch.from_numpy(p["sfa"]).to(DEV), torch.from_numpy(p["sfb"]).to(DEV)
    if layout == nv.SF_PERMUTED_128x4:
        sfa, sfb = nv.repack_scales(sfa), nv.repack_scales(sfb.view(L, 1, K // 16))
    c = torch.empty(L * M, dtype=torch.float16, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream
    report = []
    def launch(sched):
        c.fill_(0)
        if sched is None:
            nv.nvfp4_gemv(a.data_ptr(), b.data_ptr(), sfa.data_ptr(), sfb.data_ptr(), c.data_ptr(),
                          M, K, L, layout, stream)
        else:
            nv.nvfp4_gemv_explicit(a.data_ptr(), b.data_ptr(), sfa.data_ptr(), sfb.data_ptr(),
                                   c.data_ptr(), M, K, L, layout, *sched, stream=stream)
        torch.cuda.synchronize()
        assert nv.nvfp4_tensor_wait_timeouts(reset=True) == 0, "a pipeline wait ran out"
        return c.cpu().view(torch.int16).numpy().view(np.uint16).reshape(L, M)

    for label, sched in _runs(M, K, L, layout):
        whole = launch(sched)
        # run to run, every output's bits repeat (the summation order is fixed
        # by the schedule, and here the order decides the rounding)
        assert np.array_equal(whole, launch(sched)), f"{name} layout={layout} {label}: not reproducible"
        got = whole[li, mi]
        ok, tol, diff = parity.compare(got, ref, sums, sumabs)
        fin = np.isfinite(diff)
        worst = float(np.max(diff[fin] / tol[fin]))
        differs = int(np.sum(got != ref))
        report.append(f"{label}: max |d|/tol {worst:.3g}, {differs} of {got.size} differ from "
                      "the correctly rounded value")
        assert ok.all(), f"{name} layout={layout} {label}: {int((~ok).sum())} outputs fail; " + \
            "; ".join(report)
    print(f"{name} layout={layout}: " + "; ".join(report))
