"""The seeded input generator (shared by the oracle side and the CUDA side)."""
import numpy as np

from nvfp4_block_scaled_gemv_gb300 import synthetic


def test_splitmix64_published_vector():
    # splitmix64 seeded with 0: the first outputs quoted with the generator's definition
    assert [int(x) for x in synthetic.splitmix64(0, 3)] == [
        0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_counter_based_offsets_agree():
    full = synthetic.splitmix64(123, 1000)
    assert np.array_equal(synthetic.splitmix64(123, 400, start=600), full[600:])


def test_problem_shapes_and_distributions():
    p = synthetic.make_problem(256, 1024, 3, seed=0)
    assert p["a"].shape == (3, 256, 512) and p["b"].shape == (3, 512)
    assert p["sfa"].shape == (3, 256, 64) and p["sfb"].shape == (3, 64)
    nib = np.concatenate([p["a"].reshape(-1) & 15, p["a"].reshape(-1) >> 4])
    counts = np.bincount(nib, minlength=16)
    assert counts.min() > 0.9 * counts.mean()  # every E2M1 code, -0 included
    codes = np.unique(p["sfa"])
    assert codes.min() == 0x18 and codes.max() == 0x30 and codes.size == 25
    again = synthetic.make_problem(256, 1024, 3, seed=0)
    assert all(np.array_equal(p[k], again[k]) for k in p)
    other = synthetic.make_problem(256, 1024, 3, seed=1)
    assert not np.array_equal(p["a"], other["a"])


def test_algorithmic_bytes_of_the_workloads():
    want = [18832, 33092096, 132218368, 66083840, 1208557568]
    got = [synthetic.algorithmic_bytes(M, K, L) for _, M, K, L in synthetic.WORKLOADS]
    assert got == want
