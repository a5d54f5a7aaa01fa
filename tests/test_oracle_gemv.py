"""Pins for the oracle's GEMV (CPU only).

Hand-worked values (tests/golden/hand_dots.json), an exact fractions.Fraction
brute force with its own decoding (format value set + torch's float8
conversion), the oracle's second (exact int64) path, special cases that
reduce to a numpy matmul, and sign / scale invariants.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from nvfp4_block_scaled_gemv_gb300 import synthetic

E2M1_MAG = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3),
            Fraction(4), Fraction(6)]


def _e2m1_fraction(code):
    v = E2M1_MAG[code & 7]
    return -v if code & 8 else v


_E4M3_TORCH = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)


def _e4m3_fraction(code):
    v = float(_E4M3_TORCH[code])
    return None if math.isnan(v) else Fraction(v)


def _half_value(bits):
    return float(np.array([bits], dtype=np.uint16).view(np.float16)[0])


def brute_force(a, b, sfa, sfb, M, K, L):
    """Exact sum per output with Fractions, rounded to fp16 by numpy."""
    out = np.zeros((L, M), dtype=np.uint16)
    for l in range(L):
        for m in range(M):
            total = Fraction(0)
            nan = False
            for k in range(K):
                abyte = int(a[l, m, k // 2])
                bbyte = int(b[l, k // 2])
                acode = (abyte >> 4) if k % 2 else (abyte & 15)
                bcode = (bbyte >> 4) if k % 2 else (bbyte & 15)
                sa = _e4m3_fraction(int(sfa[l, m, k // 16]))
                sb = _e4m3_fraction(int(sfb[l, k // 16]))
                if sa is None or sb is None:
                    nan = True
                    continue
                total += _e2m1_fraction(acode) * sa * _e2m1_fraction(bcode) * sb
            if nan:
                out[l, m] = 0x7E00
                continue
            x = float(total)
            assert Fraction(x) == total, "brute-force sum not exact in a double"
            with np.errstate(over="ignore"):
                out[l, m] = np.array([x]).astype(np.float16).view(np.uint16)[0]
    return out


def _same_values(c1, c2):
    """Equal fp16 bit patterns, except that any NaN equals any NaN and +0 equals -0."""
    v1 = c1.view(np.float16).astype(np.float64)
    v2 = c2.view(np.float16).astype(np.float64)
    n1, n2 = np.isnan(v1), np.isnan(v2)
    return np.array_equal(n1, n2) and np.array_equal(v1[~n1], v2[~n2])


def _load_golden(golden_dir):
    with open(os.path.join(golden_dir, "hand_dots.json")) as f:
        return json.load(f)["cases"]


def test_hand_worked_dots(golden_dir):
    for case in _load_golden(golden_dir):
        a = np.frombuffer(bytes.fromhex(case["a"]), dtype=np.uint8).reshape(1, 1, 32)
        b = np.frombuffer(bytes.fromhex(case["b"]), dtype=np.uint8).reshape(1, 32)
        sfa = np.frombuffer(bytes.fromhex(case["sfa"]), dtype=np.uint8).reshape(1, 1, 4)
        sfb = np.frombuffer(bytes.fromhex(case["sfb"]), dtype=np.uint8).reshape(1, 4)
        expected = float(case["expected"])
        for c in (oracle.gemv(a, b, sfa, sfb, 1, 64, 1)[0], oracle.gemv_exact(a, b, sfa, sfb, 1, 64, 1)[0]):
            got = _half_value(c[0, 0])
            if math.isnan(expected):
                assert math.isnan(got), case["name"]
            else:
                assert got == expected, (case["name"], got, expected)
                if expected == 0.0:
                    assert math.copysign(1.0, got) > 0, case["name"]


def _random_codes(rng, M, K, L):
    a = rng.integers(0, 256, (L, M, K // 2), dtype=np.uint8)
    b = rng.integers(0, 256, (L, K // 2), dtype=np.uint8)
    # scales over every finite code of both signs: subnormals, 448 and -0 included
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    sfa = rng.choice(finite, (L, M, K // 16))
    sfb = rng.choice(finite, (L, K // 16))
    return a, b, sfa, sfb


@pytest.mark.parametrize("M,K,L,seed", [(1, 64, 1, 0), (3, 64, 2, 1), (8, 128, 1, 2),
                                        (5, 128, 3, 3), (2, 192, 1, 4)])
def test_brute_force_fraction_matches_oracle(M, K, L, seed):
    rng = np.random.default_rng(seed)
    a, b, sfa, sfb = _random_codes(rng, M, K, L)
    ref = brute_force(a, b, sfa, sfb, M, K, L)
    c64, _, _ = oracle.gemv(a, b, sfa, sfb, M, K, L)
    cex, _, _ = oracle.gemv_exact(a, b, sfa, sfb, M, K, L)
    assert _same_values(c64, ref)
    assert _same_values(cex, ref)


def test_brute_force_with_nan_and_extreme_scales():
    rng = np.random.default_rng(7)
    M, K, L = 4, 64, 2
    a, b, sfa, sfb = _random_codes(rng, M, K, L)
    sfa[0, 1, 2] = 0x7F
    sfb[1, 0] = 0xFF
    sfa[0, 2, :] = 0x7E
    sfb[0, :] = 0x7E
    a[0, 2, :] = 0x77
    b[0, :] = 0x77
    ref = brute_force(a, b, sfa, sfb, M, K, L)
    c64, _, _ = oracle.gemv(a, b, sfa, sfb, M, K, L)
    cex, _, nan = oracle.gemv_exact(a, b, sfa, sfb, M, K, L)
    assert _same_values(c64, ref) and _same_values(cex, ref)
    assert nan[0, 1] and nan[1].all()
    assert _half_value(c64[0, 2]) == math.inf


@pytest.mark.parametrize("name,M,K,L", [(w[0], min(w[1], 64), min(w[2], 2048), w[3])
                                        for w in synthetic.WORKLOADS[:3]])
def test_exact_path_equals_f64_path_on_benchmark_distributions(name, M, K, L):
    p = synthetic.make_problem(M, K, L, seed=5)
    c64, sums, sumabs = oracle.gemv(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L)
    cex, num, nan = oracle.gemv_exact(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L)
    assert not nan.any()
    assert np.array_equal(c64, cex)
    # the fp64 sum is exact on these distributions: it equals the integer sum
    assert np.array_equal(sums * 2.0 ** 20, num.astype(np.float64))
    assert np.all(sumabs >= np.abs(sums))


def test_unit_scales_reduce_to_plain_fp4_matmul():
    rng = np.random.default_rng(11)
    M, K, L = 16, 256, 2
    a = rng.integers(0, 256, (L, M, K // 2), dtype=np.uint8)
    b = rng.integers(0, 256, (L, K // 2), dtype=np.uint8)
    sfa = np.full((L, M, K // 16), 0x38, dtype=np.uint8)
    sfb = np.full((L, K // 16), 0x38, dtype=np.uint8)
    mag = np.array([float(x) for x in E2M1_MAG] + [-float(x) for x in E2M1_MAG])

    def dec(x):
        lo, hi = x & 15, x >> 4
        return np.stack([mag[lo], mag[hi]], axis=-1).reshape(*x.shape[:-1], -1)

    A, B = dec(a), dec(b)
    want = np.einsum("lmk,lk->lm", A, B)
    c, sums, _ = oracle.gemv(a, b, sfa, sfb, M, K, L)
    assert np.array_equal(sums, want)
    assert np.array_equal(c, want.astype(np.float16).view(np.uint16))


def test_unit_a_gives_scaled_block_sums_of_b():
    p = synthetic.make_problem(8, 128, 2, seed=3)
    M, K, L = 8, 128, 2
    a = np.full((L, M, K // 2), 0x22, dtype=np.uint8)  # every element 1.0
    t8 = oracle.e4m3_table()
    mag = np.array([float(x) for x in E2M1_MAG] + [-float(x) for x in E2M1_MAG])
    bvals = np.stack([mag[p["b"] & 15], mag[p["b"] >> 4]], -1).reshape(L, K)
    block_sums = bvals.reshape(L, K // 16, 16).sum(-1)  # [L, K/16]
    want = np.einsum("lmj,lj->lm", t8[p["sfa"]] * t8[p["sfb"]][:, None, :], block_sums)
    _, sums, _ = oracle.gemv(a, p["b"], p["sfa"], p["sfb"], M, K, L)
    assert np.array_equal(sums, want)


def test_sign_flip_of_b_negates_c():
    M, K, L = 32, 512, 2
    p = synthetic.make_problem(M, K, L, seed=9)
    c, _, _ = oracle.gemv(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L)
    cn, _, _ = oracle.gemv(p["a"], p["b"] ^ 0x88, p["sfa"], p["sfb"], M, K, L)
    v, vn = c.view(np.float16).astype(np.float64), cn.view(np.float16).astype(np.float64)
    assert np.array_equal(vn, -v)


def test_doubling_sfb_doubles_c():
    M, K, L = 32, 512, 2
    p = synthetic.make_problem(M, K, L, seed=10)
    c, _, _ = oracle.gemv(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L)
    c2, _, _ = oracle.gemv(p["a"], p["b"], p["sfa"], p["sfb"] + 8, M, K, L)  # exponent + 1
    v, v2 = c.view(np.float16).astype(np.float64), c2.view(np.float16).astype(np.float64)
    assert np.array_equal(v2, 2 * v)


def test_sampled_outputs_equal_full_gemv():
    M, K, L = 40, 320, 3
    p = synthetic.make_problem(M, K, L, seed=12)
    c, s, sa = oracle.gemv(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L)
    rng = np.random.default_rng(0)
    mi = rng.integers(0, M, 50)
    li = rng.integers(0, L, 50)
    cs, ss, sas = oracle.gemv_at(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L, mi, li)
    assert np.array_equal(cs, c[li, mi]) and np.array_equal(ss, s[li, mi])
    assert np.array_equal(sas, sa[li, mi])


def test_empty_and_zero_k():
    c, _, _ = oracle.gemv(np.zeros(0, np.uint8), np.zeros(0, np.uint8), np.zeros(0, np.uint8),
                          np.zeros(0, np.uint8), 4, 0, 2)
    assert c.shape == (2, 4) and np.all(c == 0)
    c, _, _ = oracle.gemv(np.zeros(0, np.uint8), np.zeros(64, np.uint8), np.zeros(0, np.uint8),
                          np.zeros(8, np.uint8), 0, 128, 1)
    assert c.shape == (1, 0)


# --- output scale and bias (nvfp4_gemv_ex) -----------------------------------

def fraction_to_fp16_bits(q: Fraction) -> int:
    """binary16 bits of an exact rational, round to nearest even (IEEE 754:
    5 exponent bits, bias 15, 10 mantissa bits, subnormals, overflow to inf)."""
    sign = 0x8000 if q < 0 else 0
    q = abs(q)
    if q == 0:
        return sign
    # e = floor(log2 q), no smaller than the subnormal exponent -14
    e = q.numerator.bit_length() - q.denominator.bit_length()
    if Fraction(2) ** e > q:
        e -= 1
    e = max(e, -14)
    ulp = Fraction(2) ** (e - 10)
    n_floor = q // ulp
    rem = q - n_floor * ulp
    n = n_floor + (1 if rem * 2 > ulp or (rem * 2 == ulp and n_floor % 2 == 1) else 0)
    if n == 2048:  # rounded up to the next binade
        n, e = 1024, e + 1
    if e > 15:
        return sign | 0x7C00
    if n < 1024:  # subnormal (e == -14)
        return sign | int(n)
    return sign | ((e + 15) << 10) | int(n - 1024)


def test_fraction_rounding_helper_matches_numpy_on_doubles():
    rng = np.random.default_rng(5)
    xs = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-9, 6, 2000),
                         [65504.0, 65519.99, 65520.0, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26]])
    for x in xs:
        want = int(np.array([x]).astype(np.float16).view(np.uint16)[0])
        assert fraction_to_fp16_bits(Fraction(float(x))) == want, x


def test_gemv_ex_defaults_equal_gemv():
    M, K, L = 24, 384, 3
    p = synthetic.make_problem(M, K, L, seed=21)
    c, s, sa = oracle.gemv(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L)
    ce, y, sae = oracle.gemv_ex(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L)
    assert np.array_equal(ce, c) and np.array_equal(y, s) and np.array_equal(sae, sa)


@pytest.mark.parametrize("alpha,shift", [(2.0, 8), (0.5, -8)])
def test_gemv_ex_power_of_two_alpha_equals_scale_exponent_change(alpha, shift):
    """alpha = 2**e scales like moving every sfb exponent by e (codes +-8)."""
    M, K, L = 32, 512, 2
    p = synthetic.make_problem(M, K, L, seed=22)
    ce, _, _ = oracle.gemv_ex(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L, alpha=alpha)
    c2, _, _ = oracle.gemv(p["a"], p["b"], p["sfa"], (p["sfb"].astype(np.int32) + shift).astype(np.uint8),
                           M, K, L)
    assert np.array_equal(ce, c2)


def test_gemv_ex_brute_force_with_alpha_and_bias():
    rng = np.random.default_rng(23)
    for case, alpha in enumerate([0.375, -1.25, 5.0, np.float32(0.3), np.float32(-7.1e-3)]):
        M, K, L = int(rng.integers(1, 7)), 64 * int(rng.integers(1, 3)), int(rng.integers(1, 3))
        p = synthetic.make_problem(M, K, L, seed=300 + case)
        bias = (rng.standard_normal((L, M)) * 4).astype(np.float16).view(np.uint16)
        ce, _, _ = oracle.gemv_ex(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L,
                                  alpha=float(alpha), bias=bias)
        for l in range(L):
            for m in range(M):
                total = Fraction(0)
                for k in range(K):
                    abyte, bbyte = int(p["a"][l, m, k // 2]), int(p["b"][l, k // 2])
                    acode = (abyte >> 4) if k % 2 else (abyte & 15)
                    bcode = (bbyte >> 4) if k % 2 else (bbyte & 15)
                    total += (_e2m1_fraction(acode) * _e4m3_fraction(int(p["sfa"][l, m, k // 16]))
                              * _e2m1_fraction(bcode) * _e4m3_fraction(int(p["sfb"][l, k // 16])))
                y = Fraction(float(alpha)) * total + Fraction(_half_value(int(bias[l, m])))
                assert int(ce[l, m]) == fraction_to_fp16_bits(y), (case, l, m)


def test_gemm_small_n_brute_force():
    """Every (l, n, m) of the small-N GEMM against an exact Fraction sum over
    b's row n, with an output scale and a bias."""
    rng = np.random.default_rng(41)
    for case in range(4):
        M, N = int(rng.integers(1, 5)), int(rng.integers(2, 5))
        K, L = 64 * int(rng.integers(1, 3)), int(rng.integers(1, 3))
        a = rng.integers(0, 256, (L, M, K // 2), dtype=np.uint8)
        b = rng.integers(0, 256, (L, N, K // 2), dtype=np.uint8)
        sfa = (0x18 + rng.integers(0, 25, (L, M, K // 16))).astype(np.uint8)
        sfb = (0x18 + rng.integers(0, 25, (L, N, K // 16))).astype(np.uint8)
        alpha = [1.0, 0.75, -2.5, 0.1][case]
        bias = None if case == 0 else (rng.standard_normal((L, N, M)) * 3).astype(
            np.float16).view(np.uint16)
        c, _, _ = oracle.gemm_small_n(a, b, sfa, sfb, M, N, K, L, alpha=alpha, bias=bias)
        assert c.shape == (L, N, M)
        for l in range(L):
            for n in range(N):
                for m in range(M):
                    total = Fraction(0)
                    for k in range(K):
                        abyte, bbyte = int(a[l, m, k // 2]), int(b[l, n, k // 2])
                        acode = (abyte >> 4) if k % 2 else (abyte & 15)
                        bcode = (bbyte >> 4) if k % 2 else (bbyte & 15)
                        total += (_e2m1_fraction(acode) * _e4m3_fraction(int(sfa[l, m, k // 16]))
                                  * _e2m1_fraction(bcode) * _e4m3_fraction(int(sfb[l, n, k // 16])))
                    y = Fraction(float(alpha)) * total
                    if bias is not None:
                        y += Fraction(_half_value(int(bias[l, n, m])))
                    assert int(c[l, n, m]) == fraction_to_fp16_bits(y), (case, l, n, m)


def test_gemm_small_n_with_one_vector_is_the_gemv():
    M, K, L = 37, 320, 3
    p = synthetic.make_problem(M, K, L, seed=8)
    c, _, _ = oracle.gemm_small_n(p["a"], p["b"].reshape(L, 1, K // 2), p["sfa"],
                                  p["sfb"].reshape(L, 1, K // 16), M, 1, K, L)
    ref, _, _ = oracle.gemv(p["a"], p["b"], p["sfa"], p["sfb"], M, K, L)
    assert np.array_equal(c[:, 0, :], ref)


def test_gemm_small_n_permuting_vectors_permutes_columns():
    rng = np.random.default_rng(3)
    M, N, K, L = 9, 5, 128, 2
    a = rng.integers(0, 256, (L, M, K // 2), dtype=np.uint8)
    b = rng.integers(0, 256, (L, N, K // 2), dtype=np.uint8)
    sfa = (0x18 + rng.integers(0, 25, (L, M, K // 16))).astype(np.uint8)
    sfb = (0x18 + rng.integers(0, 25, (L, N, K // 16))).astype(np.uint8)
    perm = rng.permutation(N)
    c, _, _ = oracle.gemm_small_n(a, b, sfa, sfb, M, N, K, L)
    cp, _, _ = oracle.gemm_small_n(a, b[:, perm], sfa, sfb[:, perm], M, N, K, L)
    assert np.array_equal(cp, c[:, perm])
