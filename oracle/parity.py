"""Parity rule between a GPU result and the oracle: TEST INFRASTRUCTURE ONLY.

A GPU output g matches the oracle output o (both fp16) when

    |g - o| <= 1e-3 * sum_k |term_k| + ulp16(o)

where sum |term_k| is the oracle's fp64 sum of absolute products for that
output and ulp16(o) the spacing of fp16 numbers at o.  NaN must meet NaN.
An infinite result on either side is accepted only when the oracle's exact
sum lies within the same tolerance of the fp16 overflow threshold (65520),
with the same sign.
"""
from __future__ import annotations

import numpy as np

REL_TOL = 1e-3
FP16_OVERFLOW = 65520.0


def half_values(bits) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def ulp16(x) -> np.ndarray:
    """Spacing of binary16 numbers at |x| (2^-24 in the subnormal range)."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    out = np.full(ax.shape, 2.0 ** -24)
    normal = np.isfinite(ax) & (ax >= 2.0 ** -14)
    e = np.floor(np.log2(ax[normal]))
    out[normal] = np.exp2(e - 10)
    return out


def compare(gpu_bits, ref_bits, ref_sums, ref_sumabs):
    """Elementwise parity; returns (ok_mask, tolerance, abs_diff)."""
    g = half_values(gpu_bits)
    o = half_values(ref_bits)
    s = np.asarray(ref_sums, dtype=np.float64)
    a = np.asarray(ref_sumabs, dtype=np.float64)
    tol = REL_TOL * np.nan_to_num(a, nan=0.0, posinf=np.inf) + ulp16(np.where(np.isfinite(o), o, 0.0))
    diff = np.abs(g - o)
    ok = np.zeros(g.shape, dtype=bool)
    gn, on = np.isnan(g), np.isnan(o)
    ok |= gn & on
    fin = np.isfinite(g) & np.isfinite(o)
    ok |= fin & (diff <= tol)
    # overflow boundary: either side infinite, the other side not NaN
    inf_case = ~gn & ~on & ~fin
    near = np.abs(s) + REL_TOL * np.nan_to_num(a, nan=0.0) >= FP16_OVERFLOW
    same_sign = np.sign(g) == np.sign(s)
    ok |= inf_case & near & same_sign & (np.isinf(g) | (np.abs(g) >= 65504.0 - tol))
    return ok, tol, diff


def assert_parity(gpu_bits, ref_bits, ref_sums, ref_sumabs, what: str = "") -> None:
    ok, tol, diff = compare(gpu_bits, ref_bits, ref_sums, ref_sumabs)
    if not ok.all():
        bad = np.argwhere(~ok.reshape(ok.shape))
        first = [tuple(int(i) for i in b) for b in bad[:5]]
        g = half_values(gpu_bits).reshape(ok.shape)
        o = half_values(ref_bits).reshape(ok.shape)
        details = ", ".join(f"{idx}: gpu={g[idx]!r} oracle={o[idx]!r} tol={tol.reshape(ok.shape)[idx]:.3g}"
                            for idx in first)
        raise AssertionError(f"parity failed {what}: {int((~ok).sum())}/{ok.size} outputs; {details}")
