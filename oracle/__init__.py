"""CPU oracle for the NVFP4 block-scaled GEMV: TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The GPU library never does, and the
two share no code.  The arithmetic lives in ``nvfp4_oracle.c`` (plain C,
fp64 and exact-int64 paths); this module only marshals numpy arrays to it.

Definition followed (kernelbot "nvfp4-gemv" submission 103289, ``cute_kernel``
k-tile loop: per element ``a*sfa*b*sfb`` accumulated, stored with
``.to(Float16)``)::

    c[m, l] = fp16( sum_k E2M1(a[m,k,l]) * E4M3(sfa[m,k//16,l])
                         * E2M1(b[k,l])  * E4M3(sfb[k//16,l]) )

Array layouts (numpy, C order): ``a`` uint8 [L, M, K//2], ``b`` uint8
[L, K//2], ``sfa`` uint8 [L, M, K//16], ``sfb`` uint8 [L, K//16]; results are
fp16 bit patterns [L, M] (uint16).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "liboracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    os.makedirs(_LIB_DIR, exist_ok=True)
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
           "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    lib.oracle_e2m1_table.argtypes = [P]
    lib.oracle_e4m3_table.argtypes = [P]
    lib.oracle_fp16_rne.argtypes = [ctypes.c_double]
    lib.oracle_fp16_rne.restype = ctypes.c_uint16
    lib.oracle_fp16_rne_array.argtypes = [P, P, I64]
    lib.oracle_fp16_from_scaled_int.argtypes = [I64]
    lib.oracle_fp16_from_scaled_int.restype = ctypes.c_uint16
    lib.oracle_gemv_f64.argtypes = [P, P, P, P, I64, I64, I64, P, P, P]
    lib.oracle_gemv_f64_at.argtypes = [P, P, P, P, I64, I64, I64, P, P, I64, P, P, P]
    lib.oracle_gemv_exact.argtypes = [P, P, P, P, I64, I64, I64, P, P, P]
    lib.oracle_gemv_exact.restype = ctypes.c_int
    lib.oracle_permuted_scale_bytes.argtypes = [I64, I64, I64]
    lib.oracle_permuted_scale_bytes.restype = I64
    lib.oracle_repack_scales.argtypes = [P, P, I64, I64, I64]
    _lib = lib
    return lib


def _p(arr: np.ndarray):
    return ctypes.c_void_p(arr.ctypes.data)


def _u8(x, shape) -> np.ndarray:
    arr = np.ascontiguousarray(np.asarray(x, dtype=np.uint8))
    if arr.size != int(np.prod(shape)):
        raise ValueError(f"expected {int(np.prod(shape))} bytes for shape {shape}, got {arr.size}")
    return arr.reshape(shape)


def _check_shape(M: int, K: int, L: int) -> None:
    if K % 16 != 0 or K % 2 != 0:
        raise ValueError("K must be a multiple of 16 (one E4M3 scale per 16 elements)")
    if M < 0 or K < 0 or L < 0:
        raise ValueError("negative size")


def e2m1_table() -> np.ndarray:
    """Value of each of the 16 E2M1 codes (fp64)."""
    out = np.zeros(16, dtype=np.float64)
    _load().oracle_e2m1_table(_p(out))
    return out


def e4m3_table() -> np.ndarray:
    """Value of each of the 256 E4M3 (finite-only) codes (fp64; NaN at 0x7F/0xFF)."""
    out = np.zeros(256, dtype=np.float64)
    _load().oracle_e4m3_table(_p(out))
    return out


def fp16_rne(x) -> np.ndarray:
    """IEEE binary16 bits of each double, round to nearest even."""
    xs = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.zeros(xs.shape, dtype=np.uint16)
    _load().oracle_fp16_rne_array(_p(xs), _p(out), xs.size)
    return out


def fp16_from_scaled_int(n: int) -> int:
    """binary16 bits of n * 2**-20, rounded to nearest even in integer arithmetic."""
    return int(_load().oracle_fp16_from_scaled_int(int(n)))


def gemv(a, b, sfa, sfb, M: int, K: int, L: int):
    """fp64 path over every output.

    Returns ``(c_bits, sums, sumabs)``: fp16 bits [L, M], the fp64 sum and
    the fp64 sum of |terms| per output (the latter sets the test tolerance).
    """
    _check_shape(M, K, L)
    a_ = _u8(a, (L, M, K // 2))
    b_ = _u8(b, (L, K // 2))
    sa_ = _u8(sfa, (L, M, K // 16))
    sb_ = _u8(sfb, (L, K // 16))
    c = np.zeros((L, M), dtype=np.uint16)
    s = np.zeros((L, M), dtype=np.float64)
    sabs = np.zeros((L, M), dtype=np.float64)
    _load().oracle_gemv_f64(_p(a_), _p(b_), _p(sa_), _p(sb_), M, K, L, _p(c), _p(s), _p(sabs))
    return c, s, sabs


# Output activations (codes of the library's nvfp4_activation_t), their
# textbook definitions, and a bound on |act'| over the reals: an error e in
# the activation's input moves its output by at most LIPSCHITZ * e.
ACT_NONE, ACT_RELU, ACT_SILU, ACT_GELU_TANH, ACT_GELU_ERF = 0, 1, 2, 3, 4
LIPSCHITZ = {ACT_NONE: 1.0, ACT_RELU: 1.0, ACT_SILU: 1.1, ACT_GELU_TANH: 1.13,
             ACT_GELU_ERF: 1.13}


def activate(y, act: int) -> np.ndarray:
    """act(y) in fp64, NaN in -> NaN out:

    * ReLU: y if y > 0 else +0;
    * SiLU (sigmoid-weighted linear unit): y * sigmoid(y) = y / (1 + exp(-y));
    * GELU, tanh form: y/2 * (1 + tanh(sqrt(2/pi) * (y + 0.044715 * y^3)));
    * GELU, erf form: y/2 * (1 + erf(y / sqrt(2))) = y * Phi(y).
    """
    y = np.asarray(y, dtype=np.float64)
    if act == ACT_NONE:
        return y
    if act == ACT_RELU:
        return np.where(y > 0, y, np.where(np.isnan(y), y, 0.0))
    with np.errstate(over="ignore", invalid="ignore"):
        if act == ACT_SILU:
            return y / (1.0 + np.exp(-y))
        if act == ACT_GELU_TANH:
            return 0.5 * y * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (y + 0.044715 * y ** 3)))
        if act == ACT_GELU_ERF:
            erf = np.vectorize(math.erf, otypes=[np.float64])
            return 0.5 * y * (1.0 + erf(y / math.sqrt(2.0)))
    raise ValueError(f"unknown activation {act}")


def gemv_ex(a, b, sfa, sfb, M: int, K: int, L: int, alpha: float = 1.0, bias=None,
            activation: int = ACT_NONE):
    """fp64 path with an output scale, bias and activation:
    ``fp16(act(alpha * sum + bias))``.

    ``bias`` is fp16 bits [L, M] (uint16) or None.  ``act(alpha * sum + bias)``
    is formed in fp64 from the fp64 sums of :func:`gemv` and rounded to
    binary16 once.  Returns ``(c_bits, values, LIPSCHITZ[act] * |alpha| *
    sumabs)``: the fp64 values before rounding and the |term| sums scaled like
    the sums (the tolerance).
    """
    _, s, sabs = gemv(a, b, sfa, sfb, M, K, L)
    y = np.float64(alpha) * s
    if bias is not None:
        bv = np.ascontiguousarray(np.asarray(bias, dtype=np.uint16)).view(np.float16)
        y = y + bv.astype(np.float64).reshape(L, M)
    y = activate(y, activation)
    return fp16_rne(y), y, LIPSCHITZ[activation] * abs(float(alpha)) * sabs


def gemm_small_n(a, b, sfa, sfb, M: int, N: int, K: int, L: int, alpha: float = 1.0,
                 bias=None, activation: int = ACT_NONE):
    """Small-N GEMM: N dot products per row of A, one per vector of b::

        c[l, n, m] = fp16(alpha * sum_k E2M1(a[m,k,l]) * E4M3(sfa[m,k//16,l])
                                      * E2M1(b[n,k,l]) * E4M3(sfb[n,k//16,l]) + bias[l, n, m])

    i.e. the GEMV definition above applied to each vector n (the pages' harness
    multiplies A by an N-column B through ``torch._scaled_mm``, submission
    103289's ``cute_jit_kernel`` padding N to 128).  ``b`` uint8 [L, N, K//2],
    ``sfb`` uint8 [L, N, K//16], ``bias`` fp16 bits [L, N, M] or None.
    Returns ``(c_bits [L, N, M], values, |alpha| * sumabs)`` as :func:`gemv_ex`.
    """
    b_ = np.ascontiguousarray(np.asarray(b, dtype=np.uint8).reshape(L, N, K // 2))
    sb_ = np.ascontiguousarray(np.asarray(sfb, dtype=np.uint8).reshape(L, N, K // 16))
    bias_ = None if bias is None else np.asarray(bias, dtype=np.uint16).reshape(L, N, M)
    c = np.zeros((L, N, M), dtype=np.uint16)
    vals = np.zeros((L, N, M), dtype=np.float64)
    tol = np.zeros((L, N, M), dtype=np.float64)
    for n in range(N):
        bn = None if bias_ is None else np.ascontiguousarray(bias_[:, n, :])
        c[:, n, :], vals[:, n, :], tol[:, n, :] = gemv_ex(
            a, np.ascontiguousarray(b_[:, n, :]), sfa, np.ascontiguousarray(sb_[:, n, :]),
            M, K, L, alpha, bn, activation)
    return c, vals, tol


def gemv_at(a, b, sfa, sfb, M: int, K: int, L: int, m_idx, l_idx):
    """fp64 path for the selected outputs ``(m_idx[i], l_idx[i])`` only."""
    _check_shape(M, K, L)
    a_ = _u8(a, (L, M, K // 2))
    b_ = _u8(b, (L, K // 2))
    sa_ = _u8(sfa, (L, M, K // 16))
    sb_ = _u8(sfb, (L, K // 16))
    mi = np.ascontiguousarray(np.asarray(m_idx, dtype=np.int64))
    li = np.ascontiguousarray(np.asarray(l_idx, dtype=np.int64))
    if mi.shape != li.shape:
        raise ValueError("m_idx and l_idx differ in shape")
    if mi.size and (mi.min() < 0 or mi.max() >= M or li.min() < 0 or li.max() >= L):
        raise ValueError("sample index out of range")
    n = mi.size
    c = np.zeros(n, dtype=np.uint16)
    s = np.zeros(n, dtype=np.float64)
    sabs = np.zeros(n, dtype=np.float64)
    _load().oracle_gemv_f64_at(_p(a_), _p(b_), _p(sa_), _p(sb_), M, K, L, _p(mi), _p(li), n,
                               _p(c), _p(s), _p(sabs))
    return c, s, sabs


def gemv_exact(a, b, sfa, sfb, M: int, K: int, L: int):
    """Exact int64 path.  Returns ``(c_bits, num, nan)`` where ``num`` is the
    exact sum times 2**20 and ``nan`` marks outputs with a NaN scale."""
    _check_shape(M, K, L)
    a_ = _u8(a, (L, M, K // 2))
    b_ = _u8(b, (L, K // 2))
    sa_ = _u8(sfa, (L, M, K // 16))
    sb_ = _u8(sfb, (L, K // 16))
    num = np.zeros((L, M), dtype=np.int64)
    nan = np.zeros((L, M), dtype=np.uint8)
    c = np.zeros((L, M), dtype=np.uint16)
    rc = _load().oracle_gemv_exact(_p(a_), _p(b_), _p(sa_), _p(sb_), M, K, L, _p(num), _p(nan),
                                   _p(c))
    if rc != 0:
        raise ValueError("exact path supports K <= 2**20")
    return c, num, nan.astype(bool)


def permuted_scale_bytes(rows: int, K: int, L: int) -> int:
    return int(_load().oracle_permuted_scale_bytes(rows, K, L))


def repack_scales(src, rows: int, K: int, L: int) -> np.ndarray:
    """Plain scales [L, rows, K//16] -> flat 128x4-atom permuted bytes."""
    if K % 16 != 0:
        raise ValueError("scales come in 16-element blocks: K % 16 == 0")
    s = _u8(src, (L, rows, K // 16))
    out = np.zeros(permuted_scale_bytes(rows, K, L), dtype=np.uint8)
    _load().oracle_repack_scales(_p(s), _p(out), rows, K, L)
    return out
