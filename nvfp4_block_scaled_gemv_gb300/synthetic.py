"""Seeded synthetic NVFP4 GEMV inputs (no GEMV arithmetic lives here).

Both the CUDA path and the CPU oracle are fed from this module; it only draws
bytes.  The generator is splitmix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014) used as a counter-based stream:
output i (i = 1, 2, ...) of stream ``s`` is ``mix(s + i * 0x9E3779B97F4A7C15)``.

Recipe (one stream per tensor, seeded ``seed * 16 + t`` with t = 0 for a,
1 for b, 2 for sfa, 3 for sfb):

* ``a``, ``b``: raw little-endian bytes of consecutive outputs, so each
  nibble is uniform over all 16 E2M1 codes, -0 (0x8) included.
* ``sfa``, ``sfb``: one output per byte, ``0x18 + out % 25``: uniform over
  the 25 positive E4M3 codes 0x18..0x30, whose values span [1/16, 1/2].

Layouts (C order): a [L, M, K//2], b [L, K//2], sfa [L, M, K//16],
sfb [L, K//16].
"""
from __future__ import annotations

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

STREAM_A, STREAM_B, STREAM_SFA, STREAM_SFB = 0, 1, 2, 3
SCALE_CODE_LO, SCALE_CODE_COUNT = 0x18, 25


def splitmix64(stream_seed: int, n: int, start: int = 0) -> np.ndarray:
    """Outputs ``start+1 .. start+n`` of the splitmix64 stream (uint64)."""
    out = np.empty(n, dtype=np.uint64)
    seed = np.uint64(stream_seed & 0xFFFFFFFFFFFFFFFF)
    with np.errstate(over="ignore"):
        for lo in range(0, n, _CHUNK):
            hi = min(n, lo + _CHUNK)
            z = np.arange(start + lo + 1, start + hi + 1, dtype=np.uint64)
            z *= GAMMA
            z += seed
            z ^= z >> np.uint64(30)
            z *= _M1
            z ^= z >> np.uint64(27)
            z *= _M2
            z ^= z >> np.uint64(31)
            out[lo:hi] = z
    return out


def random_bytes(stream_seed: int, n: int) -> np.ndarray:
    """n uniform bytes: the little-endian bytes of consecutive outputs."""
    words = splitmix64(stream_seed, (n + 7) // 8)
    return words.astype("<u8", copy=False).view(np.uint8)[:n].copy()


def scale_bytes(stream_seed: int, n: int, code_lo: int = SCALE_CODE_LO,
                code_count: int = SCALE_CODE_COUNT) -> np.ndarray:
    """n E4M3 codes uniform over code_lo .. code_lo + code_count - 1 (by
    default 0x18..0x30, values in [1/16, 1/2])."""
    out = np.empty(n, dtype=np.uint8)
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        w = splitmix64(stream_seed, hi - lo, start=lo)
        out[lo:hi] = (w % np.uint64(code_count)).astype(np.uint8) + np.uint8(code_lo)
    return out


def make_problem(M: int, K: int, L: int, seed: int = 0,
                 scale_codes: tuple = (SCALE_CODE_LO, SCALE_CODE_COUNT)) -> dict:
    """Plain-layout inputs of one batched GEMV problem, as numpy arrays.
    scale_codes = (first code, number of codes) of the uniform scale draw."""
    if K % 16 != 0:
        raise ValueError("K must be a multiple of 16")
    base = seed * 16
    return {
        "a": random_bytes(base + STREAM_A, L * M * (K // 2)).reshape(L, M, K // 2),
        "b": random_bytes(base + STREAM_B, L * (K // 2)).reshape(L, K // 2),
        "sfa": scale_bytes(base + STREAM_SFA, L * M * (K // 16), *scale_codes).reshape(L, M, K // 16),
        "sfb": scale_bytes(base + STREAM_SFB, L * (K // 16), *scale_codes).reshape(L, K // 16),
    }


def make_gemm_problem(M: int, N: int, K: int, L: int, seed: int = 0) -> dict:
    """Plain-layout inputs of a small-N GEMM: the GEMV recipe with b and sfb
    drawn as N rows per batch (b [L, N, K//2], sfb [L, N, K//16]); N = 1 gives
    make_problem's bytes."""
    if K % 64 != 0:
        raise ValueError("K must be a multiple of 64")
    base = seed * 16
    return {
        "a": random_bytes(base + STREAM_A, L * M * (K // 2)).reshape(L, M, K // 2),
        "b": random_bytes(base + STREAM_B, L * N * (K // 2)).reshape(L, N, K // 2),
        "sfa": scale_bytes(base + STREAM_SFA, L * M * (K // 16)).reshape(L, M, K // 16),
        "sfb": scale_bytes(base + STREAM_SFB, L * N * (K // 16)).reshape(L, N, K // 16),
    }


# The benchmark workloads: (name, M, K, L).  The first is a small parity case,
# the next three are the shapes the submissions time (submission 69953's
# docstring performance targets), the last a 1.2 GB sustained-bandwidth case.
WORKLOADS = [
    ("M128_K256_L1", 128, 256, 1),
    ("M7168_K2048_L4", 7168, 2048, 4),
    ("M4096_K7168_L8", 4096, 7168, 8),
    ("M7168_K16384_L1", 7168, 16384, 1),
    ("M16384_K8192_L16", 16384, 8192, 16),
]


def algorithmic_bytes(M: int, K: int, L: int) -> int:
    """Bytes one call must move at least: A + sfa + b + sfb + c."""
    return L * M * (K // 2 + K // 16 + 2) + L * (K // 2 + K // 16)


# Small-N GEMM workloads (decode batches of N vectors on the GEMV shapes):
# (name, M, N, K, L).
GEMM_WORKLOADS = [
    ("M7168_N8_K2048_L4", 7168, 8, 2048, 4),
    ("M4096_N4_K7168_L8", 4096, 4, 7168, 8),
    ("M7168_N16_K16384_L1", 7168, 16, 16384, 1),
    ("M16384_N8_K8192_L16", 16384, 8, 8192, 16),
]


def gemm_algorithmic_bytes(M: int, N: int, K: int, L: int) -> int:
    """Bytes a small-N GEMM must move: A + sfa + N x (b + sfb) read, c written."""
    return L * (M * (K // 2 + K // 16) + N * (K // 2 + K // 16) + 2 * N * M)
