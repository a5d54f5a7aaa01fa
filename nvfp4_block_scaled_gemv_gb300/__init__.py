"""NVFP4 block-scaled batched GEMV on GB300 (sm_103a): Python binding.

A thin ctypes binding of the C ABI declared in ``include/nvfp4_gemv.h``: the
functions below take device pointers as integers (or torch tensors in the
``gemv`` / ``repack_scales`` conveniences) and only marshal arguments; every
step of the computation runs in the library's CUDA kernels.  There is no
fallback: if the library is not built, or a call fails, an exception is
raised.

    c[m, l] = fp16( sum_k E2M1(a[m,k,l]) * E4M3(sfa[m,k//16,l])
                         * E2M1(b[k,l])  * E4M3(sfb[k//16,l]) )
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libnvfp4_gemv.so")

SF_PLAIN = 0
SF_PERMUTED_128x4 = 1

OK = 0
ERR_INVALID_VALUE = 1
ERR_UNSUPPORTED_SHAPE = 2
ERR_MISALIGNED = 3
ERR_CUDA = 4

# Every symbol include/nvfp4_gemv.h declares.
EXPORTS = (
    "nvfp4_gemv",
    "nvfp4_gemv_ex",
    "nvfp4_gemv_explicit",
    "nvfp4_repack_scales",
    "nvfp4_permuted_scale_bytes",
    "nvfp4_status_string",
    "nvfp4_last_cuda_error",
    "nvfp4_gemv_plan",
    "nvfp4_tensor_wait_timeouts",
    "nvfp4_selftest_bounded_wait",
    "nvfp4_gemm_small_n",
    "nvfp4_gemm_small_n_explicit",
    "nvfp4_gemm_small_n_plan",
)


class Nvfp4Error(RuntimeError):
    """A library call returned a status other than NVFP4_OK."""

    def __init__(self, status: int, where: str, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        msg = f"{where}: {status_string(status)}"
        if status == ERR_CUDA:
            msg += f" (cudaError {cuda_error})"
        super().__init__(msg)


KERNEL_DIRECT = 0
KERNEL_PIPELINED = 1
KERNEL_TENSOR = 2
KERNEL_BLOCKDOT = 3
KERNEL_BLOCKWISE = 4
ACT_NONE, ACT_RELU, ACT_SILU, ACT_GELU_TANH, ACT_GELU_ERF = 0, 1, 2, 3, 4


class _Plan(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int), ("lanes_per_row", ctypes.c_int), ("k_split", ctypes.c_int),
                ("rows_per_pass", ctypes.c_int), ("threads_per_cta", ctypes.c_int),
                ("ctas", ctypes.c_int64), ("steps", ctypes.c_int64)]


class _Options(ctypes.Structure):
    _fields_ = [("alpha", ctypes.c_float), ("bias", ctypes.c_void_p),
                ("b_batch_stride", ctypes.c_int64), ("sfb_batch_stride", ctypes.c_int64),
                ("activation", ctypes.c_int32)]


_lib = None


def library() -> ctypes.CDLL:
    """The loaded shared library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -m nvfp4_block_scaled_gemv_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.nvfp4_gemv.argtypes = [P, P, P, P, P, I64, I64, I64, I, P]
    lib.nvfp4_gemv.restype = I
    lib.nvfp4_gemv_explicit.argtypes = [P, P, P, P, P, I64, I64, I64, I, I, I, I, I64, P]
    lib.nvfp4_gemv_ex.restype = I
    lib.nvfp4_gemv_ex.argtypes = [P, P, P, P, P, I64, I64, I64, I, ctypes.POINTER(_Options), P]
    lib.nvfp4_gemv_explicit.restype = I
    lib.nvfp4_repack_scales.argtypes = [P, P, I64, I64, I64, P]
    lib.nvfp4_repack_scales.restype = I
    lib.nvfp4_permuted_scale_bytes.argtypes = [I64, I64, I64]
    lib.nvfp4_permuted_scale_bytes.restype = ctypes.c_size_t
    lib.nvfp4_status_string.argtypes = [I]
    lib.nvfp4_status_string.restype = ctypes.c_char_p
    lib.nvfp4_last_cuda_error.argtypes = []
    lib.nvfp4_last_cuda_error.restype = I
    lib.nvfp4_gemv_plan.argtypes = [I64, I64, I64, I, I, I, I, ctypes.POINTER(_Plan)]
    lib.nvfp4_gemv_plan.restype = I
    lib.nvfp4_gemm_small_n.argtypes = [P, P, P, P, P, I64, I64, I64, I64,
                                       ctypes.POINTER(_Options), P]
    lib.nvfp4_gemm_small_n.restype = I
    lib.nvfp4_gemm_small_n_explicit.argtypes = [P, P, P, P, P, I64, I64, I64, I64, I, I, I64, P]
    lib.nvfp4_gemm_small_n_explicit.restype = I
    lib.nvfp4_gemm_small_n_plan.argtypes = [I64, I64, I64, I64, ctypes.POINTER(I),
                                            ctypes.POINTER(I), ctypes.POINTER(I64),
                                            ctypes.POINTER(I)]
    lib.nvfp4_gemm_small_n_plan.restype = I
    lib.nvfp4_tensor_wait_timeouts.argtypes = [I]
    lib.nvfp4_tensor_wait_timeouts.restype = I
    lib.nvfp4_selftest_bounded_wait.argtypes = [ctypes.POINTER(I), ctypes.POINTER(I),
                                                ctypes.POINTER(I), ctypes.POINTER(I64), P]
    lib.nvfp4_selftest_bounded_wait.restype = I
    _lib = lib
    return lib


def _check(status: int, where: str) -> None:
    if status != OK:
        raise Nvfp4Error(status, where, library().nvfp4_last_cuda_error() if status == ERR_CUDA else 0)


def status_string(status: int) -> str:
    return library().nvfp4_status_string(int(status)).decode()


def nvfp4_gemv(a: int, b: int, sfa: int, sfb: int, c: int, M: int, K: int, L: int,
               sf_layout: int = SF_PLAIN, stream: int = 0) -> None:
    """Enqueue c = GEMV(a, b, sfa, sfb) on ``stream`` (device pointers as ints)."""
    _check(library().nvfp4_gemv(a, b, sfa, sfb, c, M, K, L, sf_layout, stream), "nvfp4_gemv")


def nvfp4_gemv_ex(a: int, b: int, sfa: int, sfb: int, c: int, M: int, K: int, L: int,
                  sf_layout: int = SF_PLAIN, alpha: float = 1.0, bias: int = 0,
                  b_batch_stride: int = 0, sfb_batch_stride: int = 0, stream: int = 0,
                  activation: int = 0) -> None:
    """nvfp4_gemv with an output scale, an fp16 [L][M] bias (pointer or 0),
    batch strides for b and sfb (0 = dense) and an output activation (ACT_*)."""
    opt = _Options(alpha, bias or None, b_batch_stride, sfb_batch_stride, activation)
    _check(library().nvfp4_gemv_ex(a, b, sfa, sfb, c, M, K, L, sf_layout, ctypes.byref(opt),
                                   stream), "nvfp4_gemv_ex")


def nvfp4_gemv_explicit(a: int, b: int, sfa: int, sfb: int, c: int, M: int, K: int, L: int,
                        sf_layout: int, kernel: int, lanes_per_row: int, k_split: int, ctas: int,
                        stream: int = 0) -> None:
    """nvfp4_gemv with an explicit kernel and launch schedule."""
    _check(library().nvfp4_gemv_explicit(a, b, sfa, sfb, c, M, K, L, sf_layout, kernel,
                                         lanes_per_row, k_split, ctas, stream),
           "nvfp4_gemv_explicit")


def nvfp4_gemm_small_n(a: int, b: int, sfa: int, sfb: int, c: int, M: int, N: int, K: int,
                       L: int, alpha: float = 1.0, bias: int = 0, b_batch_stride: int = 0,
                       sfb_batch_stride: int = 0, stream: int = 0, activation: int = 0) -> None:
    """Small-N GEMM: c [L][N][M] from a [L][M][K/2], b [L][N][K/2] and
    pre-permuted scales (sfb: the permuted form of [L][N][K/16])."""
    opt = _Options(alpha, bias or None, b_batch_stride, sfb_batch_stride, activation)
    _check(library().nvfp4_gemm_small_n(a, b, sfa, sfb, c, M, N, K, L, ctypes.byref(opt),
                                        stream), "nvfp4_gemm_small_n")


def nvfp4_gemm_small_n_explicit(a: int, b: int, sfa: int, sfb: int, c: int, M: int, N: int,
                                K: int, L: int, stages: int, k_split: int, ctas: int,
                                stream: int = 0) -> None:
    """nvfp4_gemm_small_n on the tensor-core kernel with a given schedule."""
    _check(library().nvfp4_gemm_small_n_explicit(a, b, sfa, sfb, c, M, N, K, L, stages,
                                                 k_split, ctas, stream),
           "nvfp4_gemm_small_n_explicit")


def nvfp4_gemm_small_n_plan(M: int, N: int, K: int, L: int) -> dict:
    """The tensor-core schedule nvfp4_gemm_small_n uses (queries the device)."""
    st, ks, ctas, res = ctypes.c_int(), ctypes.c_int(), ctypes.c_int64(), ctypes.c_int()
    _check(library().nvfp4_gemm_small_n_plan(M, N, K, L, ctypes.byref(st), ctypes.byref(ks),
                                             ctypes.byref(ctas), ctypes.byref(res)),
           "nvfp4_gemm_small_n_plan")
    return {"stages": st.value, "k_split": ks.value, "ctas": ctas.value,
            "resident_ctas": res.value}


def nvfp4_repack_scales(src: int, dst: int, rows: int, K: int, L: int, stream: int = 0) -> None:
    """Enqueue plain [L][rows][K/16] -> 128x4-atom permuted scale repack."""
    _check(library().nvfp4_repack_scales(src, dst, rows, K, L, stream), "nvfp4_repack_scales")


def nvfp4_permuted_scale_bytes(rows: int, K: int, L: int) -> int:
    return int(library().nvfp4_permuted_scale_bytes(rows, K, L))


def nvfp4_last_cuda_error() -> int:
    return int(library().nvfp4_last_cuda_error())


def nvfp4_tensor_wait_timeouts(reset: bool = False) -> int:
    """Bounded waits of the tensor-core kernel that ran out (synchronises)."""
    return int(library().nvfp4_tensor_wait_timeouts(1 if reset else 0))


def nvfp4_selftest_bounded_wait(stream: int = 0) -> dict:
    """Run the device self-test of the kernels' bounded barrier wait (about 2 s;
    synchronises): one wait that completes and one that must give up."""
    completed, gave_up, timeouts = ctypes.c_int(-1), ctypes.c_int(-1), ctypes.c_int(-1)
    waited = ctypes.c_int64(-1)
    _check(library().nvfp4_selftest_bounded_wait(ctypes.byref(completed), ctypes.byref(gave_up),
                                                 ctypes.byref(timeouts), ctypes.byref(waited),
                                                 stream), "nvfp4_selftest_bounded_wait")
    return {"completed": completed.value, "gave_up": gave_up.value, "timeouts": timeouts.value,
            "waited_ns": waited.value}


def nvfp4_gemv_plan(M: int, K: int, L: int, sf_layout: int = SF_PLAIN, num_sms: int = 152,
                    ctas_per_sm: int = 0, kernel: int = -1) -> dict:
    """The launch schedule nvfp4_gemv would use (kernel=-1) or one kernel's
    schedule (host only, no GPU)."""
    plan = _Plan()
    _check(library().nvfp4_gemv_plan(M, K, L, sf_layout, kernel, num_sms, ctas_per_sm,
                                     ctypes.byref(plan)), "nvfp4_gemv_plan")
    return {name: getattr(plan, name) for name, _ in _Plan._fields_}


# ---------------------------------------------------------------------------
# torch conveniences: argument marshalling only
# ---------------------------------------------------------------------------

def _stream_handle(stream, device) -> int:
    import torch

    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _on_device(device):
    """Makes `device` current for a call (the library plans and launches on the
    calling thread's current device)."""
    import contextlib

    import torch

    return torch.cuda.device(device) if device.type == "cuda" else contextlib.nullcontext()


def _need(t, name, dtype, numel, device):
    import torch

    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.numel() != numel:
        raise ValueError(f"{name} has {t.numel()} elements, expected {numel}")
    if numel and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def gemv(a, b, sfa, sfb, c=None, sf_layout: int = SF_PLAIN, stream=None):
    """c [L, M] float16 from a [L, M, K//2], b [L, K//2] (uint8) and uint8 scales
    (plain [L, M, K//16] / [L, K//16], or permuted flat bytes)."""
    import torch

    if a.dim() != 3:
        raise ValueError("a must be [L, M, K//2]")
    L, M, half_k = a.shape
    K = 2 * half_k
    dev = a.device
    _need(a, "a", torch.uint8, L * M * half_k, dev)
    _need(b, "b", torch.uint8, L * half_k, dev)
    if sf_layout == SF_PLAIN:
        _need(sfa, "sfa", torch.uint8, L * M * (K // 16), dev)
        _need(sfb, "sfb", torch.uint8, L * (K // 16), dev)
    else:
        _need(sfa, "sfa", torch.uint8, nvfp4_permuted_scale_bytes(M, K, L), dev)
        _need(sfb, "sfb", torch.uint8, nvfp4_permuted_scale_bytes(1, K, L), dev)
    if c is None:
        c = torch.empty((L, M), dtype=torch.float16, device=dev)
    _need(c, "c", torch.float16, L * M, dev)
    with _on_device(dev):
        nvfp4_gemv(a.data_ptr(), b.data_ptr(), sfa.data_ptr(), sfb.data_ptr(), c.data_ptr(), M, K,
                   L, sf_layout, _stream_handle(stream, dev))
    return c


def repack_scales(src, dst=None, stream=None):
    """Plain scales [L, rows, K//16] (uint8) -> flat permuted bytes (uint8)."""
    import torch

    if src.dim() != 3:
        raise ValueError("src must be [L, rows, K//16]")
    L, rows, blocks = src.shape
    K = 16 * blocks
    _need(src, "src", torch.uint8, L * rows * blocks, src.device)
    n = nvfp4_permuted_scale_bytes(rows, K, L)
    if dst is None:
        dst = torch.empty(n, dtype=torch.uint8, device=src.device)
    _need(dst, "dst", torch.uint8, n, src.device)
    with _on_device(src.device):
        nvfp4_repack_scales(src.data_ptr(), dst.data_ptr(), rows, K, L,
                            _stream_handle(stream, src.device))
    return dst
