"""Python binding for libtg_gemm.so, the GB300 fp16 tiled tensor-core GEMM.

C[i,j] = epi(sum_k A[i,k] B[k,j] + bias[j]), epi = identity or exact-erf GELU:
the GEMM of "TileLang: writing LLM GPU kernels by thinking in tiles"
(sections 2-3) with the GELU(MatMul + Bias) epilogue of "Designing
high-performance GPU kernels with TileLang ..." (section 3).

This module only marshals arguments into the C ABI declared in
include/tg_gemm.h: every step of the computation runs in the library's CUDA
kernels. Functions named tg_* mirror the C entry points one to one (raw
pointers as ints, sizes, a stream handle); ``gemm`` and ``gemm_staged`` accept
torch tensors and pass their pointers and torch's current stream. There is no
CPU path: if the library has not been built, importing this package raises.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtg_gemm.so")

EPI_NONE, EPI_GELU = 0, 1
NOALLOC_SCRATCH_BYTES = 8 * 1024 * 1024  # TG_NOALLOC_SCRATCH_BYTES
KERNEL_AUTO, KERNEL_TILED_TMA, KERNEL_TILED_LSU, KERNEL_SPLITK, KERNEL_TILED_PAIR = 0, 1, 2, 3, 4
W4_INT4, W4_FP4_E2M1 = 0, 1
W4_KERNEL_AUTO, W4_KERNEL_TMEM, W4_KERNEL_REG = 0, 1, 2
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED_DEVICE, ERR_CUDA, ERR_TIMEOUT, ERR_NO_MEMORY, ERR_BOUNDS = range(7)

# every symbol include/tg_gemm.h declares
EXPORTS = ("tg_gemm", "tg_gemm_ex", "tg_gemm_plan", "tg_gemm_staged", "tg_gemm_splitk_noalloc", "tg_gemm_w4", "tg_gemm_w4_ex",
           "tg_gemm_w4_kernel", "tg_attention_fwd",
           "tg_softmax_rows", "tg_bias_gelu",
           "tg_device_status", "tg_debug_status",
           "tg_set_watchdog_ns",
           "tg_debug_skip_first_arrive", "tg_debug_bounds_limit", "tg_debug_build", "tg_status_string",
           "tg_last_error", "tg_version",
           "tg_ring_bytes", "tg_shutdown")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
                      "(or python tiled_tensor_core_tcgen05_gb300/build.py); there is no fallback path")

_vp, _i64, _int, _u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint64


def bind(path: str) -> ctypes.CDLL:
    """Load a build of the library (this package's, or its debug build
    libtg_gemm_debug.so) with every entry point's C signature set."""
    lib = ctypes.CDLL(path)
    lib.tg_gemm.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp]
    lib.tg_gemm_ex.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _int, _int, _vp]
    lib.tg_gemm_plan.argtypes = [_vp, _vp, _i64, _i64, _i64, ctypes.POINTER(_int), ctypes.POINTER(_int),
                                 ctypes.POINTER(_int)]
    lib.tg_gemm_staged.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp]
    lib.tg_gemm_splitk_noalloc.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _int, _vp]
    lib.tg_gemm_w4.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _int, _vp]
    lib.tg_gemm_w4_ex.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _int, _int, _vp]
    lib.tg_gemm_w4_kernel.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _int, _int, _int, _vp]
    lib.tg_attention_fwd.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _int, _vp]
    lib.tg_softmax_rows.argtypes = [_vp, _vp, _i64, _i64, _vp]
    lib.tg_bias_gelu.argtypes = [_vp, _vp, _i64, _i64, _int, _vp]
    lib.tg_device_status.argtypes = [_vp, ctypes.POINTER(_int)]
    lib.tg_debug_status.argtypes = [_vp]
    lib.tg_set_watchdog_ns.argtypes = [_u64]
    lib.tg_debug_skip_first_arrive.argtypes = [_int]
    lib.tg_debug_bounds_limit.argtypes = [_i64]
    lib.tg_debug_build.argtypes = []
    lib.tg_status_string.argtypes = [_int]
    lib.tg_status_string.restype = ctypes.c_char_p
    lib.tg_last_error.argtypes = []
    lib.tg_last_error.restype = ctypes.c_char_p
    lib.tg_version.argtypes = []
    lib.tg_ring_bytes.argtypes = [_int]
    lib.tg_ring_bytes.restype = _i64
    lib.tg_shutdown.argtypes = []
    lib.tg_shutdown.restype = None
    for name in ("tg_gemm", "tg_gemm_ex", "tg_gemm_plan", "tg_gemm_staged", "tg_gemm_splitk_noalloc", "tg_gemm_w4", "tg_gemm_w4_ex",
                 "tg_gemm_w4_kernel", "tg_attention_fwd", "tg_softmax_rows", "tg_bias_gelu", "tg_device_status", "tg_debug_status",
                 "tg_set_watchdog_ns", "tg_debug_skip_first_arrive", "tg_debug_bounds_limit", "tg_debug_build",
                 "tg_version"):
        getattr(lib, name).restype = _int
    return lib


_lib = bind(LIB_PATH)


class TgError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{tg_status_string(status)}: {message}")
        self.status = status


def _check(status: int) -> None:
    if status != OK:
        raise TgError(status, tg_last_error())


def library() -> ctypes.CDLL:
    return _lib


# ---------------------------------------------------------------- raw C ABI

def tg_gemm(A: int, B: int, bias: int | None, C: int, M: int, N: int, K: int, epilogue: int,
            stream: int | None) -> None:
    _check(_lib.tg_gemm(A, B, bias, C, M, N, K, epilogue, stream))


def tg_gemm_ex(A: int, B: int, bias: int | None, C: int, M: int, N: int, K: int, epilogue: int,
               kernel: int, split_k: int, stream: int | None) -> None:
    _check(_lib.tg_gemm_ex(A, B, bias, C, M, N, K, epilogue, kernel, split_k, stream))


def tg_gemm_plan(A: int | None, B: int | None, M: int, N: int, K: int) -> tuple[int, int, int]:
    """(kernel, K slices, aligned copy 0/1) that tg_gemm would take for these operands."""
    k, s, c = _int(), _int(), _int()
    _check(_lib.tg_gemm_plan(A, B, M, N, K, ctypes.byref(k), ctypes.byref(s), ctypes.byref(c)))
    return k.value, s.value, c.value


def tg_gemm_staged(hA, hB, hbias, hC, dA, dB, dbias, dC, M, N, K, epilogue, stream) -> None:
    _check(_lib.tg_gemm_staged(hA, hB, hbias, hC, dA, dB, dbias, dC, M, N, K, epilogue, stream))


def tg_gemm_splitk_noalloc(A: int, B: int, bias: int | None, C: int, M: int, N: int, K: int, epilogue: int,
                           split_k: int, stream: int | None) -> None:
    """The skinny split-K GEMM with its scratch in the library's fixed device
    array, for callers that must not have the library allocate device memory
    (see include/tg_gemm.h for the size limit and the sharing rules)."""
    _check(_lib.tg_gemm_splitk_noalloc(A, B, bias, C, M, N, K, epilogue, split_k, stream))


def tg_gemm_w4(A: int, Bq: int, scales: int, bias: int | None, C: int, M: int, N: int, K: int, epilogue: int,
               split_k: int, stream: int | None) -> None:
    _check(_lib.tg_gemm_w4(A, Bq, scales, bias, C, M, N, K, epilogue, split_k, stream))


def tg_gemm_w4_ex(A: int, Bq: int, scales: int, bias: int | None, C: int, M: int, N: int, K: int, epilogue: int,
                  weight_format: int, split_k: int, stream: int | None) -> None:
    _check(_lib.tg_gemm_w4_ex(A, Bq, scales, bias, C, M, N, K, epilogue, weight_format, split_k, stream))


def tg_gemm_w4_kernel(A: int, Bq: int, scales: int, bias: int | None, C: int, M: int, N: int, K: int,
                      epilogue: int, weight_format: int, kernel: int, split_k: int, stream: int | None) -> None:
    _check(_lib.tg_gemm_w4_kernel(A, Bq, scales, bias, C, M, N, K, epilogue, weight_format, kernel, split_k,
                                  stream))


def tg_attention_fwd(Q: int, K: int, V: int, O: int, B: int, S: int, H: int, D: int, causal: bool,
                     stream: int | None) -> None:
    _check(_lib.tg_attention_fwd(Q, K, V, O, B, S, H, D, 1 if causal else 0, stream))


def attention(Q, K, V, causal: bool = False, out=None, stream=None):
    """O = softmax(Q K^T / sqrt(D)) V for CUDA float16 tensors of shape
    (batch, sequence, heads, 128), contiguous; optional causal mask."""
    import torch
    if Q.dim() != 4 or Q.shape != K.shape or Q.shape != V.shape:
        raise ValueError(f"Q, K, V must share one (B, S, H, D) shape: {tuple(Q.shape)} {tuple(K.shape)} {tuple(V.shape)}")
    B, S, H, D = Q.shape
    if out is None:
        out = torch.empty_like(Q)
    elif out.shape != Q.shape:
        raise ValueError("out has the wrong shape")
    if Q.numel() == 0:
        return out
    tg_attention_fwd(_dev_fp16(Q, "Q"), _dev_fp16(K, "K"), _dev_fp16(V, "V"), _dev_fp16(out, "out"), B, S, H, D,
                     causal, _stream_handle(stream))
    return out


def tg_softmax_rows(X: int, Y: int, M: int, N: int, stream: int | None) -> None:
    _check(_lib.tg_softmax_rows(X, Y, M, N, stream))


def softmax(X, out=None, stream=None):
    """Row softmax of a CUDA float16 matrix (contiguous); ``out`` may be X."""
    import torch
    if X.dim() != 2:
        raise ValueError("X must be a matrix")
    if out is None:
        out = torch.empty_like(X)
    elif out.shape != X.shape:
        raise ValueError("out has the wrong shape")
    if X.numel():
        tg_softmax_rows(_dev_fp16(X, "X"), _dev_fp16(out, "out"), X.shape[0], X.shape[1], _stream_handle(stream))
    return out


def tg_bias_gelu(C: int, bias: int | None, M: int, N: int, epilogue: int, stream: int | None) -> None:
    _check(_lib.tg_bias_gelu(C, bias, M, N, epilogue, stream))


def bias_gelu_(C, bias=None, gelu: bool = True, stream=None):
    """In place C = epi(C + bias) on a CUDA float16 matrix (the unfused epilogue pass)."""
    M, N = C.shape
    tg_bias_gelu(_dev_fp16(C, "C"), _dev_fp16(bias, "bias") if bias is not None else None, M, N,
                 EPI_GELU if gelu else EPI_NONE, _stream_handle(stream))
    return C


def tg_device_status(stream: int | None) -> tuple[int, int]:
    where = _int(0)
    st = _lib.tg_device_status(stream, ctypes.byref(where))
    return st, where.value


def tg_debug_status(stream: int | None) -> int:
    """Synchronises `stream` and returns (and clears) the kernels' watchdog status."""
    return _lib.tg_debug_status(stream)


def tg_set_watchdog_ns(ns: int) -> None:
    _check(_lib.tg_set_watchdog_ns(ns))


def tg_debug_skip_first_arrive(on: bool) -> None:
    _check(_lib.tg_debug_skip_first_arrive(1 if on else 0))


def tg_debug_bounds_limit(floats: int) -> None:
    """Debug builds: make the device-side bounds checks treat scratch as `floats` long (0: real size)."""
    _check(_lib.tg_debug_bounds_limit(floats))


def tg_debug_build() -> int:
    """1 if the loaded library was compiled with its device-side bounds checks, else 0."""
    return _lib.tg_debug_build()


def tg_status_string(status: int) -> str:
    return _lib.tg_status_string(status).decode()


def tg_last_error() -> str:
    return _lib.tg_last_error().decode()


def tg_version() -> int:
    return _lib.tg_version()


def tg_ring_bytes(kernel: int) -> int:
    return _lib.tg_ring_bytes(kernel)


def tg_shutdown() -> None:
    _lib.tg_shutdown()


# ---------------------------------------------------------------- torch form

def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _dev_fp16(t, name):
    if t.dtype.__repr__() != "torch.float16":
        raise TypeError(f"{name} must be float16, got {t.dtype}")
    if not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (row-major)")
    return t.data_ptr()


def gemm(A, B, bias=None, gelu: bool = False, out=None, kernel: int = KERNEL_AUTO, split_k: int = 0,
         stream=None):
    """C = epi(A @ B + bias) for CUDA float16 tensors A (M, K), B (K, N), bias (N,).

    Runs on ``stream`` (default: torch's current stream) and returns ``out``
    (allocated with torch when not given). Asynchronous like any CUDA op.
    """
    import torch
    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[0]:
        raise ValueError(f"shape mismatch {tuple(A.shape)} @ {tuple(B.shape)}")
    M, K = A.shape
    N = B.shape[1]
    if bias is not None and tuple(bias.shape) != (N,):
        raise ValueError(f"bias must have shape ({N},)")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=A.device)
    elif tuple(out.shape) != (M, N):
        raise ValueError("out has the wrong shape")
    pa = _dev_fp16(A, "A") if A.numel() else None
    pb = _dev_fp16(B, "B") if B.numel() else None
    pbias = _dev_fp16(bias, "bias") if bias is not None else None
    pc = _dev_fp16(out, "out") if out.numel() else None
    tg_gemm_ex(pa, pb, pbias, pc, M, N, K, EPI_GELU if gelu else EPI_NONE, kernel, split_k,
               _stream_handle(stream))
    return out


def gemm_w4(A, Bq, scales, bias=None, gelu: bool = False, out=None, split_k: int = 0, stream=None,
            fmt: int = W4_INT4, kernel: int = W4_KERNEL_AUTO):
    """C = epi(A @ W + bias) with 4-bit weights: A (M, K) float16, Bq (N, K/2)
    uint8 (low nibble = even k; two's complement for W4_INT4, E2M1 codes for
    W4_FP4_E2M1), scales (K/128, N) float16, W[k, n] = fp16(value(q[k, n]) *
    scales[k // 128, n]). CUDA tensors, contiguous. `kernel`: W4_KERNEL_AUTO,
    W4_KERNEL_TMEM or W4_KERNEL_REG (M <= 16, one K slice)."""
    import torch
    if A.dim() != 2 or Bq.dim() != 2 or scales.dim() != 2:
        raise ValueError("A, Bq and scales must be matrices")
    M, K = A.shape
    N = Bq.shape[0]
    if 2 * Bq.shape[1] != K:
        raise ValueError(f"Bq must have shape ({N}, {K // 2}), got {tuple(Bq.shape)}")
    if tuple(scales.shape) != (K // 128, N):
        raise ValueError(f"scales must have shape ({K // 128}, {N}), got {tuple(scales.shape)}")
    if Bq.dtype != torch.uint8 or not Bq.is_cuda or not Bq.is_contiguous():
        raise TypeError("Bq must be a contiguous CUDA uint8 tensor")
    if bias is not None and tuple(bias.shape) != (N,):
        raise ValueError(f"bias must have shape ({N},)")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=A.device)
    elif tuple(out.shape) != (M, N):
        raise ValueError("out has the wrong shape")
    tg_gemm_w4_kernel(_dev_fp16(A, "A") if A.numel() else None, Bq.data_ptr() if Bq.numel() else None,
                      _dev_fp16(scales, "scales") if scales.numel() else None,
                      _dev_fp16(bias, "bias") if bias is not None else None,
                      _dev_fp16(out, "out") if out.numel() else None, M, N, K, EPI_GELU if gelu else EPI_NONE, fmt,
                      kernel, split_k, _stream_handle(stream))
    return out


def gemm_staged(hA, hB, hbias, hC, dA, dB, dbias, dC, gelu: bool = False, stream=None) -> None:
    """End-to-end form: host (pinned) tensors hA, hB, hbias are copied into the
    device tensors dA, dB, dbias, the GEMM runs, and the result is copied from dC
    into host hC, all on ``stream``."""
    M, K = hA.shape
    N = hB.shape[1]
    tg_gemm_staged(hA.data_ptr(), hB.data_ptr(), hbias.data_ptr() if hbias is not None else None,
                   hC.data_ptr(), dA.data_ptr(), dB.data_ptr(),
                   dbias.data_ptr() if dbias is not None else None, dC.data_ptr(), M, N, K,
                   EPI_GELU if gelu else EPI_NONE, _stream_handle(stream))


def ring_bytes(block_M: int, block_N: int, block_K: int, num_stages: int, elem_bytes: int = 2) -> int:
    """Shared memory a pipelined tile ring needs: every stage holds one
    block_M x block_K tile of A and one block_K x block_N tile of B
    ("TileLang: you write the dataflow, the compiler owns the schedule",
    section "What a tile costs, exactly")."""
    return num_stages * (block_M * block_K + block_K * block_N) * elem_bytes
