"""CPU oracle for the fp16 GEMM + fused bias/GELU epilogue (test infrastructure).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers. The product package never
imports this module, and this module never imports the product package.

The arithmetic lives in ``oracle.c`` (plain C, fp64): see its header for the
definition followed and the passages it cites ("TileLang: writing LLM GPU
kernels by thinking in tiles", section 2, for C[i,j] = sum_k A[i,k] B[k,j];
"Designing high-performance GPU kernels with TileLang", section 3, for the
GELU(MatMul + Bias) epilogue). This file only builds the shared library and
marshals numpy arrays into it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def compile_source(src: str, out: str) -> str:
    """gcc a copy of the oracle source into a shared library (portable flags only)."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it, unless it is up to date."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    return compile_source(_SRC, _LIB_PATH)


def _bind(lib):
    u16p = ctypes.POINTER(ctypes.c_uint16)
    f64p = ctypes.POINTER(ctypes.c_double)
    i64p = ctypes.POINTER(ctypes.c_int64)
    i64 = ctypes.c_int64
    lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_half_to_double.restype = ctypes.c_double
    lib.oracle_double_to_half.argtypes = [ctypes.c_double]
    lib.oracle_double_to_half.restype = ctypes.c_uint16
    lib.oracle_gelu.argtypes = [ctypes.c_double]
    lib.oracle_gelu.restype = ctypes.c_double
    lib.oracle_gemm_rows.argtypes = [u16p, u16p, u16p, u16p, f64p, i64, i64, i64,
                                     ctypes.c_int, i64, i64, ctypes.c_int]
    lib.oracle_gemm_rows.restype = ctypes.c_int
    lib.oracle_gemm_sampled.argtypes = [u16p, u16p, u16p, i64, i64, i64, ctypes.c_int,
                                        i64p, i64p, i64, u16p, f64p, ctypes.c_int]
    lib.oracle_gemm_sampled.restype = ctypes.c_int
    u8p = ctypes.POINTER(ctypes.c_uint8)
    lib.oracle_int4_value.argtypes = [ctypes.c_uint8, ctypes.c_int]
    lib.oracle_int4_value.restype = ctypes.c_int
    lib.oracle_dequant_w4.argtypes = [u8p, u16p, u16p, i64, i64, i64]
    lib.oracle_dequant_w4.restype = ctypes.c_int
    lib.oracle_gemm_w4_rows.argtypes = [u16p, u8p, u16p, u16p, u16p, f64p, i64, i64, i64, i64, ctypes.c_int,
                                        i64, i64, ctypes.c_int]
    lib.oracle_gemm_w4_rows.restype = ctypes.c_int
    lib.oracle_e2m1_value.argtypes = [ctypes.c_uint8, ctypes.c_int]
    lib.oracle_e2m1_value.restype = ctypes.c_double
    lib.oracle_dequant_w4f.argtypes = [u8p, u16p, u16p, i64, i64, i64, ctypes.c_int]
    lib.oracle_dequant_w4f.restype = ctypes.c_int
    lib.oracle_gemm_w4f_rows.argtypes = [u16p, u8p, u16p, u16p, u16p, f64p, i64, i64, i64, i64, ctypes.c_int,
                                         ctypes.c_int, i64, i64, ctypes.c_int]
    lib.oracle_gemm_w4f_rows.restype = ctypes.c_int
    lib.oracle_attention_rows.argtypes = [u16p, u16p, u16p, u16p, f64p, i64, i64, i64, i64, ctypes.c_int,
                                          ctypes.c_double, i64p, i64, ctypes.c_int]
    lib.oracle_attention_rows.restype = ctypes.c_int
    lib.oracle_softmax_rows.argtypes = [u16p, u16p, f64p, i64, i64, i64, i64, ctypes.c_int]
    lib.oracle_softmax_rows.restype = ctypes.c_int
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def _bits(x) -> np.ndarray:
    """A C-contiguous uint16 view of binary16 data (np.float16 or uint16 input,
    or a CPU torch.float16 tensor)."""
    if x is None:
        return None
    if hasattr(x, "numpy") and hasattr(x, "dtype") and not isinstance(x, np.ndarray):
        x = x.detach().contiguous().view(dtype=_torch_int16()).numpy()
    x = np.ascontiguousarray(x)
    if x.dtype == np.float16 or x.dtype == np.int16:
        x = x.view(np.uint16)
    if x.dtype != np.uint16:
        raise TypeError(f"expected binary16 data, got {x.dtype}")
    return x


def _torch_int16():
    import torch
    return torch.int16


def _ptr(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


class Oracle:
    """The oracle's entry points bound to one build of oracle.c."""

    def __init__(self, lib):
        self._lib = lib

    def half_to_double(self, h: int) -> float:
        return self._lib.oracle_half_to_double(int(h) & 0xFFFF)

    def double_to_half(self, x: float) -> int:
        return int(self._lib.oracle_double_to_half(float(x)))

    def gelu(self, x: float) -> float:
        return self._lib.oracle_gelu(float(x))

    def max_threads(self) -> int:
        return int(self._lib.oracle_max_threads())

    def gemm(self, A, B, bias=None, gelu: bool = False, rows: tuple[int, int] | None = None,
             want_f64: bool = False, threads: int = 0):
        """C = epi(A @ B + bias) in fp64, rounded once to binary16.

        A: (M, K), B: (K, N), bias: (N,) or None; binary16 data (np.float16/uint16
        arrays or CPU float16 tensors). ``rows=(r0, n)`` computes only rows
        r0..r0+n-1. Returns C as np.float16 (n, N), plus the fp64 values before
        rounding when ``want_f64``.
        """
        a, b, c = _bits(A), _bits(B), _bits(bias)
        if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[0]:
            raise ValueError(f"shape mismatch {a.shape} @ {b.shape}")
        M, K = a.shape
        N = b.shape[1]
        if c is not None and c.shape != (N,):
            raise ValueError(f"bias must have shape ({N},), got {c.shape}")
        r0, nr = (0, M) if rows is None else rows
        out = np.empty((nr, N), dtype=np.uint16)
        out64 = np.empty((nr, N), dtype=np.float64) if want_f64 else None
        rc = self._lib.oracle_gemm_rows(_ptr(a, ctypes.c_uint16), _ptr(b, ctypes.c_uint16),
                                      _ptr(c, ctypes.c_uint16), _ptr(out, ctypes.c_uint16),
                                      _ptr(out64, ctypes.c_double), M, N, K, int(bool(gelu)),
                                      r0, nr, int(threads))
        if rc != 0:
            raise RuntimeError("oracle_gemm_rows failed")
        out = out.view(np.float16)
        return (out, out64) if want_f64 else out

    def int4_value(self, byte: int, high: bool) -> int:
        return int(self._lib.oracle_int4_value(int(byte) & 0xFF, 4 if high else 0))

    def e2m1_value(self, byte: int, high: bool) -> float:
        """Value of the FP4 (E2M1) field in the low (or high) nibble of `byte`."""
        return float(self._lib.oracle_e2m1_value(int(byte) & 0xFF, 4 if high else 0))

    def dequant_w4(self, Bq, scales, group: int = 128, fmt: int = 0):
        """W (K x N, np.float16) from Bq (N x K/2 bytes, low nibble = even k):
        value * scale rounded once to binary16; fmt 0 = INT4, 1 = FP4 (E2M1)."""
        q, sc = _u8(Bq), _bits(scales)
        N, half_k = q.shape
        K = 2 * half_k
        W = np.empty((K, N), dtype=np.uint16)
        rc = self._lib.oracle_dequant_w4f(_ptr(q, ctypes.c_uint8), _ptr(sc, ctypes.c_uint16),
                                          _ptr(W, ctypes.c_uint16), N, K, int(group), int(fmt))
        if rc != 0:
            raise RuntimeError("oracle_dequant_w4f failed")
        return W.view(np.float16)

    def gemm_w4(self, A, Bq, scales, bias=None, gelu: bool = False, group: int = 128,
                rows: tuple[int, int] | None = None, want_f64: bool = False, threads: int = 0, fmt: int = 0):
        """C = epi(A @ W + bias) with W the dequantized 4-bit weights (fmt 0 =
        INT4, 1 = FP4 E2M1)."""
        a, q, sc, c = _bits(A), _u8(Bq), _bits(scales), _bits(bias)
        M, K = a.shape
        if 2 * q.shape[1] != K:
            raise ValueError(f"packed weights hold {2 * q.shape[1]} values per row, A has K={K}")
        N = q.shape[0]
        if sc.shape != ((K + group - 1) // group, N):
            raise ValueError(f"scales must have shape ({(K + group - 1) // group}, {N}), got {sc.shape}")
        r0, nr = (0, M) if rows is None else rows
        out = np.empty((nr, N), dtype=np.uint16)
        out64 = np.empty((nr, N), dtype=np.float64) if want_f64 else None
        rc = self._lib.oracle_gemm_w4f_rows(_ptr(a, ctypes.c_uint16), _ptr(q, ctypes.c_uint8),
                                            _ptr(sc, ctypes.c_uint16), _ptr(c, ctypes.c_uint16),
                                            _ptr(out, ctypes.c_uint16), _ptr(out64, ctypes.c_double),
                                            M, N, K, int(group), int(fmt), int(bool(gelu)), r0, nr, int(threads))
        if rc != 0:
            raise RuntimeError("oracle_gemm_w4f_rows failed")
        out = out.view(np.float16)
        return (out, out64) if want_f64 else out

    def attention(self, Q, K, V, causal: bool = False, rows=None, want_f64: bool = False, threads: int = 0):
        """Attention forward O = softmax(Q K^T / sqrt(D)) V on (B, S, H, D)
        binary16 tensors (bshd). rows: flat query indices (b * S + s) * H + h to
        evaluate (default all, returned as (B, S, H, D)); else (len(rows), D)."""
        q, k, v = _bits(Q), _bits(K), _bits(V)
        if q.ndim != 4 or q.shape != k.shape or q.shape != v.shape:
            raise ValueError(f"Q, K, V must share one (B, S, H, D) shape, got {q.shape} {k.shape} {v.shape}")
        B, S, H, D = q.shape
        full = rows is None
        r = np.arange(B * S * H, dtype=np.int64) if full else np.ascontiguousarray(rows, dtype=np.int64)
        out = np.empty((len(r), D), dtype=np.uint16)
        out64 = np.empty((len(r), D), dtype=np.float64) if want_f64 else None
        rc = self._lib.oracle_attention_rows(_ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16),
                                             _ptr(v, ctypes.c_uint16), _ptr(out, ctypes.c_uint16),
                                             _ptr(out64, ctypes.c_double), B, S, H, D, int(bool(causal)),
                                             1.0 / np.sqrt(D) if D > 0 else 1.0, _ptr(r, ctypes.c_int64), len(r),
                                             int(threads))
        if rc != 0:
            raise RuntimeError("oracle_attention_rows failed")
        out = out.view(np.float16)
        if full:
            out = out.reshape(B, S, H, D)
            out64 = out64.reshape(B, S, H, D) if want_f64 else None
        return (out, out64) if want_f64 else out

    def softmax(self, X, rows: tuple[int, int] | None = None, want_f64: bool = False, threads: int = 0):
        """Row softmax of an M x N binary16 matrix, rows [r0, r0 + n) (default all)."""
        x = _bits(X)
        if x.ndim != 2:
            raise ValueError(f"X must be a matrix, got shape {x.shape}")
        M, N = x.shape
        r0, nr = (0, M) if rows is None else rows
        out = np.empty((nr, N), dtype=np.uint16)
        out64 = np.empty((nr, N), dtype=np.float64) if want_f64 else None
        rc = self._lib.oracle_softmax_rows(_ptr(x, ctypes.c_uint16), _ptr(out, ctypes.c_uint16),
                                           _ptr(out64, ctypes.c_double), M, N, r0, nr, int(threads))
        if rc != 0:
            raise RuntimeError("oracle_softmax_rows failed")
        out = out.view(np.float16)
        return (out, out64) if want_f64 else out

    def gemm_sampled(self, A, B, bias, gelu: bool, rows, cols, want_f64: bool = False, threads: int = 0):
        """C[rows[t], cols[t]] for each t, each evaluated from the definition alone."""
        a, b, c = _bits(A), _bits(B), _bits(bias)
        M, K = a.shape
        N = b.shape[1]
        r = np.ascontiguousarray(rows, dtype=np.int64)
        q = np.ascontiguousarray(cols, dtype=np.int64)
        if r.shape != q.shape:
            raise ValueError("rows and cols differ in length")
        out = np.empty(r.shape, dtype=np.uint16)
        out64 = np.empty(r.shape, dtype=np.float64) if want_f64 else None
        rc = self._lib.oracle_gemm_sampled(_ptr(a, ctypes.c_uint16), _ptr(b, ctypes.c_uint16),
                                         _ptr(c, ctypes.c_uint16), M, N, K, int(bool(gelu)),
                                         _ptr(r, ctypes.c_int64), _ptr(q, ctypes.c_int64), r.size,
                                         _ptr(out, ctypes.c_uint16), _ptr(out64, ctypes.c_double),
                                         int(threads))
        if rc != 0:
            raise RuntimeError("oracle_gemm_sampled failed")
        out = out.view(np.float16)
        return (out, out64) if want_f64 else out


def _u8(x) -> np.ndarray:
    if hasattr(x, "numpy") and not isinstance(x, np.ndarray):
        x = x.detach().contiguous().numpy()
    x = np.ascontiguousarray(x)
    if x.dtype == np.int8:
        x = x.view(np.uint8)
    if x.dtype != np.uint8:
        raise TypeError(f"expected packed bytes, got {x.dtype}")
    return x


def load_library(path: str) -> Oracle:
    """Bind an explicitly built copy of the oracle (used by the tests that check
    that the pins reject deliberately broken copies)."""
    return Oracle(_bind(ctypes.CDLL(path)))


class _Default(Oracle):
    def __init__(self):
        pass

    @property
    def _lib(self):
        return _load()


_default = _Default()
half_to_double = _default.half_to_double
double_to_half = _default.double_to_half
gelu = _default.gelu
max_threads = _default.max_threads
gemm = _default.gemm
gemm_sampled = _default.gemm_sampled
int4_value = _default.int4_value
e2m1_value = _default.e2m1_value
dequant_w4 = _default.dequant_w4
gemm_w4 = _default.gemm_w4
attention = _default.attention
softmax = _default.softmax
