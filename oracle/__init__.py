"""fp64 CPU oracle for the weight-streaming GEMV (test infrastructure).

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference
leg may import this package. The arithmetic lives in ``oracle.c`` (plain C,
fp64, scalar nibble unpacking); this module compiles it with gcc and wraps it
with ctypes. It imports nothing from the CUDA package.

All arrays are numpy; bf16 / fp16 values travel as their uint16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_CFLAGS = ["-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-std=c11"]


def build(src: str = _SRC, out: str = _LIB, extra_flags: tuple = ()) -> str:
    """Compile oracle.c (or a variant of it) into a shared library; returns its path."""
    cmd = ["gcc", *_CFLAGS, *extra_flags, src, "-o", out + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def _needs_build() -> bool:
    return not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)


_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def load(path: str | None = None) -> "Oracle":
    """The oracle library at `path` (default: the built oracle.c)."""
    global _lib
    if path is not None:
        return Oracle(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if _needs_build():
                build()
            _lib = Oracle(ctypes.CDLL(_LIB))
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags.c_contiguous
    return a.ctypes.data


class Oracle:
    """Typed numpy wrappers over one loaded oracle library."""

    def __init__(self, lib: ctypes.CDLL):
        self.lib = lib
        lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_double.restype = ctypes.c_double
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_double_to_bf16_rne.argtypes = [ctypes.c_double]
        lib.oracle_double_to_bf16_rne.restype = ctypes.c_uint16
        lib.oracle_dequant_int4_g64.argtypes = [_P, _P, _I64, _I64, _P]
        lib.oracle_dequant_int4_awq_g128.argtypes = [_P, _P, _P, _I64, _I64, _P]
        lib.oracle_gemm_bf16.argtypes = [_P, _P, _I64, _I64, _I64, _P, _P]
        lib.oracle_gemm_int4_g64.argtypes = [_P, _P, _P, _I64, _I64, _I64, _P, _P]
        lib.oracle_gemm_int4_awq_g128.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _P, _P]
        lib.oracle_gemm_int4_awq_g128_repacked.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _P, _P]
        lib.oracle_repack_int4.argtypes = [_P, _I64, _I64, _P]
        lib.oracle_gemm_int8_pc.argtypes = [_P, _P, _P, _I64, _I64, _I64, _P, _P]
        lib.oracle_quantize_int8_pc.argtypes = [_P, _I64, _I64, _P, _P]
        lib.oracle_rmsnorm_bf16.argtypes = [_P, _P, _I64, _I64, ctypes.c_double, _P]
        lib.oracle_rmsnorm_f64.argtypes = [_P, _P, _I64, _I64, ctypes.c_double, _P]
        lib.oracle_swiglu.argtypes = [_P, _P, _I64, _P]
        lib.oracle_add_residual.argtypes = [_P, _P, _I64, _P]
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        for f in ("oracle_dequant_int4_g64", "oracle_dequant_int4_awq_g128", "oracle_gemm_bf16",
                  "oracle_gemm_int4_g64", "oracle_gemm_int4_awq_g128", "oracle_gemm_int4_awq_g128_repacked",
                  "oracle_repack_int4", "oracle_gemm_int8_pc",
                  "oracle_quantize_int8_pc", "oracle_rmsnorm_bf16", "oracle_rmsnorm_f64", "oracle_swiglu", "oracle_add_residual",
                  "oracle_set_num_threads"):
            getattr(lib, f).restype = None

    # ---- scalar formats
    def f16_to_double(self, h: int) -> float:
        return self.lib.oracle_f16_to_double(int(h))

    def bf16_to_double(self, b: int) -> float:
        return self.lib.oracle_bf16_to_double(int(b))

    def double_to_bf16(self, v: float) -> int:
        return int(self.lib.oracle_double_to_bf16_rne(float(v)))

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def set_num_threads(self, n: int) -> None:
        self.lib.oracle_set_num_threads(int(n))

    # ---- dequant
    def dequant_int4_g64(self, codes: np.ndarray, scales: np.ndarray, N: int, K: int) -> np.ndarray:
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        scales = np.ascontiguousarray(scales, dtype=np.uint16)
        assert codes.size == N * K // 2 and scales.size == N * K // 64
        out = np.empty((N, K), dtype=np.float64)
        self.lib.oracle_dequant_int4_g64(_ptr(codes), _ptr(scales), N, K, _ptr(out))
        return out

    def dequant_int4_awq_g128(self, codes, scales, zeros, N: int, K: int) -> np.ndarray:
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        scales = np.ascontiguousarray(scales, dtype=np.uint16)
        zeros = np.ascontiguousarray(zeros, dtype=np.uint8)
        G = K // 128
        assert codes.size == N * K // 2 and scales.size == N * G and zeros.size == N * ((G + 1) // 2)
        out = np.empty((N, K), dtype=np.float64)
        self.lib.oracle_dequant_int4_awq_g128(_ptr(codes), _ptr(scales), _ptr(zeros), N, K, _ptr(out))
        return out

    # ---- products: return (Y, Yabs), each (M, N) float64
    def gemm_bf16(self, W: np.ndarray, X: np.ndarray):
        W = np.ascontiguousarray(W, dtype=np.uint16)
        X = np.ascontiguousarray(np.atleast_2d(X), dtype=np.uint16)
        N, K = W.shape
        M = X.shape[0]
        assert X.shape[1] == K
        Y = np.empty((M, N), dtype=np.float64)
        A = np.empty((M, N), dtype=np.float64)
        self.lib.oracle_gemm_bf16(_ptr(W), _ptr(X), M, N, K, _ptr(Y), _ptr(A))
        return Y, A

    def gemm_int4_g64(self, codes: np.ndarray, scales: np.ndarray, X: np.ndarray):
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        scales = np.ascontiguousarray(scales, dtype=np.uint16)
        X = np.ascontiguousarray(np.atleast_2d(X), dtype=np.uint16)
        M, K = X.shape
        N = codes.shape[0]
        assert codes.shape == (N, K // 2) and scales.shape == (N, K // 64)
        Y = np.empty((M, N), dtype=np.float64)
        A = np.empty((M, N), dtype=np.float64)
        self.lib.oracle_gemm_int4_g64(_ptr(codes), _ptr(scales), _ptr(X), M, N, K, _ptr(Y), _ptr(A))
        return Y, A

    def gemm_int4_awq_g128(self, codes, scales, zeros, X: np.ndarray, repacked: bool = False):
        """codes uint8 (N, K/2) (canonical, or the load-time repacked layout when
        `repacked`), scales fp16 bits (N, K/128), zeros uint8 (N, (K/128+1)/2),
        X bf16 bits (M, K) or (K,) -> (Y, Yabs), each (M, N)."""
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        scales = np.ascontiguousarray(scales, dtype=np.uint16)
        zeros = np.ascontiguousarray(zeros, dtype=np.uint8)
        X = np.ascontiguousarray(np.atleast_2d(X), dtype=np.uint16)
        M, K = X.shape
        N = codes.shape[0]
        G = K // 128
        assert codes.shape == (N, K // 2) and scales.shape == (N, G) and zeros.shape == (N, (G + 1) // 2)
        Y = np.empty((M, N), dtype=np.float64)
        A = np.empty((M, N), dtype=np.float64)
        fn = self.lib.oracle_gemm_int4_awq_g128_repacked if repacked else self.lib.oracle_gemm_int4_awq_g128
        fn(_ptr(codes), _ptr(scales), _ptr(zeros), _ptr(X), M, N, K, _ptr(Y), _ptr(A))
        return Y, A

    def repack_int4(self, codes: np.ndarray) -> np.ndarray:
        """Canonical INT4 codes uint8 (N, K/2), K % 8 == 0 -> the load-time repacked layout."""
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        N, half = codes.shape
        K = 2 * half
        assert K % 8 == 0
        out = np.empty_like(codes)
        self.lib.oracle_repack_int4(_ptr(codes), N, K, _ptr(out))
        return out

    # ---- symmetric INT8, per-output-channel scale
    def gemm_int8_pc(self, codes, scales, X: np.ndarray):
        """codes int8 (N, K), scales float32 (N,), X bf16 bits (M, K) or (K,) -> (Y, Yabs), each (M, N)."""
        codes = np.ascontiguousarray(codes, dtype=np.int8)
        scales = np.ascontiguousarray(scales, dtype=np.float32)
        X = np.ascontiguousarray(np.atleast_2d(X), dtype=np.uint16)
        M, K = X.shape
        N = codes.shape[0]
        assert codes.shape == (N, K) and scales.shape == (N,)
        Y = np.empty((M, N), dtype=np.float64)
        A = np.empty((M, N), dtype=np.float64)
        self.lib.oracle_gemm_int8_pc(_ptr(codes), _ptr(scales), _ptr(X), M, N, K, _ptr(Y), _ptr(A))
        return Y, A

    def quantize_int8_pc(self, W: np.ndarray):
        """W bf16 bits (N, K) -> (codes int8 (N, K), scales float32 (N,))."""
        W = np.ascontiguousarray(W, dtype=np.uint16)
        N, K = W.shape
        Q = np.empty((N, K), dtype=np.int8)
        S = np.empty((N,), dtype=np.float32)
        self.lib.oracle_quantize_int8_pc(_ptr(W), N, K, _ptr(Q), _ptr(S))
        return Q, S

    # ---- fusions around the GEMV
    def rmsnorm_bf16(self, X: np.ndarray, G: np.ndarray, eps: float):
        """X bf16 bits (M, K) or (K,), G bf16 bits (K,) -> Xn bf16 bits, same shape as X."""
        X = np.ascontiguousarray(X, dtype=np.uint16)
        shape = X.shape
        X2 = np.atleast_2d(X)
        M, K = X2.shape
        G = np.ascontiguousarray(G, dtype=np.uint16)
        assert G.shape == (K,)
        out = np.empty((M, K), dtype=np.uint16)
        self.lib.oracle_rmsnorm_bf16(_ptr(X2), _ptr(G), M, K, float(eps), _ptr(out))
        return out.reshape(shape)

    def rmsnorm_f64(self, X: np.ndarray, G: np.ndarray, eps: float):
        """X bf16 bits (M, K) or (K,), G bf16 bits (K,) -> the normalised values
        x * g / sqrt(mean(x^2) + eps) in float64, before the bf16 rounding."""
        X = np.ascontiguousarray(X, dtype=np.uint16)
        shape = X.shape
        X2 = np.atleast_2d(X)
        M, K = X2.shape
        G = np.ascontiguousarray(G, dtype=np.uint16)
        assert G.shape == (K,)
        out = np.empty((M, K), dtype=np.float64)
        self.lib.oracle_rmsnorm_f64(_ptr(X2), _ptr(G), M, K, float(eps), _ptr(out))
        return out.reshape(shape)

    def swiglu(self, A: np.ndarray, B: np.ndarray):
        """silu(A) * B elementwise (float64 arrays of one shape)."""
        A = np.ascontiguousarray(A, dtype=np.float64)
        B = np.ascontiguousarray(B, dtype=np.float64)
        assert A.shape == B.shape
        out = np.empty_like(A)
        self.lib.oracle_swiglu(_ptr(A), _ptr(B), A.size, _ptr(out))
        return out

    def add_residual(self, Y: np.ndarray, R: np.ndarray):
        """Y (float64) + R (bf16 bits), elementwise."""
        Y = np.ascontiguousarray(Y, dtype=np.float64)
        R = np.ascontiguousarray(R, dtype=np.uint16)
        assert Y.shape == R.shape
        out = np.empty_like(Y)
        self.lib.oracle_add_residual(_ptr(Y), _ptr(R), Y.size, _ptr(out))
        return out
