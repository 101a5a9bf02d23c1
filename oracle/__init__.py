"""CPU oracle for the split-K BF16 decode GEMM -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the package
``split_bf16_gemm_swapped_gb300``) never imports, calls or links it, and the
two share no code: the oracle is plain C in ``splitk_oracle.c`` (float64
accumulation, one round-to-nearest-even to bf16), loaded here through ctypes.

Definition (module docstring of the vLLM ``splitk`` API page, SplitKGemm and
its ``kernel`` / ``epilog_warp`` methods):

    C[l, m, n] = RNE_bf16( sum_k f64(A[l, n, k]) * f64(B[l, m, k]) )

with A[L, N, K] the weights, B[L, M, K] the tokens, C[L, M, N]; all bf16,
passed here as uint16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "splitk_oracle.c"
_LIB = _HERE / "_lib" / "liboracle.so"

_lib = None


def build(force: bool = False) -> Path:
    """Compile splitk_oracle.c with gcc into oracle/_lib/liboracle.so."""
    _LIB.parent.mkdir(parents=True, exist_ok=True)
    if force or not _LIB.exists() or _LIB.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = _LIB.with_suffix(f".{os.getpid()}.tmp")
        cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-fPIC", "-shared",
               "-pthread", str(_SRC), "-o", str(tmp), "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(str(_LIB))
    u16p = ctypes.POINTER(ctypes.c_uint16)
    i64 = ctypes.c_int64
    lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f64.restype = ctypes.c_double
    lib.oracle_f64_to_bf16.argtypes = [ctypes.c_double]
    lib.oracle_f64_to_bf16.restype = ctypes.c_uint16
    lib.oracle_dot_f64.argtypes = [u16p, u16p, i64, i64, i64, i64, i64, i64]
    lib.oracle_dot_f64.restype = ctypes.c_double
    lib.oracle_element.argtypes = [u16p, u16p, i64, i64, i64, i64, i64, i64]
    lib.oracle_element.restype = ctypes.c_uint16
    lib.oracle_elements.argtypes = [u16p, u16p, u16p, i64, i64, i64, i64,
                                    ctypes.POINTER(ctypes.c_int64), i64]
    lib.oracle_elements.restype = None
    lib.oracle_gemm.argtypes = [u16p, u16p, u16p, i64, i64, i64, i64]
    lib.oracle_gemm.restype = None
    lib.oracle_gemm_threaded.argtypes = [u16p, u16p, u16p, i64, i64, i64, i64,
                                         ctypes.c_int]
    lib.oracle_gemm_bias.argtypes = [u16p, u16p, u16p, u16p, i64, i64, i64, i64]
    lib.oracle_gemm_bias.restype = None
    lib.oracle_gemm_threaded.restype = ctypes.c_int
    u8p = ctypes.POINTER(ctypes.c_uint8)
    f64p = ctypes.POINTER(ctypes.c_double)
    lib.oracle_e2m1_to_f64.argtypes = [ctypes.c_uint]
    lib.oracle_e2m1_to_f64.restype = ctypes.c_double
    lib.oracle_e8m0_to_f64.argtypes = [ctypes.c_uint]
    lib.oracle_e8m0_to_f64.restype = ctypes.c_double
    lib.oracle_w4_dequant.argtypes = [u8p, u8p, f64p, i64, i64, i64]
    lib.oracle_w4_dequant.restype = None
    lib.oracle_gemm_w4a16.argtypes = [u8p, u8p, u16p, u16p, i64, i64, i64, i64]
    lib.oracle_gemm_w4a16.restype = None
    lib.oracle_w4_elements.argtypes = [u8p, u8p, u16p, u16p, i64, i64, i64, i64,
                                       ctypes.POINTER(ctypes.c_int64), i64]
    lib.oracle_w4_elements.restype = None
    lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint]
    lib.oracle_e4m3_to_f64.restype = ctypes.c_double
    lib.oracle_w8_dequant.argtypes = [u8p, u8p, f64p, i64, i64, i64]
    lib.oracle_w8_dequant.restype = None
    lib.oracle_gemm_w8a16.argtypes = [u8p, u8p, u16p, u16p, i64, i64, i64, i64]
    lib.oracle_gemm_w8a16.restype = None
    _lib = lib
    return lib


def _u16(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 operands are passed as uint16 bit patterns")
    return a


def _ptr(a: np.ndarray, ctype=ctypes.c_uint16):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def bf16_to_f64(h: int) -> float:
    return _load().oracle_bf16_to_f64(int(h) & 0xFFFF)


def f64_to_bf16(x: float) -> int:
    return int(_load().oracle_f64_to_bf16(float(x)))


def _shape(A: np.ndarray, B: np.ndarray):
    if A.ndim == 2:
        A = A[None]
    if B.ndim == 2:
        B = B[None]
    L, N, K = A.shape
    Lb, M, Kb = B.shape
    if (Lb, Kb) != (L, K):
        raise ValueError(f"shape mismatch A{A.shape} B{B.shape}")
    return A, B, M, N, K, L


def gemm(A: np.ndarray, B: np.ndarray, threads: int = 1) -> np.ndarray:
    """C[L, M, N] (uint16 bf16 bits) for A[L, N, K], B[L, M, K] (2-D = L of 1)."""
    squeeze = A.ndim == 2
    A, B, M, N, K, L = _shape(_u16(A), _u16(B))
    A = np.ascontiguousarray(A)
    B = np.ascontiguousarray(B)
    C = np.empty((L, M, N), dtype=np.uint16)
    if threads <= 1:
        _load().oracle_gemm(_ptr(A), _ptr(B), _ptr(C), M, N, K, L)
    else:
        _load().oracle_gemm_threaded(_ptr(A), _ptr(B), _ptr(C), M, N, K, L,
                                     int(threads))
    return C[0] if squeeze else C


def gemm_bias(A: np.ndarray, B: np.ndarray, bias: np.ndarray) -> np.ndarray:
    """C[L, M, N] = RNE(sum_k A[l,n,k] B[l,m,k] + bias[l,n]), float64 then one rounding."""
    squeeze = A.ndim == 2
    A, B, M, N, K, L = _shape(_u16(A), _u16(B))
    A = np.ascontiguousarray(A)
    B = np.ascontiguousarray(B)
    bias = np.ascontiguousarray(_u16(bias)).reshape(L, N)
    C = np.empty((L, M, N), dtype=np.uint16)
    _load().oracle_gemm_bias(_ptr(A), _ptr(B), _ptr(bias), _ptr(C), M, N, K, L)
    return C[0] if squeeze else C


def gemm_threaded(A: np.ndarray, B: np.ndarray, threads: int):
    """Like gemm(); also returns the number of host threads actually used."""
    A, B, M, N, K, L = _shape(_u16(A), _u16(B))
    A = np.ascontiguousarray(A)
    B = np.ascontiguousarray(B)
    C = np.empty((L, M, N), dtype=np.uint16)
    used = _load().oracle_gemm_threaded(_ptr(A), _ptr(B), _ptr(C), M, N, K, L,
                                        int(threads))
    return C, int(used)


def elements(A: np.ndarray, B: np.ndarray, flat_idx) -> np.ndarray:
    """Selected outputs, flat index l*M*N + m*N + n, each computed alone."""
    A, B, M, N, K, L = _shape(_u16(A), _u16(B))
    A = np.ascontiguousarray(A)
    B = np.ascontiguousarray(B)
    idx = np.ascontiguousarray(np.asarray(flat_idx, dtype=np.int64))
    out = np.empty(idx.shape[0], dtype=np.uint16)
    _load().oracle_elements(_ptr(A), _ptr(B), _ptr(out), M, N, K, L,
                            _ptr(idx, ctypes.c_int64), idx.shape[0])
    return out


def dot_f64(A: np.ndarray, B: np.ndarray, l: int, m: int, n: int) -> float:
    """The unrounded float64 sum behind C[l, m, n]."""
    A, B, M, N, K, L = _shape(_u16(A), _u16(B))
    A = np.ascontiguousarray(A)
    B = np.ascontiguousarray(B)
    return float(_load().oracle_dot_f64(_ptr(A), _ptr(B), M, N, K, l, m, n))


# --------------------------------------------------------------------------
# A16W4: E2M1 weights with E8M0 scales per 32 k, bf16 activations
# --------------------------------------------------------------------------
def e2m1_to_f64(code: int) -> float:
    return _load().oracle_e2m1_to_f64(int(code) & 0xF)


def e8m0_to_f64(code: int) -> float:
    return _load().oracle_e8m0_to_f64(int(code) & 0xFF)


def _w4_shape(Aq: np.ndarray, As: np.ndarray, B: np.ndarray):
    Aq = np.ascontiguousarray(Aq, dtype=np.uint8)
    As = np.ascontiguousarray(As, dtype=np.uint8)
    B = _u16(B)
    if Aq.ndim == 2:
        Aq, As, B = Aq[None], As[None], B[None]
    L, N, K2 = Aq.shape
    K = 2 * K2
    Lb, M, Kb = B.shape
    if (Lb, Kb) != (L, K) or As.shape != (L, N, K // 32) or K % 32:
        raise ValueError(f"shape mismatch Aq{Aq.shape} As{As.shape} B{B.shape}")
    return Aq, As, np.ascontiguousarray(B), M, N, K, L


def w4_dequant(Aq: np.ndarray, As: np.ndarray) -> np.ndarray:
    """The float64 weights W[L, N, K] that A_q, A_s encode."""
    squeeze = Aq.ndim == 2
    Aq = np.ascontiguousarray(Aq, dtype=np.uint8)
    As = np.ascontiguousarray(As, dtype=np.uint8)
    if squeeze:
        Aq, As = Aq[None], As[None]
    L, N, K2 = Aq.shape
    W = np.empty((L, N, 2 * K2), dtype=np.float64)
    _load().oracle_w4_dequant(_ptr(Aq, ctypes.c_uint8), _ptr(As, ctypes.c_uint8),
                              _ptr(W, ctypes.c_double), N, 2 * K2, L)
    return W[0] if squeeze else W


def gemm_w4a16(Aq: np.ndarray, As: np.ndarray, B: np.ndarray) -> np.ndarray:
    """C[L, M, N] bf16 bits = RNE(sum_k w[l,n,k] * B[l,m,k]) in float64."""
    squeeze = np.asarray(Aq).ndim == 2
    Aq, As, B, M, N, K, L = _w4_shape(Aq, As, B)
    C = np.empty((L, M, N), dtype=np.uint16)
    _load().oracle_gemm_w4a16(_ptr(Aq, ctypes.c_uint8), _ptr(As, ctypes.c_uint8), _ptr(B), _ptr(C),
                              M, N, K, L)
    return C[0] if squeeze else C


def w4_elements(Aq: np.ndarray, As: np.ndarray, B: np.ndarray, flat_idx) -> np.ndarray:
    """Selected A16W4 outputs, flat index l*M*N + m*N + n, each computed alone."""
    Aq, As, B, M, N, K, L = _w4_shape(Aq, As, B)
    idx = np.ascontiguousarray(np.asarray(flat_idx, dtype=np.int64))
    out = np.empty(idx.shape[0], dtype=np.uint16)
    _load().oracle_w4_elements(_ptr(Aq, ctypes.c_uint8), _ptr(As, ctypes.c_uint8), _ptr(B), _ptr(out),
                               M, N, K, L, _ptr(idx, ctypes.c_int64), idx.shape[0])
    return out


# --------------------------------------------------------------------------
# A16W8: E4M3 weights with E8M0 scales per 32 k, bf16 activations
# --------------------------------------------------------------------------
def e4m3_to_f64(code: int) -> float:
    return _load().oracle_e4m3_to_f64(int(code) & 0xFF)


def _w8_shape(Aq: np.ndarray, As: np.ndarray, B: np.ndarray):
    Aq = np.ascontiguousarray(Aq, dtype=np.uint8)
    As = np.ascontiguousarray(As, dtype=np.uint8)
    B = _u16(B)
    if Aq.ndim == 2:
        Aq, As, B = Aq[None], As[None], B[None]
    L, N, K = Aq.shape
    Lb, M, Kb = B.shape
    if (Lb, Kb) != (L, K) or As.shape != (L, N, K // 32) or K % 32:
        raise ValueError(f"shape mismatch Aq{Aq.shape} As{As.shape} B{B.shape}")
    return Aq, As, np.ascontiguousarray(B), M, N, K, L


def w8_dequant(Aq: np.ndarray, As: np.ndarray) -> np.ndarray:
    """The float64 weights W[L, N, K] that the E4M3 codes A_q and scales A_s encode."""
    squeeze = Aq.ndim == 2
    Aq = np.ascontiguousarray(Aq, dtype=np.uint8)
    As = np.ascontiguousarray(As, dtype=np.uint8)
    if squeeze:
        Aq, As = Aq[None], As[None]
    L, N, K = Aq.shape
    W = np.empty((L, N, K), dtype=np.float64)
    _load().oracle_w8_dequant(_ptr(Aq, ctypes.c_uint8), _ptr(As, ctypes.c_uint8),
                              _ptr(W, ctypes.c_double), N, K, L)
    return W[0] if squeeze else W


def gemm_w8a16(Aq: np.ndarray, As: np.ndarray, B: np.ndarray) -> np.ndarray:
    """C[L, M, N] bf16 bits = RNE(sum_k w[l,n,k] * B[l,m,k]) in float64, 8-bit weights."""
    squeeze = np.asarray(Aq).ndim == 2
    Aq, As, B, M, N, K, L = _w8_shape(Aq, As, B)
    C = np.empty((L, M, N), dtype=np.uint16)
    _load().oracle_gemm_w8a16(_ptr(Aq, ctypes.c_uint8), _ptr(As, ctypes.c_uint8), _ptr(B), _ptr(C),
                              M, N, K, L)
    return C[0] if squeeze else C
