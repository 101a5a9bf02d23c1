"""Seeded synthetic bf16 inputs (the shared input source of tests and bench).

Holds no GEMM arithmetic: it only draws normal numbers and rounds them to
bf16 bit patterns (see ``csrc/synthetic.c`` for the exact generator:
SplitMix64 counter stream + Box-Muller, rounded once from f64 to bf16,
nearest-even).

Streams: A (weights) draws from stream 0, B (activations) from stream 1, the
outlier mask of B from stream 2, all under the workload's seed.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import _build

STREAM_A = 0
STREAM_B = 1
STREAM_OUTLIER = 2
STREAM_A_CODES = 3      # packed 4-bit weight codes (A16W4)
STREAM_A_SCALES = 4     # 8-bit scale codes (A16W4)
STREAM_A_CODES8 = 5     # 8-bit E4M3 weight codes (A16W8)
STREAM_A_SCALES8 = 6    # their scale codes

_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(str(_build.build_synthetic()))
        lib.synthetic_normal_bf16.argtypes = [
            ctypes.POINTER(ctypes.c_uint16), ctypes.c_uint64, ctypes.c_uint64,
            ctypes.c_uint64, ctypes.c_uint64, ctypes.c_double, ctypes.c_double,
            ctypes.c_double, ctypes.c_uint64, ctypes.c_int]
        lib.synthetic_normal_bf16.restype = ctypes.c_int
        lib.synthetic_bytes.argtypes = [
            ctypes.POINTER(ctypes.c_uint8), ctypes.c_uint64, ctypes.c_uint64,
            ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint, ctypes.c_uint]
        lib.synthetic_bytes.restype = None
        lib.synthetic_word.argtypes = [ctypes.c_uint64] * 3
        lib.synthetic_word.restype = ctypes.c_uint64
        _lib = lib
    return _lib


def host_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def normal_bf16(shape, seed: int, stream: int, sigma: float,
                outlier_p: float = 0.0, outlier_scale: float = 1.0,
                offset: int = 0, threads: int | None = None,
                out: np.ndarray | None = None) -> np.ndarray:
    """bf16 bit patterns (uint16) of sigma * N(0, 1), C-contiguous ``shape``.

    ``offset`` starts the draw at that element of the stream, so a slice of
    a large tensor can be drawn alone (the values equal those of the full
    draw at the same positions).
    """
    shape = tuple(int(s) for s in (shape if isinstance(shape, (tuple, list)) else (shape,)))
    count = int(np.prod(shape)) if shape else 1
    if out is None:
        out = np.empty(shape, dtype=np.uint16)
    if out.dtype != np.uint16 or not out.flags.c_contiguous or out.size != count:
        raise ValueError("out must be a C-contiguous uint16 array of the shape's size")
    if count:
        _load().synthetic_normal_bf16(
            out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)), int(offset), count,
            int(seed), int(stream), float(sigma), float(outlier_p),
            float(outlier_scale), STREAM_OUTLIER,
            int(threads if threads is not None else host_threads()))
    return out


def word(seed: int, stream: int, i: int) -> int:
    """The i-th raw 64-bit SplitMix64 word of (seed, stream)."""
    return int(_load().synthetic_word(int(seed), int(stream), int(i)))


def uniform_bytes(shape, seed: int, stream: int, lo: int = 0, span: int = 256,
                  offset: int = 0) -> np.ndarray:
    """uint8 array: lo + (SplitMix64 word i of (seed, stream)) mod span."""
    shape = tuple(int(s) for s in (shape if isinstance(shape, (tuple, list)) else (shape,)))
    count = int(np.prod(shape)) if shape else 1
    out = np.empty(shape, dtype=np.uint8)
    if count:
        _load().synthetic_bytes(out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)), int(offset),
                                count, int(seed), int(stream), int(lo), int(span))
    return out


# Scale codes of the A16W4 weights: 2^-9 ... 2^-3, so that the 4-bit
# magnitudes (0 ... 6) span the range of N(0, 0.02)-like weights.
W4_SCALE_LO = 118
W4_SCALE_SPAN = 7


def w4_weights(L: int, N: int, K: int, seed: int):
    """Seeded A16W4 weights: packed E2M1 codes A_q[L][N][K/2] (uniform over
    the 16 codes) and E8M0 scale codes A_s[L][N][K/32]."""
    if K % 32:
        raise ValueError("K must be a multiple of 32 (the scale block)")
    aq = uniform_bytes((L, N, K // 2), seed, STREAM_A_CODES)
    a_s = uniform_bytes((L, N, K // 32), seed, STREAM_A_SCALES, W4_SCALE_LO, W4_SCALE_SPAN)
    return aq, a_s


# Scale codes of the A16W8 weights: 2^-13 ... 2^-7, so that E4M3 magnitudes
# (2^-9 ... 448) land in the range of N(0, 0.02)-like weights.
W8_SCALE_LO = 114
W8_SCALE_SPAN = 7


def w8_weights(L: int, N: int, K: int, seed: int):
    """Seeded A16W8 weights: E4M3 codes A_q[L][N][K] (uniform over the 254
    finite codes: the two not-a-number codes 0x7F and 0xFF become 0x7E and
    0xFE) and E8M0 scale codes A_s[L][N][K/32]."""
    if K % 32:
        raise ValueError("K must be a multiple of 32 (the scale block)")
    aq = uniform_bytes((L, N, K), seed, STREAM_A_CODES8)
    aq[(aq & 0x7F) == 0x7F] ^= 1
    a_s = uniform_bytes((L, N, K // 32), seed, STREAM_A_SCALES8, W8_SCALE_LO, W8_SCALE_SPAN)
    return aq, a_s
