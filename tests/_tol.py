"""The parity tolerance between the GPU result and the oracle.

An element passes when either bound holds:
  * |gpu - oracle| <= one bf16 ulp at |oracle| (for 2^e <= |x| < 2^(e+1)
    the spacing is 2^(e-7); below 2^-126 it is 2^-133), or
  * |gpu - oracle| <= 1e-3 * sqrt(K) * max|A| * max|B| (outputs near zero).
+0 and -0 compare equal.  NaN or Inf on either side fails.
"""
from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    ulp = np.exp2(e - 7)
    return np.where(ax >= 2.0 ** -126, ulp, 2.0 ** -133)


def abs_bound(K: int, max_a: float, max_b: float) -> float:
    return 1e-3 * np.sqrt(K) * max_a * max_b


def check(gpu_bits, oracle_bits, K: int, max_a: float, max_b: float):
    """Returns (ok, report) for two arrays of bf16 bit patterns."""
    g = bf16_bits_to_f64(gpu_bits)
    o = bf16_bits_to_f64(oracle_bits)
    if not np.all(np.isfinite(g)):
        bad = np.flatnonzero(~np.isfinite(g))[:8]
        return False, f"non-finite GPU outputs at {bad.tolist()}"
    err = np.abs(g - o)
    ok = (err <= bf16_ulp(o)) | (err <= abs_bound(K, max_a, max_b))
    if ok.all():
        return True, f"max|err|={err.max() if err.size else 0.0:.3g}"
    bad = np.flatnonzero(~ok)
    i = bad[0]
    return False, (f"{bad.size} of {ok.size} elements out of tolerance; first at "
                   f"flat {i}: gpu={g.flat[i]!r} oracle={o.flat[i]!r}")


def max_abs_bf16(bits) -> float:
    v = bf16_bits_to_f64(bits)
    return float(np.max(np.abs(v))) if v.size else 0.0
