"""Exact emulation of fp32 multiply and fused multiply-add in numpy.

Used by the CPU checks of the kernels' division-free arithmetic. For fp32
inputs a, b, c (as float32 arrays):

* a*b is exact in float64 (24 + 24 significant bits);
* a*b + c is split exactly into s + err with TwoSum (s = the float64 sum);
* fp32 rounding of s + err: the float32 cast of s is the nearest-even fp32
  value of s; it differs from the nearest-even value of the exact sum only
  when s lies exactly on an fp32 midpoint (fp32 midpoints are float64 values,
  so none can lie strictly between s and the exact sum), and then the sign
  of err decides.

Valid while nothing overflows and the exact sum is not below 2^-1000 or so
(the float64 TwoSum is exact there); subnormal fp32 results are rounded
correctly (their midpoints are odd multiples of 2^-150).
"""
import numpy as np


def is_f32_midpoint(s: np.ndarray) -> np.ndarray:
    """float64 values exactly halfway between two fp32 neighbours."""
    a = np.abs(s)
    bits = a.view(np.uint64)
    normal = a >= 2.0 ** -126
    mid_n = (bits & np.uint64(0x1FFFFFFF)) == np.uint64(0x10000000)
    k = a * 2.0 ** 150                       # exact: subnormal fp32 midpoints are odd k
    mid_s = (k == np.floor(k)) & (np.mod(k, 2.0) == 1.0)
    return np.where(normal, mid_n, mid_s)


def round_sum32(x: np.ndarray, y: np.ndarray) -> np.ndarray:
    """fp32 nearest-even rounding of the exact sum of float64 arrays x + y."""
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    s = x + y                                        # TwoSum: s + err == x + y
    bb = s - x
    err = (x - (s - bb)) + (y - bb)
    out = s.astype(np.float32)
    fix = is_f32_midpoint(s) & (err != 0.0)
    if np.any(fix):
        up = np.nextafter(out, np.float32(np.inf))
        dn = np.nextafter(out, np.float32(-np.inf))
        want_up = err > 0.0
        out = np.where(fix & want_up & (out.astype(np.float64) < s), up, out)
        out = np.where(fix & ~want_up & (out.astype(np.float64) > s), dn, out)
    return out


def mul32(a, b) -> np.ndarray:
    """RN_fp32(a*b) for fp32 a, b."""
    return (np.asarray(a, np.float32).astype(np.float64) *
            np.asarray(b, np.float32).astype(np.float64)).astype(np.float32)


def fma32(a, b, c) -> np.ndarray:
    """RN_fp32(a*b + c) for fp32 a, b, c, with a single rounding."""
    p = (np.asarray(a, np.float32).astype(np.float64) *
         np.asarray(b, np.float32).astype(np.float64))
    return round_sum32(p, np.asarray(c, np.float32).astype(np.float64))
