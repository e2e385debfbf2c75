"""Round-to-nearest-even from float64 into the storage formats.

Parameters may be stored as fp32, bf16 or fp16 and 16-bit moments as bf16
("Fused Optimizers and State Precision", section 05, two 16-bit moments). The
pages name no rounding mode; IEEE round-to-nearest-even is the reading used.

Every format is described by three numbers: ``p`` significant bits (including
the implicit one), the exponent of the smallest subnormal (the finest quantum),
and the largest finite value. For a finite x with 2^(e-1) <= |x| < 2^e the
quantum is 2^max(e-p, q_min); the rounded value is rint(x / quantum) * quantum
(rint ties to even), and a result above the largest finite value is infinite.
"""
from __future__ import annotations

import dataclasses

import numpy as np


@dataclasses.dataclass(frozen=True)
class Format:
    name: str
    p: int            # significant bits, implicit bit included
    q_min: int        # exponent of the smallest subnormal
    max_finite: float


FORMATS = {
    "f32": Format("f32", 24, -149, float((2.0 - 2.0 ** -23) * 2.0 ** 127)),
    "bf16": Format("bf16", 8, -133, float((2.0 - 2.0 ** -7) * 2.0 ** 127)),
    "f16": Format("f16", 11, -24, 65504.0),
    "f64": None,
}


def round_to(x, fmt: str) -> np.ndarray:
    """Round float64 values to the nearest ``fmt`` value, ties to even.

    Returns float64 holding exactly representable values of ``fmt``.
    NaN stays NaN, infinities and signed zeros are kept.
    """
    x = np.array(x, dtype=np.float64, copy=True)
    f = FORMATS[fmt]
    if f is None:
        return x
    sel = np.isfinite(x) & (x != 0.0)
    xs = x[sel]
    _, e = np.frexp(xs)                       # |xs| in [2^(e-1), 2^e)
    qexp = np.maximum(e - f.p, f.q_min)       # exponent of one unit in the last place
    y = np.ldexp(np.rint(np.ldexp(xs, -qexp)), qexp)
    over = np.abs(y) > f.max_finite
    y[over] = np.copysign(np.inf, y[over])
    x[sel] = y
    return x


def representable(x, fmt: str) -> bool:
    """True when every value of ``x`` is exactly a ``fmt`` value."""
    x = np.asarray(x, dtype=np.float64)
    r = round_to(x, fmt)
    same = (r == x) | (np.isnan(r) & np.isnan(x))
    return bool(np.all(same))
