"""Block-wise signed 8-bit moment codec.

"Fused Optimizers and State Precision", section 05, teaching codec: a block of
moment values shares one scale, scale = max|x| / 127, each value is stored as
the signed 8-bit code q = round(x / scale) and restored as q * scale; all-zero
blocks are handled separately. The benchmark page's state-memory figure for the
8-bit optimizer (47.101 MB for 24,313,856 params over 392 tensors) matches
blocks of 256 elements with one fp32 scale per block per moment.

Readings (the pages fix none of these):

* Blocks are 256 consecutive elements of a tensor's flat order, restarting at
  every tensor; the last block of a tensor is ragged and scaled over its own
  elements only.
* The scale is the fp32 quotient absmax/127 and the code is rint of the fp32
  quotient x/scale, ties to even, clamped to [-127, 127]. Because a float
  result here decides an integer code, the decision is taken in fp32, the
  precision of the GPU kernel: ``x`` is first rounded to fp32.
* "Handled separately": a block whose absmax is 0 stores scale 0 and codes 0,
  with no division; it decodes to exact zeros.
* A block holding a NaN or an infinity cannot be coded. It stores its absmax
  (NaN or +inf) as the scale and zero codes, so it decodes to NaN everywhere
  (0 * inf and 0 * NaN are NaN): non-finite values propagate, none is masked.
* The same signed codec serves both moments; codes of the second moment are
  therefore in [0, 127].
* Decoding q * scale is exact in float64.

Variant (section 05 says real 8-bit optimizers differ from the teaching
codec): the second moment is never negative, so an unsigned codec spends the
sign bit on resolution: scale = max|x| / 255, q = rint(x / scale) clamped to
[0, 255] as an unsigned byte, with the same zero-block, non-finite and fp32
decision rules (``encode_unsigned`` / ``decode_unsigned``).
"""
from __future__ import annotations

import numpy as np

from .formats import round_to

BLOCK = 256
QMAX = 127
UQMAX = 255


def n_blocks(n: int, block: int = BLOCK) -> int:
    return -(-int(n) // block)


def _encode_linear(x, block, qmin, qmax, code_dtype):
    x32 = round_to(np.asarray(x, dtype=np.float64).reshape(-1), "f32").astype(np.float32)
    n = x32.size
    nb = n_blocks(n, block)
    codes = np.zeros(n, dtype=code_dtype)
    scales = np.zeros(nb, dtype=np.float32)
    if n == 0:
        return codes, scales
    padded = np.zeros(nb * block, dtype=np.float32)
    padded[:n] = x32
    blocks = padded.reshape(nb, block)
    absmax = np.max(np.abs(blocks), axis=1)           # NaN propagates
    finite_nonzero = np.isfinite(absmax) & (absmax > 0)
    scales[:] = absmax                                  # 0, NaN or +inf blocks
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        s = (absmax[finite_nonzero] / np.float32(qmax)).astype(np.float32)
        scales[finite_nonzero] = s
        quot = (blocks[finite_nonzero] / s[:, None]).astype(np.float32)
    q = np.clip(np.rint(quot), qmin, qmax).astype(code_dtype)
    qb = np.zeros((nb, block), dtype=code_dtype)
    qb[finite_nonzero] = q
    codes[:] = qb.reshape(-1)[:n]
    return codes, scales


def encode(x, block: int = BLOCK):
    """Encode one tensor's moment values. Returns (codes int8[n], scales f32[nb])."""
    return _encode_linear(x, block, -QMAX, QMAX, np.int8)


def encode_unsigned(x, block: int = BLOCK):
    """Unsigned variant for non-negative values (the second moment).
    Returns (codes uint8[n], scales f32[nb]) with scale = max|x| / 255."""
    return _encode_linear(x, block, 0, UQMAX, np.uint8)


def decode_unsigned(codes, scales, block: int = BLOCK) -> np.ndarray:
    """Restore float64 values q * scale from unsigned codes (exact in float64)."""
    return decode(np.asarray(codes, dtype=np.uint8), scales, block)


def decode(codes, scales, block: int = BLOCK) -> np.ndarray:
    """Restore float64 moment values q * scale (exact in float64)."""
    codes = np.asarray(codes).reshape(-1)
    if codes.dtype not in (np.int8, np.uint8):
        codes = codes.astype(np.int8)
    scales = np.asarray(scales, dtype=np.float32).reshape(-1)
    n = codes.size
    if n == 0:
        return np.zeros(0, dtype=np.float64)
    per_elem = np.repeat(scales.astype(np.float64), block)[:n]
    with np.errstate(invalid="ignore"):
        return codes.astype(np.float64) * per_elem
