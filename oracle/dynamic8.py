"""Block-wise 8-bit moment codec with a non-linear (dynamic exponent) codebook.

"Fused Optimizers and State Precision", section 05: the uniform teaching codec
lets outliers crush small moments; real 8-bit optimizers may use a non-linear
codebook with block statistics instead. The ApexW Unsloth benchmark page
describes bitsandbytes' 8-bit AdamW as block-wise quantization with dynamic
scaling. The pages give no codebook, so this follows the published dynamic
tree quantization (Dettmers, Lewis, Shleifer, Zettlemoyer, "8-bit Optimizers
via Block-wise Quantization", ICLR 2022, section 2): a code's bits are a sign
bit, a run of zeros whose length is a base-10 exponent, an indicator 1 bit,
and linear fraction bits.

Readings (one concrete table from that description):

* Signed map (first moment), byte b = s<<7 | r: r = 0 is zero; otherwise E =
  the number of leading zeros of r in 7 bits (0..6), the indicator is r's
  highest 1 bit, F = 6 - E fraction bits hold f = r - 2^F, and the magnitude
  is 10^-E * (0.1 + 0.9 * (f + 1) / 2^F) = (2^F + 9 (f + 1)) / (2^F 10^(E+1)):
  2^F equal steps over (0.1, 1] of each decade, the top code of a decade
  exactly 10^-E, the largest 1.0, the smallest 1e-6. Magnitudes increase with
  r. The value is (-1)^s times the magnitude; b = 0x80 (a negative zero) is
  never produced.
* Unsigned map (second moment, never negative): the same rule over all 8 bits
  (E = leading zeros of b in 8 bits, 0..7; F = 7 - E): 255 non-zero values
  from 1e-7 to 1.0.
* Table values are the fp32 roundings of the exact rationals (one float64
  division, then a cast to fp32).
* Blocks are 256 elements as in the linear codec; a block's scale is its
  fp32 absmax (no division). Zero blocks store scale 0 and code 0; a block
  holding NaN/inf stores that absmax and code 0, so it decodes to NaN.
* Encoding: y = fp32(x / scale) (IEEE fp32 division of the fp32-rounded x),
  and the code is the nearest table value to |y| (sign from y): with the
  midpoints mid[k] = fp32((c[k] + c[k+1]) / 2) (float64 sum of the fp32
  values), the index is the number of midpoints <= |y|, so a tie goes to the
  larger magnitude. Every decision is taken in fp32, the kernel's precision.
* Decoding: table value times scale, exact in float64.
"""
from __future__ import annotations

import numpy as np

from .formats import round_to
from .int8_block import BLOCK, n_blocks


def _magnitudes(bits: int) -> np.ndarray:
    """Codebook magnitudes for codes 0 .. 2^bits - 1 (fp32 values as float64)."""
    out = np.zeros(1 << bits, dtype=np.float64)
    for r in range(1, 1 << bits):
        top = r.bit_length() - 1          # position of the indicator bit
        e = bits - 1 - top                # leading zeros
        fbits = top                       # bits below the indicator
        f = r - (1 << fbits)
        num = (1 << fbits) + 9 * (f + 1)
        den = (1 << fbits) * 10 ** (e + 1)
        out[r] = float(np.float32(num / den))
    return out


SIGNED = _magnitudes(7)       # r = 0..127
UNSIGNED = _magnitudes(8)     # b = 0..255


def midpoints(table: np.ndarray) -> np.ndarray:
    """fp32 midpoints between consecutive table values (as float64)."""
    t = np.asarray(table, dtype=np.float64)
    return round_to((t[:-1] + t[1:]) / 2.0, "f32")


SIGNED_MID = midpoints(SIGNED)
UNSIGNED_MID = midpoints(UNSIGNED)


def _block_view(x, block):
    x32 = round_to(np.asarray(x, dtype=np.float64).reshape(-1), "f32").astype(np.float32)
    n = x32.size
    nb = n_blocks(n, block)
    padded = np.zeros(nb * block, dtype=np.float32)
    padded[:n] = x32
    return padded.reshape(nb, block), n, nb


def _encode(x, block, table_mid, signed):
    blocks, n, nb = _block_view(x, block)
    codes = np.zeros(n, dtype=np.uint8)
    scales = np.zeros(nb, dtype=np.float32)
    if n == 0:
        return codes, scales
    absmax = np.max(np.abs(blocks), axis=1)           # NaN propagates
    ok = np.isfinite(absmax) & (absmax > 0)
    scales[:] = absmax
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        y = (blocks[ok] / absmax[ok][:, None]).astype(np.float32)
    mag = np.abs(y).astype(np.float64)
    idx = np.searchsorted(table_mid, mag, side="right")   # midpoints <= |y|
    if signed:
        idx = np.where((y < 0) & (idx > 0), idx | 0x80, idx)
    qb = np.zeros((nb, block), dtype=np.uint8)
    qb[ok] = idx.astype(np.uint8)
    codes[:] = qb.reshape(-1)[:n]
    return codes, scales


def _decode(codes, scales, block, signed):
    codes = np.asarray(codes, dtype=np.uint8).reshape(-1)
    scales = np.asarray(scales, dtype=np.float32).reshape(-1)
    n = codes.size
    if n == 0:
        return np.zeros(0, dtype=np.float64)
    if signed:
        val = SIGNED[codes & 0x7F] * np.where(codes & 0x80, -1.0, 1.0)
    else:
        val = UNSIGNED[codes]
    per_elem = np.repeat(scales.astype(np.float64), block)[:n]
    with np.errstate(invalid="ignore"):
        return val * per_elem


def encode_signed(x, block: int = BLOCK):
    """First moment: (codes uint8[n] = sign<<7 | r, scales f32[nb] = absmax)."""
    return _encode(x, block, SIGNED_MID, True)


def decode_signed(codes, scales, block: int = BLOCK) -> np.ndarray:
    return _decode(codes, scales, block, True)


def encode_unsigned(x, block: int = BLOCK):
    """Second moment: (codes uint8[n], scales f32[nb] = absmax)."""
    return _encode(x, block, UNSIGNED_MID, False)


def decode_unsigned(codes, scales, block: int = BLOCK) -> np.ndarray:
    return _decode(codes, scales, block, False)
