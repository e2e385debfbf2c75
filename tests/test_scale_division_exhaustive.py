"""The int8 scale fl(absmax / Q) without a division, checked exhaustively.

The step kernel stores a block's scale as the IEEE quotient fl(a / Q), Q = 127
(signed codes) or 255 (unsigned codes), but forms it without a division:

    q0 = RN(a * c)            c = RN(1/Q), an fp32 constant
    r  = RN(a - Q * q0)       one FMA: the exact residual, rounded once
    s  = RN(r * c + q0)       one FMA

(Markstein's residual correction). This test emulates those three fp32
roundings exactly in float64 arithmetic and compares s with numpy's IEEE
float32 division for every positive finite a that matters:

* every significand at exponent fields 0..8, where a / Q, q0 or r is
  subnormal or within a few binades of it;
* every significand at one middle exponent field (127). For exponent fields
  9..254 every step scales by the same power of two (nothing is subnormal,
  nothing overflows), so field 127 stands for all of them; a seeded sample of
  significands at every field checks that reading as well.

``--run-slow`` adds the literal sweep over all 2^31 - 2^23 finite positive
values. Both checks emulate the FMAs exactly (tests/fp32_exact.py): products
are exact in float64, and each fused sum is split exactly by TwoSum and
rounded to fp32 with its error deciding where float64 lands on an fp32
midpoint.
"""
from fractions import Fraction

import numpy as np
import pytest

from tests.fp32_exact import fma32, mul32

KERNEL_RCP = {127: float.fromhex("0x1.020408p-7"), 255: float.fromhex("0x1.010102p-8")}


def _rn32_exact(x: Fraction) -> np.float32:
    """fp32 round-to-nearest-even of an exact rational (brute force)."""
    f = np.float32(float(x))               # within one fp32 ulp of x
    cands = [np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))]
    best = min(cands, key=lambda c: (abs(Fraction(float(c)) - x),
                                     int(np.array(c).view(np.uint32)) & 1))
    return np.float32(best)


def test_reciprocal_constants_are_correctly_rounded():
    for q, c in KERNEL_RCP.items():
        assert np.float32(c) == _rn32_exact(Fraction(1, q)), q
        assert float(np.float32(c)) == c


def emulate(a32: np.ndarray, q: int, q_res: int = None, correct: bool = True) -> np.ndarray:
    """The kernel's three roundings, exactly, for fp32 inputs a32 > 0.
    ``q_res`` and ``correct`` exist only to plant mistakes: the divisor used in
    the residual, and whether the correction step runs at all."""
    c = np.float32(KERNEL_RCP[q])
    q0 = mul32(a32, c)
    if not correct:
        return q0
    qr = np.float32(q if q_res is None else q_res)
    r = fma32(-qr, q0, a32)
    return fma32(r, c, q0)


def _check(bits: np.ndarray, q: int, **plant) -> None:
    a = bits.view(np.float32)
    got = emulate(a, q, **plant)
    ref = a / np.float32(q)                          # IEEE float32 division
    bad = got.view(np.uint32) != ref.view(np.uint32)
    assert not np.any(bad), (q, [(float(x), float(y), float(z)) for x, y, z in
                                 zip(a[bad][:5], got[bad][:5], ref[bad][:5])])


def _field(e: int) -> np.ndarray:
    m = np.arange(1 << 23, dtype=np.uint32)
    bits = (np.uint32(e) << np.uint32(23)) | m
    return bits[1:] if e == 0 else bits             # a > 0


@pytest.mark.parametrize("plant", [dict(correct=False), dict(q_res=128), dict(q_res=126)])
def test_emulation_catches_planted_mistakes(plant):
    """A dropped correction step or a wrong divisor in the residual must be
    seen. (A reciprocal constant a few ulps off is not a mistake here: the
    residual correction absorbs it, which is why the constant is not what the
    result rests on.)"""
    with pytest.raises(AssertionError):
        _check(_field(127), 127, **plant)


@pytest.mark.parametrize("q", [127, 255])
def test_scale_equals_ieee_division_on_the_classes_that_decide_it(q):
    for e in list(range(0, 9)) + [127]:
        _check(_field(e), q)


@pytest.mark.parametrize("q", [127, 255])
def test_scaling_reading_on_a_sample_of_every_exponent(q):
    rng = np.random.default_rng(q)
    m = rng.integers(0, 1 << 23, size=2048, dtype=np.uint32)
    for e in range(1, 255):
        _check((np.uint32(e) << np.uint32(23)) | m, q)


@pytest.mark.slow
@pytest.mark.parametrize("q", [127, 255])
def test_scale_equals_ieee_division_for_every_finite_value(q):
    for e in range(0, 255):
        _check(_field(e), q)
