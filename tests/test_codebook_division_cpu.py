"""The codebook encoder's division by the block scale, checked on the CPU.

The step kernel divides every moment of a codebook block by the block's
absmax s without a division per element:

* per block, r = RN(1/s) from a faithful reciprocal y by one Newton-Raphson
  step, RN(y + y * RN(1 - s*y)) (the kernel reaches a faithful y with one
  step from rcp.approx first);
* per element, Markstein's division: q0 = RN(x*r), e = RN(x - s*q0),
  y = RN(q0 + e*r).

Markstein's theorems say the first step returns RN(1/s) from either faithful
neighbour unless s's significand is all ones (the kernel then divides by IEEE
division), and the second gives the IEEE quotient when r = RN(1/s), q0 is
faithful and nothing underflows or overflows (the kernel keeps s within
[2^-64, 2^64] for that). The first is checked here for every significand and
both faithful neighbours of 1/s (exponents scale out inside that range); the
second on several million seeded pairs and on quotients placed exactly at
and next to the codebook's decision midpoints, against numpy's IEEE float32
division. A planted mistake (r one ulp off) must make the division check
fail.
"""
import numpy as np
import pytest

from tests.fp32_exact import fma32, mul32

ALL_ONES = 0x7FFFFF


def _rn_recip(s32):
    return (np.float32(1.0) / s32).astype(np.float32)


def _nr_step(y, s):
    e = fma32(-s, y, np.float32(1.0))
    return fma32(y, e, y)


def test_newton_step_rounds_the_reciprocal_correctly_for_every_significand():
    m = np.arange(1 << 23, dtype=np.uint32)
    s = ((np.uint32(127) << np.uint32(23)) | m).view(np.float32)      # [1, 2)
    rn = _rn_recip(s)
    exact = 1.0 / s.astype(np.float64)                                # within 2^-53
    lo = np.where(rn.astype(np.float64) <= exact, rn, np.nextafter(rn, np.float32(0)))
    hi = np.nextafter(lo, np.float32(2))                              # the two faithful values
    special = m == ALL_ONES
    for y in (lo, hi):
        got = _nr_step(y, s)
        bad = (got.view(np.uint32) != rn.view(np.uint32)) & ~special
        assert not np.any(bad), s[bad][:5]
    # in the kernel's range every exponent behaves the same: spot-check a few
    for k in (-63, -20, 20, 63):
        sk = (s[::4097] * np.float32(2.0 ** k)).astype(np.float32)
        rk = _rn_recip(sk)
        yk = np.nextafter(rk, np.float32(0))
        got = _nr_step(yk, sk)
        ok = (got == rk) | ((sk.view(np.uint32) & ALL_ONES) == ALL_ONES)
        assert np.all(ok)


def _markstein(x, s, r):
    q0 = mul32(x, r)
    e = fma32(-s, q0, x)
    return fma32(e, r, q0)


def _division_cases(n, seed):
    rng = np.random.default_rng(seed)
    s = (rng.uniform(1.0, 2.0, n) * 2.0 ** rng.integers(-64, 64, n)).astype(np.float32)
    s = s[(s.view(np.uint32) & ALL_ONES) != ALL_ONES]
    # quotients over the codebook's whole range (magnitudes 2^-27 .. 1)
    y = (np.sign(rng.standard_normal(s.size)) *
         2.0 ** rng.uniform(-27, 0, s.size)).astype(np.float64)
    x = (y * s.astype(np.float64)).astype(np.float32)
    x = np.where(np.abs(x) > s, s, x).astype(np.float32)             # |x| <= absmax
    return x, s


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_markstein_division_equals_ieee_division(seed):
    x, s = _division_cases(1 << 21, seed)
    r = _rn_recip(s)
    got = _markstein(x, s, r)
    ref = (x / s).astype(np.float32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_markstein_division_at_the_codebook_midpoints():
    """Quotients placed at, and one ulp either side of, every decision
    midpoint of both maps (the values where a wrong rounding would change a
    code), for many scales."""
    from oracle import dynamic8
    mids = np.concatenate([dynamic8.SIGNED_MID, dynamic8.UNSIGNED_MID])
    mids = mids[np.isfinite(mids) & (mids > 0)].astype(np.float32)
    targets = np.concatenate([mids, np.nextafter(mids, np.float32(0)),
                              np.nextafter(mids, np.float32(2))])
    rng = np.random.default_rng(7)
    s = (rng.uniform(1.0, 2.0, 4096) * 2.0 ** rng.integers(-60, 60, 4096)).astype(np.float32)
    s = s[(s.view(np.uint32) & ALL_ONES) != ALL_ONES]
    X, S = np.meshgrid(targets, s)
    S = S.reshape(-1)
    # x = fl(t*s) and its two neighbours, so fl(x/s) lands on and around t
    base = mul32(X.reshape(-1), S)
    for x in (base, np.nextafter(base, np.float32(0)), np.nextafter(base, np.float32(np.inf))):
        x = np.minimum(x, S)
        got = _markstein(x, S, _rn_recip(S))
        ref = (x / S).astype(np.float32)
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("plant", ["no_correction", "coarse_reciprocal"])
def test_planted_mistakes_are_caught(plant):
    """The check must see a dropped correction step, or a reciprocal far
    from RN(1/s) (a quotient q0 that is no longer faithful). (A reciprocal
    one ulp off is not enough to show: the correction absorbs it in almost
    every case, which is why the theorem asks for more than the tests show.)"""
    x, s = _division_cases(1 << 20, 11)
    r = _rn_recip(s)
    if plant == "no_correction":
        got = mul32(x, r)
    else:
        got = _markstein(x, s, (r * np.float32(1 + 2.0 ** -10)).astype(np.float32))
    ref = (x / s).astype(np.float32)
    assert not np.array_equal(got.view(np.uint32), ref.view(np.uint32))
