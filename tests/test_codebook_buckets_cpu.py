"""The codebook encoder's bucket entries, checked on the CPU.

The step kernel finds a codebook code without searching: it cuts |y| in
[2^-21, 1) (signed map) or [2^-25, 1) (unsigned map) into buckets of 1/64 or
1/128 of a binary octave, keyed by the float's exponent and top mantissa
bits, and keeps one 32-bit entry per bucket,

    E = base * 2^24 + (2^24 - in) - bits(S)   (mod 2^32),

with S the bucket's first float, base the number of midpoints below S, and
`in` the bits of the bucket's midpoint above S (2^17 or 2^16, the bucket's
width in low bits, when it holds none). The code is the top byte of
bits(|y|) + E, with |y| first raised to the first bucket's start. Each
bucket holds at most one midpoint (pinned against the oracle's tables in
test_oracle_codec_variants.py), so this is the number of midpoints <= |y|,
the oracle's nearest-code rule with ties to the larger magnitude.

This module builds the entries from the oracle's midpoints as the kernel
builds them from its own, applies the same 32-bit arithmetic, and compares
with numpy's search over the oracle's midpoints: on every float of the
octaves around the smallest midpoints, around every midpoint and every
bucket start, and on a seeded sample of the rest. ``--run-slow`` sweeps
every float in [0, 1] for both maps. A planted mistake in the entry (an
off-by-one midpoint offset, the shift of an 18-bit layout) must fail.
"""
import numpy as np
import pytest

from oracle import dynamic8 as d8

# (midpoints, first exponent field, buckets per octave, low bits, octaves)
MAPS = {
    "signed": (d8.SIGNED_MID, 106, 64, 17, 21),
    "unsigned": (d8.UNSIGNED_MID, 102, 128, 16, 25),
}
ONE = 0x3F800000


def entries(mid, e0, per, low, noct, shift=24, in_bias=0):
    """Bucket entries (one past the last for |y| = 1.0), as uint64 < 2^32."""
    mid32 = np.asarray(mid, dtype=np.float32)
    midb = mid32.view(np.uint32).astype(np.int64)
    i = np.arange(noct * per + 1, dtype=np.int64)
    start = ((e0 + i // per) << 23) | ((i % per) << low)
    base = np.searchsorted(midb, start, side="left")          # midpoints below S
    nxt = midb[np.minimum(base, len(midb) - 1)]
    inside = (base < len(midb)) & (nxt < start + (1 << low))
    inn = np.where(inside, nxt - start + in_bias, 1 << low)
    return (((base << shift) + ((1 << shift) - inn) - start) % (1 << 32)).astype(np.uint64)


def codes(bits, ent, e0, per, low, shift=24):
    """The kernel's code for the floats with bit patterns `bits` (|y| <= 1)."""
    clamp = np.uint64(e0) << np.uint64(23)
    b = np.maximum(bits.astype(np.uint64), clamp)
    idx = (b >> np.uint64(low)) - np.uint64(e0 * per)
    return ((b + ent[idx.astype(np.int64)]) % np.uint64(1 << 32)) >> np.uint64(shift)


def oracle_codes(bits, mid):
    y = bits.astype(np.uint32).view(np.float32).astype(np.float64)
    return np.searchsorted(mid, y, side="right")


def probe_bits(mid, e0, per, low, noct, seed):
    """Every float of the two lowest octaves, +-8 ulps around every midpoint
    and every bucket start, zero, the clamp region, 1.0, and a seeded sample."""
    parts = [np.arange(e0 << 23, (e0 + 2) << 23, dtype=np.int64)]
    midb = np.asarray(mid, dtype=np.float32).view(np.uint32).astype(np.int64)
    d = np.arange(-8, 9, dtype=np.int64)
    parts.append((midb[:, None] + d[None, :]).ravel())
    i = np.arange(noct * per + 1, dtype=np.int64)
    starts = ((e0 + i // per) << 23) | ((i % per) << low)
    parts.append((starts[:, None] + d[None, :]).ravel())
    parts.append(np.arange(0, 1 << 16, dtype=np.int64))                 # zero, subnormals
    parts.append(np.array([ONE, ONE - 1, (e0 << 23) - 1], dtype=np.int64))
    rng = np.random.default_rng(seed)
    parts.append(rng.integers(0, ONE + 1, 1 << 22, dtype=np.int64))
    b = np.concatenate(parts)
    return b[(b >= 0) & (b <= ONE)]


@pytest.mark.parametrize("name", list(MAPS))
def test_bucket_entries_give_the_oracle_codes(name):
    mid, e0, per, low, noct = MAPS[name]
    ent = entries(mid, e0, per, low, noct)
    b = probe_bits(mid, e0, per, low, noct, seed=7)
    got = codes(b, ent, e0, per, low)
    ref = oracle_codes(b, mid)
    bad = np.flatnonzero(got.astype(np.int64) != ref)
    assert bad.size == 0, [(hex(int(b[k])), int(got[k]), int(ref[k])) for k in bad[:5]]
    # the top byte never exceeds the map's largest code
    assert int(got.max()) == len(mid)


@pytest.mark.parametrize("name", list(MAPS))
@pytest.mark.parametrize("plant", ["in_off_by_one", "shift_18_layout"])
def test_planted_entry_mistakes_fail(name, plant):
    mid, e0, per, low, noct = MAPS[name]
    if plant == "in_off_by_one":
        ent = entries(mid, e0, per, low, noct, in_bias=1)
        shift = 24
    else:
        ent = entries(mid, e0, per, low, noct, shift=18)
        shift = 24                 # read with the top-byte rule: wrong codes
    b = probe_bits(mid, e0, per, low, noct, seed=8)
    got = codes(b, ent, e0, per, low, shift=shift)
    assert np.any(got.astype(np.int64) != oracle_codes(b, mid))


@pytest.mark.slow
@pytest.mark.parametrize("name", list(MAPS))
def test_bucket_entries_every_float_in_0_1(name):
    mid, e0, per, low, noct = MAPS[name]
    ent = entries(mid, e0, per, low, noct)
    bad = 0
    for c0 in range(0, ONE + 1, 1 << 24):
        b = np.arange(c0, min(c0 + (1 << 24), ONE + 1), dtype=np.int64)
        bad += int(np.count_nonzero(codes(b, ent, e0, per, low).astype(np.int64)
                                    != oracle_codes(b, mid)))
    assert bad == 0
