"""Pins of the 8-bit codec variants ("Fused Optimizers and State Precision",
section 05: real 8-bit optimizers may use other codebooks than the uniform
teaching codec).

Unsigned linear codec for the second moment (scale = max/255): the
reconstruction bound, max -> 255, exact multiples, brute-force nearest code
with ties to even, zero and non-finite blocks, and half the signed codec's
worst error.

Dynamic-exponent codebook (the published dynamic tree quantization): the
table's structure from its bit layout (codes per decade, decade tops equal
to fp32(10^-E) by an independent route, equal steps inside a decade, the
extremes); encoding equals a brute-force nearest search; the per-decade error
bound; small values next to an outlier keep their sign and magnitude where
the linear codec zeroes them; zero and non-finite blocks.
"""
import numpy as np
import pytest

from oracle import dynamic8, int8_block
from oracle.formats import round_to


def _f32(x):
    return np.asarray(x, dtype=np.float64).astype(np.float32)


# ----------------------------------------------------------- unsigned linear

@pytest.mark.parametrize("n", [1, 255, 256, 257, 1000])
def test_unsigned_bound_and_max(n):
    rng = np.random.default_rng(n)
    x = rng.random(n) ** 3 * 1e-3
    q, s = int8_block.encode_unsigned(x)
    assert q.dtype == np.uint8
    x32 = _f32(x).astype(np.float64)
    d = int8_block.decode_unsigned(q, s)
    per = np.repeat(s.astype(np.float64), 256)[:n]
    assert np.all(np.abs(x32 - d) <= per * (0.5 + 2e-5))
    for b in range(len(s)):
        blk = x32[b * 256:(b + 1) * 256]
        assert q[b * 256 + int(np.argmax(blk))] == 255


def test_unsigned_exact_multiples_and_zero_block():
    k = np.arange(256, dtype=np.float64)
    k[0], k[-1] = 0, 255
    x = k * 2.0 ** -10          # scale = 255 * 2^-10 / 255 = 2^-10 exactly
    q, s = int8_block.encode_unsigned(x)
    assert s[0] == 2.0 ** -10 and np.array_equal(q, k.astype(np.uint8))
    q, s = int8_block.encode_unsigned(np.zeros(300))
    assert np.all(q == 0) and np.all(s == 0)
    assert np.all(int8_block.decode_unsigned(q, s) == 0)


def test_unsigned_codes_are_nearest_even_by_search():
    rng = np.random.default_rng(5)
    x = rng.random(256) * 3.7
    x[7] = 0.0
    q, s = int8_block.encode_unsigned(x)
    y = (_f32(x) / s[0]).astype(np.float32).astype(np.float64)
    for i in range(256):
        dist = np.abs(y[i] - np.arange(256))
        best = np.flatnonzero(dist == dist.min())
        want = best[0] if len(best) == 1 else [c for c in best if c % 2 == 0][0]
        assert q[i] == want


def test_unsigned_nonfinite_block_is_nan():
    x = np.linspace(0, 1, 256)
    x[3] = np.inf
    q, s = int8_block.encode_unsigned(x)
    assert np.all(q == 0) and np.isinf(s[0])
    assert np.all(np.isnan(int8_block.decode_unsigned(q, s)))


def test_unsigned_halves_the_worst_error():
    rng = np.random.default_rng(9)
    x = rng.random(256 * 64)
    es = np.max(np.abs(int8_block.decode(*int8_block.encode(x)) - _f32(x)))
    eu = np.max(np.abs(int8_block.decode_unsigned(*int8_block.encode_unsigned(x)) - _f32(x)))
    assert eu < 0.55 * es


# --------------------------------------------------------- dynamic codebook

@pytest.mark.parametrize("table,bits", [(dynamic8.SIGNED, 7), (dynamic8.UNSIGNED, 8)])
def test_codebook_structure(table, bits):
    assert table[0] == 0 and table[-1] == 1.0
    assert np.all(np.diff(table) > 0)
    assert table[1] == float(np.float32(10.0 ** -(bits - 1)))    # code 1: all leading zeros
    for e in range(bits):
        fb = bits - 1 - e                                           # fraction bits
        lo, hi = 1 << fb, (1 << (fb + 1)) - 1                       # codes of the decade
        assert hi - lo + 1 == 2 ** fb
        assert table[hi] == float(np.float32(10.0 ** -e))          # the decade's top
        step = np.diff(table[lo:hi + 1])
        if len(step):
            want = 0.9 * 10.0 ** -e / 2 ** fb
            assert np.allclose(step, want, rtol=1e-5, atol=0)


def test_codebook_encode_is_nearest_by_search():
    rng = np.random.default_rng(11)
    for signed in (True, False):
        mag = 10.0 ** rng.uniform(-8, 0, 2048)
        x = mag * (np.where(rng.random(2048) < 0.5, -1, 1) if signed else 1)
        x = x.reshape(8, 256)
        x[:, 0] = 1.0                              # scale 1: y = fp32(x)
        table = dynamic8.SIGNED if signed else dynamic8.UNSIGNED
        enc = dynamic8.encode_signed if signed else dynamic8.encode_unsigned
        q, s = enc(x.reshape(-1))
        assert np.all(s == 1.0)
        y = _f32(x.reshape(-1)).astype(np.float64)
        for i in range(y.size):
            d = np.abs(np.abs(y[i]) - table)
            best = np.flatnonzero(d == d.min())[-1]            # ties: larger magnitude
            code = best if not signed or y[i] >= 0 or best == 0 else best | 0x80
            assert q[i] == code, (i, y[i], q[i], code)


def test_codebook_midpoint_tie_goes_up():
    t = dynamic8.SIGNED
    for k in (0, 5, 40, 100, 125):
        mid = np.float32((t[k] + t[k + 1]) / 2)
        below = np.nextafter(mid, np.float32(0))
        x = np.zeros(256)
        x[0], x[1], x[2] = 1.0, float(mid), float(below)
        q, _ = dynamic8.encode_signed(x)
        assert q[1] == k + 1 and q[2] == k, (k, q[1], q[2])


def test_codebook_error_bound_per_decade():
    rng = np.random.default_rng(12)
    x = 10.0 ** rng.uniform(-6, 0, 256 * 16)
    x[::256] = 1.0
    q, s = dynamic8.encode_unsigned(x)
    d = dynamic8.decode_unsigned(q, s)
    y = _f32(x).astype(np.float64)
    e = np.floor(-np.log10(y) + 1e-12).clip(0, 7)      # decade of y
    fb = 7 - e
    half = 0.45 * 10.0 ** -e / 2 ** fb
    assert np.all(np.abs(d - y) <= half * (1 + 1e-5) + 1e-7)


def test_small_values_survive_next_to_an_outlier():
    x = np.full(256, 0.0)
    x[0] = 1.0
    x[1:128] = np.linspace(1e-5, 2e-3, 127)
    x[128:] = -np.linspace(1e-5, 2e-3, 128)
    lin = int8_block.decode(*int8_block.encode(x))
    dyn = dynamic8.decode_signed(*dynamic8.encode_signed(x))
    small = slice(1, 256)
    rel = lambda d: np.abs(d[small] - x[small]) / np.abs(x[small])
    assert np.mean(lin[small] == 0) > 0.5            # the linear codec loses most of them
    assert np.median(rel(lin)) >= 0.5
    assert np.all(np.sign(dyn[small]) == np.sign(x[small]))   # none lost, signs kept
    assert np.median(rel(dyn)) < 0.1


def test_codebook_zero_and_nonfinite_blocks():
    for enc, dec in ((dynamic8.encode_signed, dynamic8.decode_signed),
                     (dynamic8.encode_unsigned, dynamic8.decode_unsigned)):
        q, s = enc(np.zeros(300))
        assert np.all(q == 0) and np.all(s == 0) and np.all(dec(q, s) == 0)
        x = np.linspace(0, 1, 256)
        x[9] = np.nan
        q, s = enc(x)
        assert np.all(q == 0) and np.isnan(s[0]) and np.all(np.isnan(dec(q, s)))


def test_codebook_negative_zero_never_produced():
    x = np.concatenate([[1.0], -np.full(255, 1e-9)])   # rounds to zero magnitude
    q, _ = dynamic8.encode_signed(x)
    assert np.all(q[1:] == 0)


@pytest.mark.parametrize("mid,first_exp,mbits", [(dynamic8.SIGNED_MID, -21, 6),
                                                  (dynamic8.UNSIGNED_MID, -25, 7)])
def test_codebook_midpoints_one_per_fine_bucket(mid, first_exp, mbits):
    """Cut [2^first_exp, 1) into 2^mbits equal buckets per binary octave: each
    holds at most one midpoint of the map, and everything below holds none,
    so a code is a bucket's first midpoint index plus one comparison."""
    m = mid.astype(np.float32).astype(np.float64)
    assert m[0] > 2.0 ** first_exp
    for e in range(first_exp, 0):
        edges = 2.0 ** e * (1 + np.arange((1 << mbits) + 1) / 2 ** mbits)
        counts = np.histogram(m, bins=edges)[0]
        assert counts.max() <= 1, (e, counts.max())
