"""Pins of the oracle's storage rounding and 8-bit block codec.

``formats.round_to`` is pinned to library casts (numpy float64->float32 and
float64->float16 are correctly rounded; torch's CPU float32->bfloat16 cast is
round-to-nearest-even) and to a brute-force nearest-neighbour search.
``int8_block`` is pinned to the reconstruction bound, max -> +-127, the zero
block rule and a brute-force nearest-code search ("Fused Optimizers and State
Precision", section 05 teaching codec).
"""
import numpy as np
import pytest
import torch

from oracle import int8_block
from oracle.formats import round_to


def _wide_doubles(rng, n):
    mant = rng.random(n) + 0.5
    exp = rng.integers(-160, 140, n)
    x = np.ldexp(mant, exp) * np.where(rng.random(n) < 0.5, -1, 1)
    return x


@pytest.mark.parametrize("fmt,npdt", [("f32", np.float32), ("f16", np.float16)])
def test_round_to_matches_numpy_casts(fmt, npdt):
    rng = np.random.default_rng(0)
    x = np.concatenate([_wide_doubles(rng, 200000),
                        np.array([0.0, -0.0, np.inf, -np.inf, 1e-50, -1e-50,
                                  65504.0, 65519.99, 65520.0, 3.5e38, 3.4028235e38,
                                  3.40282357e38, 3.4028236e38])])
    # exact ties between adjacent values of the target format
    base = rng.random(20000).astype(npdt).astype(np.float64)
    nxt = np.nextafter(base.astype(npdt), npdt(np.inf)).astype(np.float64)
    x = np.concatenate([x, 0.5 * (base + nxt), -0.5 * (base + nxt)])
    with np.errstate(over="ignore"):
        ref = x.astype(npdt).astype(np.float64)
    got = round_to(x, fmt)
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all(), x[~same][:5]
    assert np.array_equal(np.signbit(got), np.signbit(ref))


def test_round_to_bf16_matches_torch_on_fp32_inputs():
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x4000, 0xC000],
                    dtype=np.uint32)
    bits = (hi[:, None] | lows[None, :]).reshape(-1)
    f32 = bits.view(np.float32)
    ref = torch.from_numpy(f32.copy()).to(torch.bfloat16).to(torch.float32).numpy()
    got = round_to(f32.astype(np.float64), "bf16")
    same = (got == ref.astype(np.float64)) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_round_to_bf16_is_nearest_even_by_search():
    rng = np.random.default_rng(1)
    x = _wide_doubles(rng, 20000)
    x = x[np.abs(x) < 3e38]
    got = round_to(x, "bf16")
    # neighbours by walking bf16 bit patterns (torch's bf16 view)
    lo = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    lo_bits = lo.view(torch.int16).numpy().astype(np.int64) & 0xFFFF
    cands = []
    for d in (-2, -1, 0, 1, 2):
        b = ((lo_bits + d) & 0xFFFF).astype(np.uint16)
        c = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
        cands.append((c, b))
    for j in range(x.size):
        best = None
        for c, b in cands:
            cj = c[j]
            if not np.isfinite(cj) or np.sign(cj) * np.sign(x[j]) < 0:
                continue
            dist = abs(cj - x[j])
            key = (dist, int(b[j]) & 1)          # ties: even pattern wins
            if best is None or key < best[0]:
                best = (key, cj)
        assert got[j] == best[1], (x[j], got[j], best)


def test_round_to_special_values():
    for fmt in ("f32", "bf16", "f16"):
        r = round_to([np.nan, np.inf, -np.inf, 0.0, -0.0], fmt)
        assert np.isnan(r[0]) and r[1] == np.inf and r[2] == -np.inf
        assert r[3] == 0 and not np.signbit(r[3]) and np.signbit(r[4])


# ----------------------------------------------------------------- int8 codec

def _blocks(rng, n):
    x = rng.normal(0, 1e-3, n) * np.exp(rng.normal(0, 2, n))
    return x


@pytest.mark.parametrize("n", [1, 5, 255, 256, 257, 1000, 4096 + 17])
def test_int8_reconstruction_bound_and_extremes(n):
    rng = np.random.default_rng(n)
    x = _blocks(rng, n)
    codes, scales = int8_block.encode(x)
    assert codes.dtype == np.int8 and scales.dtype == np.float32
    assert scales.size == -(-n // 256)
    x32 = x.astype(np.float32).astype(np.float64)
    dec = int8_block.decode(codes, scales)
    s = np.repeat(scales.astype(np.float64), 256)[:n]
    # |x - q*scale| <= scale/2, plus the rounding of the fp32 quotient x/scale
    assert np.all(np.abs(x32 - dec) <= s * (0.5 + 128 * 2.0 ** -24))
    for b in range(scales.size):
        blk = x32[b * 256:(b + 1) * 256]
        j = int(np.argmax(np.abs(blk)))
        assert abs(int(codes[b * 256 + j])) == 127
        assert np.sign(codes[b * 256 + j]) == np.sign(blk[j])
        # scale is the fp32 quotient of the block's own absmax by 127
        assert scales[b] == np.float32(np.float32(np.max(np.abs(blk))) / np.float32(127))
    assert np.all(np.abs(codes.astype(int)) <= 127)


def test_int8_zero_block_is_exact_and_division_free():
    x = np.zeros(600)
    x[300] = 1e-3
    codes, scales = int8_block.encode(x)
    assert scales[0] == 0 and scales[2] == 0 and scales[1] > 0
    assert np.all(codes[:256] == 0) and np.all(codes[512:] == 0)
    dec = int8_block.decode(codes, scales)
    assert np.all(dec[:256] == 0) and np.all(dec[512:] == 0)


def test_int8_exact_multiples_round_trip():
    rng = np.random.default_rng(2)
    s = np.float32(3.0517578125e-05)          # a power of two: k*s exact
    k = rng.integers(-127, 128, 256)
    k[0] = 127
    x = k.astype(np.float64) * float(s)
    codes, scales = int8_block.encode(x)
    assert scales[0] == s
    assert np.array_equal(codes.astype(int), k)
    assert np.array_equal(int8_block.decode(codes, scales), x)


def test_int8_codes_are_nearest_by_search():
    rng = np.random.default_rng(3)
    for trial in range(40):
        n = int(rng.integers(1, 300))
        x = _blocks(rng, n)
        codes, scales = int8_block.encode(x)
        x32 = x.astype(np.float32)
        for b in range(scales.size):
            blk = x32[b * 256:(b + 1) * 256]
            s = scales[b]
            quot = (blk / s).astype(np.float32).astype(np.float64)
            qs = np.arange(-127, 128)
            dist = np.abs(quot[:, None] - qs[None, :])
            best = dist.min(axis=1)
            # the nearest code; among equally near codes the even one
            cand = np.where(dist == best[:, None], qs[None, :], 10 ** 6)
            even = np.where((cand % 2 == 0) & (cand != 10 ** 6), cand, 10 ** 6)
            pick = np.where(even.min(axis=1) != 10 ** 6, even.min(axis=1), cand.min(axis=1))
            assert np.array_equal(codes[b * 256:b * 256 + blk.size].astype(int), pick)


def test_int8_ties_go_to_even():
    s = np.float32(2.0 ** -10)
    x = np.array([127.0, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5]) * float(s)
    codes, scales = int8_block.encode(x)
    assert scales[0] == s
    assert list(codes) == [127, 0, 2, 2, 0, -2, -2]


def test_int8_nonfinite_block_decodes_to_nan():
    x = np.ones(512) * 1e-3
    x[3] = np.nan
    x[300] = np.inf
    codes, scales = int8_block.encode(x)
    assert np.isnan(scales[0]) and scales[1] == np.inf
    assert np.all(codes == 0)
    assert np.all(np.isnan(int8_block.decode(codes, scales)))


def test_int8_second_moment_codes_nonnegative():
    rng = np.random.default_rng(4)
    v = rng.random(1000) ** 4 * 1e-6
    codes, _ = int8_block.encode(v)
    assert codes.min() >= 0 and codes.max() == 127
