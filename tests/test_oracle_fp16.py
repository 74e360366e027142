"""Pins for the oracle's own IEEE 754 binary16 encoder / decoder.

The oracle writes binary16 conversion from the standard's definition; here it
is checked against two independent library conversions (numpy and torch), and
against the tie-to-even rule stated directly on the bit patterns.
"""
import numpy as np
import torch

import oracle


def test_decode_all_65536_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.f16_bits_to_f32(bits)
    ref = bits.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_encode_random_matches_numpy_and_torch():
    rng = np.random.default_rng(1)
    n = 400_000
    # log-uniform magnitudes from deep subnormal to overflow, random signs
    mag = np.exp2(rng.uniform(-27.0, 17.0, n)).astype(np.float32)
    sign = np.where(rng.random(n) < 0.5, -1.0, 1.0).astype(np.float32)
    x = mag * sign
    ours = oracle.f32_to_f16_bits(x)
    ref_np = x.astype(np.float16).view(np.uint16)
    ref_t = torch.from_numpy(x).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref_np)
    assert np.array_equal(ours, ref_t)


def test_ties_round_to_even_and_neighbours():
    # every midpoint between consecutive positive finite halves (exact in fp32)
    lo = np.arange(0, 0x7BFF, dtype=np.uint16)
    a = lo.view(np.float16).astype(np.float64)
    b = (lo + 1).view(np.float16).astype(np.float64)
    mid = ((a + b) / 2).astype(np.float32)
    assert np.array_equal(mid.astype(np.float64), (a + b) / 2)  # midpoints are exact
    enc = oracle.f32_to_f16_bits(mid)
    want = np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint16)  # the even neighbour
    assert np.array_equal(enc, want)
    # one fp32 ulp either side of the tie goes to the nearer neighbour
    below = np.nextafter(mid, np.float32(0))
    above = np.nextafter(mid, np.float32(np.inf))
    assert np.array_equal(oracle.f32_to_f16_bits(below), lo)
    assert np.array_equal(oracle.f32_to_f16_bits(above), (lo + 1).astype(np.uint16))
    # and negative values mirror positive ones with the sign bit set
    assert np.array_equal(oracle.f32_to_f16_bits(-mid), want | 0x8000)


def test_special_values():
    vals = np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, np.inf, -np.inf,
                     2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0001, 2.0 ** -14, 6e-8],
                    dtype=np.float32)
    want = vals.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.f32_to_f16_bits(vals), want)
    assert oracle.f32_to_f16_bits([np.float32(np.nan)])[0] & 0x7C00 == 0x7C00
