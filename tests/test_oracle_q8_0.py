"""Pins for the oracle's Q8_0 quantizer and dequantizer.

Q8_0 (mistral.rs docs, "Quantization types", table "Legacy GGML types":
q8_0, 8 bits) is read as 32-weight blocks holding a binary16 scale d and
32 int8 codes (34 bytes).  Nothing here compares the oracle with a retyped
copy of itself: the checks are the nearest-grid property (brute force over all
255 codes), the nearest-binary16 property of d, the round-trip bound d/2,
exact reconstruction of inputs on the grid, and the bit widths on the page.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from ggml_block_quantized_linear_b300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def split_q8_0(packed, rows, cols):
    blk = packed.reshape(rows, cols // 32, 34)
    d = np.ascontiguousarray(blk[:, :, 0:2]).view(np.float16)[..., 0].astype(np.float32)
    q = np.ascontiguousarray(blk[:, :, 2:34]).view(np.int8).astype(np.int32)
    return d, q


def sample_bf16(rows, cols, seed):
    w = inputs.weights(rows, cols, seed)
    return inputs.bf16_bits(w), w.float().numpy()


def test_bits_per_weight_and_code_width():
    g = json.load(open(os.path.join(GOLDEN, "paper_widths.json")))
    assert oracle.packed_bytes(oracle.Q8_0, 7, 256) * 8 / (7 * 256) == 8.5
    bits, x = sample_bf16(16, 1024, 11)
    _, q = split_q8_0(oracle.quantize(oracle.Q8_0, bits), 16, 1024)
    # codes use the full signed 8-bit range that the page's width names
    assert q.min() >= -127 and q.max() <= 127
    assert (np.abs(q) == 127).any()
    assert int(np.ceil(np.log2(q.max() - q.min() + 1))) == g["nominal_bits"]["q8_0"]


def test_nearest_grid_brute_force():
    rows, cols = 24, 512
    bits, x = sample_bf16(rows, cols, 12)
    d, q = split_q8_0(oracle.quantize(oracle.Q8_0, bits), rows, cols)
    xb = x.reshape(rows, cols // 32, 32).astype(np.float64)
    codes = np.arange(-127, 128, dtype=np.float64)
    dist = np.abs(xb[..., None] - d[..., None, None].astype(np.float64) * codes)  # exact in fp64
    best = dist.min(axis=-1)
    chosen = np.abs(xb - d[..., None].astype(np.float64) * q)
    # the chosen code is the nearest grid point; the quotient x/d is formed in
    # fp32 before rounding, so a near-tie may differ by one fp32 ulp of it
    slack = d[..., None].astype(np.float64) * 128 * 2.0 ** -23
    assert np.all(chosen <= best + slack)
    strict = chosen == best
    assert strict.mean() > 0.999


def test_scale_is_nearest_binary16_of_amax_over_127():
    rows, cols = 8, 256
    bits, x = sample_bf16(rows, cols, 13)
    packed = oracle.quantize(oracle.Q8_0, bits)
    blk = packed.reshape(rows, cols // 32, 34)
    dbits = np.ascontiguousarray(blk[:, :, 0:2]).view(np.uint16)[..., 0]
    amax = np.abs(x.reshape(rows, cols // 32, 32)).max(axis=-1).astype(np.float32)
    target = amax / np.float32(127)  # IEEE single division
    for db, t in zip(dbits.ravel(), target.ravel()):
        t = Fraction(float(t))
        here = Fraction(float(np.uint16(db).view(np.float16)))
        for nb in (int(db) - 1, int(db) + 1):
            other = Fraction(float(np.uint16(nb).view(np.float16)))
            assert abs(here - t) < abs(other - t) or (
                abs(here - t) == abs(other - t) and db % 2 == 0)


def test_round_trip_bound_half_step():
    rows, cols = 32, 1024
    bits, x = sample_bf16(rows, cols, 14)
    packed = oracle.quantize(oracle.Q8_0, bits)
    deq = oracle.dequantize(oracle.Q8_0, packed, rows, cols)
    d, _ = split_q8_0(packed, rows, cols)
    assert (d > 6.2e-5).all()  # normal binary16 scales for this distribution
    err = np.abs(x - deq).reshape(rows, cols // 32, 32)
    assert np.all(err <= d[..., None] / 2)


@pytest.mark.parametrize("e", [-14, -9, -6, -3, 0])
def test_on_grid_inputs_reconstruct_exactly(e):
    rng = np.random.default_rng(100 + e)
    rows, cols = 4, 128
    q = rng.integers(-127, 128, size=(rows, cols // 32, 32))
    q[:, :, rng.integers(0, 32)] = rng.choice([-127, 127])  # each block reaches |q| = 127
    d0 = np.float32(2.0 ** e)
    x = (q * d0).astype(np.float32).reshape(rows, cols)
    xb = torch.from_numpy(x).to(torch.bfloat16)
    assert torch.equal(xb.float(), torch.from_numpy(x))  # exact in bf16 (7-bit codes)
    packed = oracle.quantize(oracle.Q8_0, inputs.bf16_bits(xb))
    want = np.zeros((rows, cols // 32, 34), dtype=np.uint8)
    want[:, :, 0:2] = np.frombuffer(np.float16(d0).tobytes(), dtype=np.uint8)
    want[:, :, 2:] = q.astype(np.int8).view(np.uint8)
    assert np.array_equal(packed.reshape(rows, cols // 32, 34), want)
    assert np.array_equal(oracle.dequantize(oracle.Q8_0, packed, rows, cols), x)


def test_zero_block_and_tiny_scale():
    x = np.zeros((2, 64), dtype=np.float32)
    x[1, 32:] = 1e-12  # amax / 127 underflows binary16 -> d = 0, all codes 0
    packed = oracle.quantize(oracle.Q8_0, x)
    assert not packed.any()
    assert not oracle.dequantize(oracle.Q8_0, packed, 2, 64).any()


def test_fp32_and_bf16_sources_agree_on_bf16_values():
    bits, x = sample_bf16(8, 256, 15)
    a = oracle.quantize(oracle.Q8_0, bits)
    b = oracle.quantize(oracle.Q8_0, np.ascontiguousarray(x, dtype=np.float32))
    assert np.array_equal(a, b)


def test_rejects_ragged_cols():
    with pytest.raises(ValueError):
        oracle.quantize(oracle.Q8_0, np.zeros((1, 48), dtype=np.float32))
