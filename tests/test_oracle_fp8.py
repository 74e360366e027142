"""Pins for the oracle's FP8 E4M3 weights with a scale per row (W8A16).

mistral.rs docs, "Quantization types", section "FP8": E4M3 FP8 can be
produced with ISQ, and the FP8 table lists fp8 at 8 bits, E4M3; symmetric
E4M3 W8A16 is listed with tensor, channel or block weight scales.  The
reading here: one fp32 scale per output row, s = max|x| / 448, codes
E4M3(x / s) rounded to nearest even and saturated at +-448.  The E4M3
encoder and decoder are pinned against torch's float8_e4m3fn (an independent
implementation, which rounds the same way but gives NaN above 464 instead of
saturating), the quantizer against hand-built rows.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from ggml_block_quantized_linear_b300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_all_256_decodes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_bits_to_f32(codes)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2  # S.1111.111
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6


def test_encoder_matches_torch_inside_the_range():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.uniform(-464, 464, 200000),
        rng.normal(0, 1, 100000) * np.exp2(rng.integers(-14, 8, 100000)),
        np.arange(-464, 464.5, 0.5),
    ]).astype(np.float32)
    x = x[np.abs(x) <= 464]
    got = oracle.f32_to_e4m3_bits(x)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, want)


def test_midpoints_go_to_the_even_code_and_large_values_saturate():
    vals = oracle.e4m3_bits_to_f32(np.arange(0x7F, dtype=np.uint8))  # 0 .. 448
    mids = ((vals[:-1].astype(np.float64) + vals[1:]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (vals[:-1].astype(np.float64) + vals[1:]) / 2)
    got = oracle.f32_to_e4m3_bits(mids)
    lo = np.arange(0x7E, dtype=np.uint8)
    want = np.where(lo % 2 == 0, lo, lo + 1)  # the even neighbour's code
    assert np.array_equal(got, want)
    assert np.array_equal(oracle.f32_to_e4m3_bits(-mids), want | 0x80)
    big = np.array([448.0, 449.0, 464.0, 465.0, 1e6, 3e38], dtype=np.float32)
    assert np.array_equal(oracle.f32_to_e4m3_bits(big), np.full(6, 0x7E))
    assert np.array_equal(oracle.f32_to_e4m3_bits(-big), np.full(6, 0xFE))


def split(packed, K):
    codes = packed[:, :K]
    s = np.ascontiguousarray(packed[:, K:K + 4]).view(np.float32)[:, 0]
    return codes, s, packed[:, K + 4:]


def test_row_scale_codes_and_layout():
    K = 1024
    x = inputs.weights(12, K, 81, fp32=True).numpy()
    packed = oracle.quantize(oracle.FP8, x)
    assert packed.shape == (12, K + 16) and oracle.packed_bytes(oracle.FP8, 12, K) == 12 * (K + 16)
    codes, s, pad = split(packed, K)
    amax = np.abs(x).max(axis=1).astype(np.float32)
    assert np.array_equal(s, (amax / np.float32(448)).astype(np.float32))  # fp32 division
    assert not pad.any()
    q = (x / s[:, None]).astype(np.float32)
    want = torch.from_numpy(np.clip(q, -464, 464)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    want = np.where(np.abs(q) > 448, np.where(q > 0, 0x7E, 0xFE), want)
    assert np.array_equal(codes, want)
    # the largest weight of each row maps to +-448
    top = np.argmax(np.abs(x), axis=1)
    assert np.all(codes[np.arange(12), top] & 0x7F == 0x7E)
    deq = oracle.dequantize(oracle.FP8, packed, 12, K)
    assert np.array_equal(deq, (oracle.e4m3_bits_to_f32(codes).reshape(12, K) * s[:, None]).astype(np.float32))


def test_on_grid_rows_reconstruct_exactly():
    rng = np.random.default_rng(2)
    K = 512
    vals = oracle.e4m3_bits_to_f32(rng.integers(0, 0x7F, (4, K)).astype(np.uint8)).reshape(4, K)
    sign = rng.choice([-1.0, 1.0], (4, K)).astype(np.float32)
    v = vals * sign
    v[:, 7] = 448.0
    s0 = np.float32(2.0 ** -10)
    x = (v * s0).astype(np.float32)
    packed = oracle.quantize(oracle.FP8, x)
    codes, s, _ = split(packed, K)
    assert np.all(s == s0)
    assert np.array_equal(oracle.e4m3_bits_to_f32(codes).reshape(4, K), v)
    assert np.array_equal(oracle.dequantize(oracle.FP8, packed, 4, K), x)


def test_zero_row_and_width():
    g = json.load(open(os.path.join(GOLDEN, "paper_widths.json")))
    packed = oracle.quantize(oracle.FP8, np.zeros((2, 256), dtype=np.float32))
    assert not packed.any()
    assert g["nominal_bits"]["fp8"] == 8 and g["fp8_type"] == "E4M3"
    assert oracle.packed_bytes(oracle.FP8, 1, 4096) * 8 / 4096 == 8 + 128 / 4096
    assert oracle.packed_bytes(oracle.FP8, 1, 300) < 0  # rows are whole 256-weight groups


def test_fp32_and_bf16_sources_agree_on_bf16_values():
    w = inputs.weights(3, 768, 82)
    assert np.array_equal(oracle.quantize(oracle.FP8, inputs.bf16_bits(w)),
                          oracle.quantize(oracle.FP8, w.float().numpy()))
