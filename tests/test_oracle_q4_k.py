"""Pins for the oracle's Q4_K quantizer and dequantizer.

Q4_K (mistral.rs docs, "Quantization types", table "Q*K family": q4k, 4 bits)
is read as a 256-weight superblock of eight 32-weight sub-blocks: binary16
d and dmin, eight 6-bit scale codes and eight 6-bit min codes packed into 12
bytes, and 4-bit codes (144 bytes).  The checks: the scale-byte packing is a
bit permutation equal to an independently written bit-position table
(exhaustive over every code pair), each 4-bit code is the nearest grid point
(brute force over 16 codes), the reconstruction bound, exact reconstruction
of on-grid inputs, degenerate superblocks, and the page's width.
"""
import json
import os

import numpy as np
import pytest

import oracle
from ggml_block_quantized_linear_b300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

# Bit-position table of the 12 scale bytes: (kind, sub-block j, code bit b)
# -> (byte, bit).  kind 0 = scale code sc_j, kind 1 = min code mc_j.
POS = {}
for j in range(4):
    for b in range(6):
        POS[(0, j, b)] = (j, b)
        POS[(1, j, b)] = (j + 4, b)
    for b in range(4):
        POS[(0, j + 4, b)] = (j + 8, b)
        POS[(1, j + 4, b)] = (j + 8, b + 4)
    for b in (4, 5):
        POS[(0, j + 4, b)] = (j, b + 2)
        POS[(1, j + 4, b)] = (j + 4, b + 2)


def table_decode(s12):
    sc = np.zeros(8, dtype=np.int32)
    mc = np.zeros(8, dtype=np.int32)
    for (kind, j, b), (byte, bit) in POS.items():
        v = (int(s12[byte]) >> bit) & 1
        (sc if kind == 0 else mc)[j] |= v << b
    return sc, mc


def table_encode(sc, mc):
    s = np.zeros(12, dtype=np.uint8)
    for (kind, j, b), (byte, bit) in POS.items():
        v = ((sc if kind == 0 else mc)[j] >> b) & 1
        s[byte] |= np.uint8(v << bit)
    return s


def split_q4_k(packed, rows, cols):
    blk = packed.reshape(rows, cols // 256, 144)
    d = np.ascontiguousarray(blk[..., 0:2]).view(np.float16)[..., 0].astype(np.float32)
    dmin = np.ascontiguousarray(blk[..., 2:4]).view(np.float16)[..., 0].astype(np.float32)
    sc = np.zeros(blk.shape[:2] + (8,), dtype=np.int32)
    mc = np.zeros_like(sc)
    for r in range(blk.shape[0]):
        for b in range(blk.shape[1]):
            sc[r, b], mc[r, b] = table_decode(blk[r, b, 4:16])
    qs = blk[..., 16:144].reshape(rows, cols // 256, 4, 32)
    q = np.zeros(blk.shape[:2] + (8, 32), dtype=np.int32)
    q[:, :, 0::2, :] = qs & 15
    q[:, :, 1::2, :] = qs >> 4
    return d, dmin, sc, mc, q


def test_position_table_is_a_bit_permutation():
    targets = list(POS.values())
    assert len(POS) == 96 and len(set(targets)) == 96  # all 96 bits of 12 bytes, once


def test_scale_packing_exhaustive():
    rng = np.random.default_rng(3)
    grid = np.arange(64)
    for j in range(8):
        for sval in grid:
            for mval in grid:
                sc = rng.integers(0, 64, 8)
                mc = rng.integers(0, 64, 8)
                sc[j], mc[j] = sval, mval
                s12 = oracle.pack_scales_q4_k(sc, mc)
                if sval % 9 == 0 and mval % 9 == 0:  # the table encoder is slow
                    assert np.array_equal(s12, table_encode(sc, mc))
                dsc, dmc = table_decode(s12)
                assert np.array_equal(dsc, sc) and np.array_equal(dmc, mc)
                osc, omc = oracle.unpack_scales_q4_k(s12)
                assert np.array_equal(osc, sc) and np.array_equal(omc, mc)


def test_scale_packing_hand_examples():
    z = np.zeros(8, dtype=np.int32)
    sc = z.copy(); sc[0] = 63
    assert list(oracle.pack_scales_q4_k(sc, z)) == [63] + [0] * 11
    sc = z.copy(); sc[4] = 63            # low nibble in byte 8, top two bits in byte 0
    assert list(oracle.pack_scales_q4_k(sc, z)) == [192, 0, 0, 0, 0, 0, 0, 0, 15, 0, 0, 0]
    mc = z.copy(); mc[7] = 63            # high nibble of byte 11, top two bits of byte 7
    assert list(oracle.pack_scales_q4_k(z, mc)) == [0, 0, 0, 0, 0, 0, 0, 192, 0, 0, 0, 240]
    mc = z.copy(); mc[2] = 5
    assert list(oracle.pack_scales_q4_k(z, mc)) == [0, 0, 0, 0, 0, 0, 5, 0, 0, 0, 0, 0]


def test_bits_per_weight_and_code_width():
    g = json.load(open(os.path.join(GOLDEN, "paper_widths.json")))
    assert oracle.packed_bytes(oracle.Q4_K, 3, 512) * 8 / (3 * 512) == 4.5
    w = inputs.weights(8, 1024, 21)
    packed = oracle.quantize(oracle.Q4_K, inputs.bf16_bits(w))
    _, _, sc, mc, q = split_q4_k(packed, 8, 1024)
    assert q.min() == 0 and q.max() == 15
    assert int(np.log2(q.max() + 1)) == g["nominal_bits"]["q4k"]
    assert sc.max() <= 63 and mc.max() <= 63


def sample(rows, cols, seed):
    w = inputs.weights(rows, cols, seed)
    bits = inputs.bf16_bits(w)
    return bits, w.float().numpy()


def test_nearest_code_brute_force():
    rows, cols = 16, 1024
    bits, x = sample(rows, cols, 22)
    packed = oracle.quantize(oracle.Q4_K, bits)
    d, dmin, sc, mc, q = split_q4_k(packed, rows, cols)
    S = (d[..., None] * sc).astype(np.float64)      # exact products
    Mn = (dmin[..., None] * mc).astype(np.float64)
    xs = x.reshape(rows, cols // 256, 8, 32).astype(np.float64)
    codes = np.arange(16, dtype=np.float64)
    grid = S[..., None, None] * codes - Mn[..., None, None]
    dist = np.abs(xs[..., None] - grid)
    best = dist.min(axis=-1)
    chosen = np.abs(xs - (S[..., None] * q - Mn[..., None]))
    slack = S[..., None] * 32 * 2.0 ** -23 + np.abs(xs) * 2.0 ** -22
    assert np.all(chosen <= best + slack)
    assert (chosen == best).mean() > 0.999


def test_reconstruction_bound_and_full_range_codes():
    rows, cols = 16, 2048
    bits, x = sample(rows, cols, 23)
    packed = oracle.quantize(oracle.Q4_K, bits)
    d, dmin, sc, mc, q = split_q4_k(packed, rows, cols)
    deq = oracle.dequantize(oracle.Q4_K, packed, rows, cols).reshape(rows, cols // 256, 8, 32)
    xs = x.reshape(deq.shape)
    S = d[..., None] * sc
    bound = np.maximum(S / 2, 7.5 * d[..., None] + 0.5 * dmin[..., None])
    err = np.abs(xs - deq).max(axis=-1)
    assert np.all(err <= bound * (1 + 1e-6) + 1e-9)
    # the largest sub-block range / offset maps to the top 6-bit code
    assert np.all(sc.max(axis=-1) == 63)
    assert np.all(mc.max(axis=-1)[dmin > 0] == 63)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_on_grid_inputs_reconstruct_exactly(seed):
    rng = np.random.default_rng(seed)
    rows, nsb = 3, 4
    d0, dmin0 = np.float32(2.0 ** -10), np.float32(2.0 ** -11)
    sc = rng.integers(1, 64, (rows, nsb, 8))
    mc = rng.integers(0, 64, (rows, nsb, 8))
    sc[..., rng.integers(0, 8)] = 63
    mc[..., rng.integers(0, 8)] = 63
    q = rng.integers(0, 16, (rows, nsb, 8, 32))
    q[..., 0] = 0
    q[..., 31] = 15
    x = (d0 * sc[..., None] * q - dmin0 * mc[..., None]).astype(np.float32)
    x2 = x.reshape(rows, nsb * 256)
    packed = oracle.quantize(oracle.Q4_K, x2, oracle.SRC_F32).reshape(rows, nsb, 144)
    want = np.zeros_like(packed)
    want[..., 0:2] = np.frombuffer(np.float16(d0).tobytes(), dtype=np.uint8)
    want[..., 2:4] = np.frombuffer(np.float16(dmin0).tobytes(), dtype=np.uint8)
    for r in range(rows):
        for b in range(nsb):
            want[r, b, 4:16] = table_encode(sc[r, b], mc[r, b])
            for j in range(8):
                c, hi = divmod(j, 2)
                want[r, b, 16 + 32 * c:48 + 32 * c] |= (q[r, b, j] << (4 * hi)).astype(np.uint8)
    assert np.array_equal(packed, want)
    deq = oracle.dequantize(oracle.Q4_K, packed.reshape(rows, -1), rows, nsb * 256)
    assert np.array_equal(deq, x2)


def test_degenerate_superblocks():
    x = np.zeros((4, 256), dtype=np.float32)
    x[1] = np.linspace(0.0, 1.0, 256, dtype=np.float32)        # no negatives: dmin = 0
    x[2] = -np.linspace(0.01, 1.0, 256, dtype=np.float32)      # all negative
    x[3, :32] = -0.0                                           # signed zeros only
    packed = oracle.quantize(oracle.Q4_K, x)
    d, dmin, sc, mc, q = split_q4_k(packed, 4, 256)
    assert not packed[0].any() and not packed[3].any()
    assert dmin[1, 0] == 0 and not mc[1].any()
    deq = oracle.dequantize(oracle.Q4_K, packed, 4, 256)
    assert np.all(deq[1] >= 0)
    assert np.all(np.abs(deq[2] - x[2]) <= np.maximum(d[2, 0] * 63 / 2, 7.5 * d[2, 0] + 0.5 * dmin[2, 0]))


def test_fp32_and_bf16_sources_agree_on_bf16_values():
    bits, x = sample(4, 512, 24)
    assert np.array_equal(oracle.quantize(oracle.Q4_K, bits),
                          oracle.quantize(oracle.Q4_K, np.ascontiguousarray(x)))
