"""Pins for the oracle's Q6_K quantizer, dequantizer and embedding gather.

Q6_K (mistral.rs docs, "Quantization types": table "Q*K family", q6k at 6
bits; section "Numeric shorthands", `--isq 6` -> Q6K on CUDA; section
"Sensitive tensor precision", Q6K embeddings and output head for Q4K models)
is read as 256-weight superblocks of 16 sub-blocks, a binary16 d, 16 int8
sub-block scales and 6-bit codes (GGUF-shaped bytes, 210 per superblock).
The checks do not retype the oracle: an independently derived bit-position
table (walking the bytes, not the weights), hand-assembled on-grid bytes,
brute force over all 64 codes, exact-rational checks of d, exact half-step
quotients for the rounding rule, and the bit widths on the page.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from ggml_block_quantized_linear_b300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def byte_walk_table():
    """weight -> (ql byte, high nibble?, qh byte, shift), built by walking the
    170 code-carrying bytes: ql byte b holds, in its low nibble, weight
    128 (b // 64) + 32 ((b % 64) // 32) + b % 32 and in its high nibble the
    weight 64 further on; qh byte b holds, in bit pair s, weight
    128 (b // 32) + 32 s + b % 32."""
    table = {}
    for b in range(128):
        base = 128 * (b // 64) + 32 * ((b % 64) // 32) + b % 32
        table.setdefault(base, {})["lo"] = (b, 0)
        table.setdefault(base + 64, {})["lo"] = (b, 1)
    for b in range(64):
        for s in range(4):
            w = 128 * (b // 32) + 32 * s + b % 32
            table.setdefault(w, {})["hi"] = (128 + b, 2 * s)
    return {w: v["lo"] + v["hi"] for w, v in table.items()}


def test_position_table_is_a_bijection_and_matches():
    t = byte_walk_table()
    assert sorted(t) == list(range(256))
    lo_bits = {(b, h) for (b, h, _, _) in t.values()}
    hi_bits = {(b, s) for (_, _, b, s) in t.values()}
    assert len(lo_bits) == 256 and len(hi_bits) == 256  # every nibble / bit pair used once
    for w in range(256):
        assert oracle.q6_k_position(w) == t[w], w


def codes_of(packed_block):
    """(d, sc[16], q[256]) of one superblock, decoded with the byte-walk table."""
    blk = np.asarray(packed_block, dtype=np.uint8)
    t = byte_walk_table()
    q = np.zeros(256, dtype=np.int64)
    for w, (lb, lh, hb, hs) in t.items():
        lo = (int(blk[lb]) >> (4 * lh)) & 15
        hi = (int(blk[hb]) >> hs) & 3
        q[w] = lo | (hi << 4)
    sc = blk[192:208].view(np.int8).astype(np.int64)
    d = float(blk[208:210].view(np.float16)[0])
    return d, sc, q


def test_bits_per_weight_and_code_width():
    g = json.load(open(os.path.join(GOLDEN, "paper_widths.json")))
    assert oracle.packed_bytes(oracle.Q6_K, 3, 512) * 8 / (3 * 512) == 6.5625
    x = inputs.weights(8, 1024, 21, fp32=True).numpy()
    packed = oracle.quantize(oracle.Q6_K, x)
    qs = np.concatenate([codes_of(b)[2] for b in packed.reshape(-1, 210)])
    assert qs.min() >= 0 and qs.max() <= 63
    assert int(np.ceil(np.log2(qs.max() - qs.min() + 1))) == g["nominal_bits"]["q6k"]
    assert g["isq_shorthand_cuda"]["6"] == "Q6K"


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_on_grid_inputs_reconstruct_exactly(seed):
    # x = d0 * sc_j * c with d0 a power of two, one sub-block at sc = 127 and
    # every sub-block holding c = +-31: then s_j = d0 sc_j exactly, d = d0,
    # and the bytes are the hand-assembled ones
    rng = np.random.default_rng(seed)
    d0 = 2.0 ** -int(rng.integers(6, 12))
    sc = rng.integers(1, 128, 16)
    sc[rng.integers(0, 16)] = 127
    c = rng.integers(-31, 32, (16, 16))
    c[np.arange(16), rng.integers(0, 16, 16)] = rng.choice([-31, 31], 16)
    x = (d0 * sc[:, None] * c).astype(np.float32).reshape(1, 256)
    assert np.array_equal(x.astype(np.float64).ravel(), (d0 * sc[:, None] * c).ravel())
    packed = oracle.quantize(oracle.Q6_K, x).reshape(210)
    want = np.zeros(210, dtype=np.uint8)
    t = byte_walk_table()
    for w in range(256):
        q = int(c.ravel()[w]) + 32
        lb, lh, hb, hs = t[w]
        want[lb] |= (q & 15) << (4 * lh)
        want[hb] |= (q >> 4) << hs
    want[192:208] = sc.astype(np.int8).view(np.uint8)
    want[208:210] = np.array([d0], dtype=np.float16).view(np.uint8)
    assert np.array_equal(packed, want)
    assert np.array_equal(oracle.dequantize(oracle.Q6_K, packed, 1, 256), x)


def test_scale_is_nearest_binary16_and_codes_are_nearest():
    x = inputs.weights(6, 1024, 22, fp32=True).numpy()
    packed = oracle.quantize(oracle.Q6_K, x).reshape(-1, 210)
    blocks = x.reshape(-1, 16, 16)
    for blk, xb in zip(packed, blocks):
        d, sc, q = codes_of(blk)
        s = (np.abs(xb).max(axis=1).astype(np.float32) / np.float32(31)).astype(np.float32)
        target = Fraction(float(np.float32(s.max()) / np.float32(127)))
        dbits = int(blk[208:210].view(np.uint16)[0])
        here = Fraction(d)
        for nb in (dbits - 1, dbits + 1):
            other = Fraction(float(np.uint16(nb).view(np.float16)))
            assert abs(here - target) < abs(other - target) or (
                abs(here - target) == abs(other - target) and dbits % 2 == 0)
        # scale codes: nearest integer to s_j / d (fp32 quotient), in 0..127
        ratio = s.astype(np.float64) / d
        assert np.all(np.abs(ratio - sc) <= 0.5 + 1e-6)
        assert sc.min() >= 0 and sc.max() <= 127 and sc.max() >= 126
        # codes: the nearest of the 64 grid points S_j * (q - 32)
        S = (np.float32(d) * sc.astype(np.float32)).astype(np.float64)
        grid = S[:, None, None] * (np.arange(64) - 32)[None, None, :]
        dist = np.abs(xb.astype(np.float64)[:, :, None] - grid)
        chosen = np.abs(xb.astype(np.float64) - S[:, None] * (q.reshape(16, 16) - 32))
        slack = S[:, None] * 64 * 2.0 ** -23
        assert np.all(chosen <= dist.min(axis=-1) + slack)


U = 2.0 ** -10


def test_half_steps_round_away_from_zero():
    x = np.zeros((16, 16), dtype=np.float32)
    x[0, 0] = 3937 * U             # s_0 = 3937 U / 31 = 127 U: d = 127 U / 127 = U
    x[1, 0] = 1271 * U / 2         # s_1 = 635.5 U / 31 = 20.5 U: sc_1 = 20.5 -> 21 (even: 20)
    x[2, 0] = 496 * U              # s_2 = 16 U: sc_2 = 16, S_2 = 2^-6
    ks = [0, 2, 4, 10, 20, 30]
    for i, k in enumerate(ks):     # c = +-(k + 1/2) -> +-(k + 1) (even: +-k)
        x[2, 1 + i] = (k + 0.5) * 16 * U
        x[2, 8 + i] = -(k + 0.5) * 16 * U
    packed = oracle.quantize(oracle.Q6_K, x.reshape(1, 256)).reshape(210)
    d, sc, q = codes_of(packed)
    assert d == U
    assert sc[0] == 127 and sc[1] == 21 and sc[2] == 16
    c = q.reshape(16, 16) - 32
    assert c[2, 0] == 31
    assert c[2, 1:1 + len(ks)].tolist() == [k + 1 for k in ks]
    assert c[2, 8:8 + len(ks)].tolist() == [-(k + 1) for k in ks]
    assert not c[3:].any() and sc[3:].tolist() == [0] * 13


def test_zero_and_tiny_superblocks():
    z = oracle.quantize(oracle.Q6_K, np.zeros((2, 256), dtype=np.float32))
    d, sc, q = codes_of(z[0])
    assert d == 0.0 and not sc.any() and np.all(q == 32)
    assert not oracle.dequantize(oracle.Q6_K, z, 2, 256).any()
    tiny = np.full((1, 256), 1e-9, dtype=np.float32)  # d underflows binary16
    d, sc, q = codes_of(oracle.quantize(oracle.Q6_K, tiny)[0])
    assert d == 0.0 and not sc.any() and np.all(q == 32)


def test_fp32_and_bf16_sources_agree_on_bf16_values():
    w = inputs.weights(4, 512, 23)
    a = oracle.quantize(oracle.Q6_K, inputs.bf16_bits(w))
    b = oracle.quantize(oracle.Q6_K, w.float().numpy())
    assert np.array_equal(a, b)


@pytest.mark.parametrize("fmt", [oracle.Q8_0, oracle.Q4_K, oracle.Q6_K, oracle.FP8, oracle.Q5_K, oracle.Q3_K, oracle.Q2_K])
def test_gather_is_dequantize_of_the_listed_rows(fmt):
    V, D = 37, 512
    packed = oracle.quantize(fmt, inputs.bf16_bits(inputs.weights(V, D, 24)))
    full = oracle.dequantize(fmt, packed, V, D)
    ids = np.array([0, 36, 5, 5, 17, 0, 1], dtype=np.int64)
    assert np.array_equal(oracle.gather(fmt, packed, V, D, ids), full[ids])
    assert np.array_equal(oracle.gather(fmt, packed, V, D, np.arange(V)), full)
    assert oracle.gather(fmt, packed, V, D, np.zeros(0, dtype=np.int64)).shape == (0, D)
    for bad in ([V], [-1], [0, V + 3]):
        with pytest.raises(ValueError):
            oracle.gather(fmt, packed, V, D, np.array(bad, dtype=np.int64))
