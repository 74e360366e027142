"""Pins for the oracle's Q5_K, Q3_K and Q2_K quantizers and dequantizers.

mistral.rs documentation, "Quantization types": table "Q*K family" (q2k, q3k,
q5k at 2, 3 and 5 bits) and section "Numeric shorthands" (`--isq 2 / 3 / 5`
resolve to Q2K / Q3K / Q5K on CUDA).  The byte layouts are the library's
GGUF-shaped reading (176, 110 and 84 bytes per 256 weights) and the
quantizers follow the same plain style as Q4_K (affine: Q5_K, Q2_K) and Q6_K
(symmetric: Q3_K).  The checks do not retype the oracle: bit-position tables
built by walking the bytes, hand-assembled bytes for inputs on the grid,
brute force over every code, exact-rational checks of the binary16 scales,
exact half-step quotients for the rounding rule, and the page's widths.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from ggml_block_quantized_linear_b300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
U = 2.0 ** -10


# ------------------------------------------------------------ decoders by byte walking
def q5_walk(blk):
    """(d, dmin, sc[8], mc[8], q[256]) of a Q5_K superblock, decoded by walking
    the bytes: qs byte 48 + 32c + l -> weight l of sub-blocks 2c (low nibble)
    and 2c + 1 (high nibble); qh byte 16 + l, bit j -> bit 4 of weight l of
    sub-block j; the scale bytes through the Q4_K unpacking pinned elsewhere."""
    blk = np.asarray(blk, dtype=np.uint8)
    q = np.zeros(256, dtype=np.int64)
    for b in range(128):
        c, l = divmod(b, 32)
        q[32 * (2 * c) + l] |= int(blk[48 + b]) & 15
        q[32 * (2 * c + 1) + l] |= int(blk[48 + b]) >> 4
    for l in range(32):
        for j in range(8):
            q[32 * j + l] |= ((int(blk[16 + l]) >> j) & 1) << 4
    sc, mc = oracle.unpack_scales_q4_k(blk[4:16])
    d = float(blk[0:2].view(np.float16)[0])
    dmin = float(blk[2:4].view(np.float16)[0])
    return d, dmin, sc.astype(np.int64), mc.astype(np.int64), q


def q3_walk_table():
    """weight -> (qs byte, shift, hmask byte, bit), built from the bytes: qs
    byte 32 + 32h + l holds, in bit pair s, weight 128h + 32s + l; hmask byte
    l holds, in bit t, weight 128 (t div 4) + 32 (t mod 4) + l."""
    t = {}
    for b in range(64):
        h, l = divmod(b, 32)
        for s in range(4):
            t.setdefault(128 * h + 32 * s + l, {})["lo"] = (32 + b, 2 * s)
    for l in range(32):
        for bit in range(8):
            t.setdefault(128 * (bit // 4) + 32 * (bit % 4) + l, {})["hi"] = (l, bit)
    return {w: v["lo"] + v["hi"] for w, v in t.items()}


def q3_field_writer(values):
    """The 12 scale bytes holding sixteen 6-bit fields, written from the
    reading in the oracle's header (an independent writer)."""
    sb = np.zeros(12, dtype=np.uint8)
    for j, v in enumerate(values):
        sb[j % 8] |= (v & 15) << (0 if j < 8 else 4)
        sb[8 + j % 4] |= ((v >> 4) & 3) << (2 * (j // 4))
    return sb


def q3_walk(blk):
    blk = np.asarray(blk, dtype=np.uint8)
    tab = q3_walk_table()
    q = np.zeros(256, dtype=np.int64)
    for w, (lb, ls, hb, hbit) in tab.items():
        q[w] = ((int(blk[lb]) >> ls) & 3) | (((int(blk[hb]) >> hbit) & 1) << 2)
    fields = np.array([oracle.q3_k_scale_field(blk[96:108], j) for j in range(16)], dtype=np.int64)
    d = float(blk[108:110].view(np.float16)[0])
    return d, fields, q


def q2_walk(blk):
    blk = np.asarray(blk, dtype=np.uint8)
    q = np.zeros(256, dtype=np.int64)
    for b in range(64):
        h, l = divmod(b, 32)
        for s in range(4):
            q[128 * h + 32 * s + l] = (int(blk[16 + b]) >> (2 * s)) & 3
    sc = (blk[0:16] & 15).astype(np.int64)
    mc = (blk[0:16] >> 4).astype(np.int64)
    d = float(blk[80:82].view(np.float16)[0])
    dmin = float(blk[82:84].view(np.float16)[0])
    return d, dmin, sc, mc, q


# ------------------------------------------------------------ layout tables
def test_q3_k_positions_are_a_bijection_and_match():
    t = q3_walk_table()
    assert sorted(t) == list(range(256))
    assert len({(b, s) for b, s, _, _ in t.values()}) == 256
    assert len({(b, s) for _, _, b, s in t.values()}) == 256
    for w in range(256):
        assert oracle.q3_k_position(w) == t[w], w


def test_q3_k_scale_fields_exhaustive():
    # every field value alone, and random field sets, through the independent writer
    for j in range(16):
        for v in range(64):
            vals = [0] * 16
            vals[j] = v
            sb = q3_field_writer(vals)
            assert [oracle.q3_k_scale_field(sb, i) for i in range(16)] == vals
    rng = np.random.default_rng(3)
    for _ in range(200):
        vals = rng.integers(0, 64, 16).tolist()
        sb = q3_field_writer(vals)
        assert [oracle.q3_k_scale_field(sb, i) for i in range(16)] == vals
    # the 96 field bits cover the 12 bytes exactly once
    seen = set()
    for j in range(16):
        for bit in range(6):
            vals = [0] * 16
            vals[j] = 1 << bit
            sb = q3_field_writer(vals)
            (byte,) = np.nonzero(sb)[0]
            seen.add((int(byte), int(sb[byte]).bit_length() - 1))
    assert len(seen) == 96


def test_widths_and_bits_per_weight():
    g = json.load(open(os.path.join(GOLDEN, "paper_widths.json")))
    for fmt, key, bpw in ((oracle.Q5_K, "q5k", 5.5), (oracle.Q3_K, "q3k", 3.4375), (oracle.Q2_K, "q2k", 2.625)):
        assert oracle.packed_bytes(fmt, 3, 512) * 8 / (3 * 512) == bpw
        x = inputs.weights(6, 1024, 31, fp32=True).numpy()
        blocks = oracle.quantize(fmt, x).reshape(-1, oracle.BLOCK[fmt][1])
        walk = {oracle.Q5_K: lambda b: q5_walk(b)[4], oracle.Q3_K: lambda b: q3_walk(b)[2],
                oracle.Q2_K: lambda b: q2_walk(b)[4]}[fmt]
        qs = np.concatenate([walk(b) for b in blocks])
        assert qs.min() >= 0 and int(np.ceil(np.log2(qs.max() + 1))) == g["nominal_bits"][key]
    assert [g["isq_shorthand_cuda"][k] for k in "235"] == ["Q2K", "Q3K", "Q5K"]


# ------------------------------------------------------------ inputs on the grid
@pytest.mark.parametrize("seed", [1, 2])
def test_q5_k_on_grid_exact(seed):
    # x = d0 sc_j q - dmin0 mc_j with max sc = max mc = 63 and every sub-block
    # holding q = 0 and q = 31: then s_j = d0 sc_j, m_j = dmin0 mc_j exactly
    rng = np.random.default_rng(seed)
    d0, dm0 = 2.0 ** -int(rng.integers(8, 12)), 2.0 ** -int(rng.integers(8, 12))
    sc = rng.integers(1, 64, 8)
    mc = rng.integers(1, 64, 8)
    sc[rng.integers(0, 8)] = 63
    mc[rng.integers(0, 8)] = 63
    q = rng.integers(0, 32, (8, 32))
    q[:, 0], q[:, 1] = 0, 31
    x = (d0 * sc[:, None] * q - dm0 * mc[:, None]).astype(np.float32).reshape(1, 256)
    assert np.array_equal(x.ravel().astype(np.float64), (d0 * sc[:, None] * q - dm0 * mc[:, None]).ravel())
    blk = oracle.quantize(oracle.Q5_K, x).reshape(176)
    want = np.zeros(176, dtype=np.uint8)
    want[0:2] = np.array([d0], dtype=np.float16).view(np.uint8)
    want[2:4] = np.array([dm0], dtype=np.float16).view(np.uint8)
    want[4:16] = oracle.pack_scales_q4_k(sc, mc)
    for j in range(8):
        for l in range(32):
            want[48 + 32 * (j // 2) + l] |= (int(q[j, l]) & 15) << (4 * (j % 2))
            want[16 + l] |= (int(q[j, l]) >> 4) << j
    assert np.array_equal(blk, want)
    assert np.array_equal(oracle.dequantize(oracle.Q5_K, blk, 1, 256), x)


@pytest.mark.parametrize("seed", [1, 2])
def test_q3_k_on_grid_exact(seed):
    # x = d0 sc_j c with c in -3..3, |c| = 3 in every sub-block, max sc = 31
    rng = np.random.default_rng(seed)
    d0 = 2.0 ** -int(rng.integers(6, 12))
    sc = rng.integers(1, 32, 16)
    sc[rng.integers(0, 16)] = 31
    c = rng.integers(-3, 4, (16, 16))
    c[np.arange(16), rng.integers(0, 16, 16)] = rng.choice([-3, 3], 16)
    x = (d0 * sc[:, None] * c).astype(np.float32).reshape(1, 256)
    blk = oracle.quantize(oracle.Q3_K, x).reshape(110)
    want = np.zeros(110, dtype=np.uint8)
    tab = q3_walk_table()
    for w in range(256):
        qv = int(c.ravel()[w]) + 4
        lb, ls, hb, hbit = tab[w]
        want[lb] |= (qv & 3) << ls
        want[hb] |= (qv >> 2) << hbit
    want[96:108] = q3_field_writer((sc + 32).tolist())
    want[108:110] = np.array([d0], dtype=np.float16).view(np.uint8)
    assert np.array_equal(blk, want)
    assert np.array_equal(oracle.dequantize(oracle.Q3_K, blk, 1, 256), x)


@pytest.mark.parametrize("seed", [1, 2])
def test_q2_k_on_grid_exact(seed):
    rng = np.random.default_rng(seed)
    d0, dm0 = 2.0 ** -int(rng.integers(6, 10)), 2.0 ** -int(rng.integers(6, 10))
    sc = rng.integers(1, 16, 16)
    mc = rng.integers(1, 16, 16)
    sc[rng.integers(0, 16)] = 15
    mc[rng.integers(0, 16)] = 15
    q = rng.integers(0, 4, (16, 16))
    q[:, 0], q[:, 1] = 0, 3
    x = (d0 * sc[:, None] * q - dm0 * mc[:, None]).astype(np.float32).reshape(1, 256)
    blk = oracle.quantize(oracle.Q2_K, x).reshape(84)
    want = np.zeros(84, dtype=np.uint8)
    want[0:16] = (sc | (mc << 4)).astype(np.uint8)
    for w in range(256):
        h, s, l = w // 128, (w // 32) % 4, w % 32
        want[16 + 32 * h + l] |= int(q.ravel()[w]) << (2 * s)
    want[80:82] = np.array([d0], dtype=np.float16).view(np.uint8)
    want[82:84] = np.array([dm0], dtype=np.float16).view(np.uint8)
    assert np.array_equal(blk, want)
    assert np.array_equal(oracle.dequantize(oracle.Q2_K, blk, 1, 256), x)


# ------------------------------------------------------------ scales and codes on random data
def nearest_binary16(bits, target):
    here = Fraction(float(np.uint16(bits).view(np.float16)))
    for nb in (int(bits) - 1, int(bits) + 1):
        other = Fraction(float(np.uint16(nb).view(np.float16)))
        if abs(other - target) < abs(here - target):
            return False
        if abs(other - target) == abs(here - target) and bits % 2 == 1:
            return False
    return True


def affine_stats(xb, levels):
    mx = xb.max(axis=1).astype(np.float32)
    mn = np.minimum(xb.min(axis=1), 0).astype(np.float32)
    s = ((mx - mn) / np.float32(levels)).astype(np.float32)
    m = (np.float32(0) - mn).astype(np.float32)
    return s, m


@pytest.mark.parametrize("fmt", [oracle.Q5_K, oracle.Q2_K])
def test_affine_scales_and_codes_are_nearest(fmt):
    x = inputs.weights(6, 1024, 41, fp32=True).numpy()
    nbytes = oracle.BLOCK[fmt][1]
    blocks = oracle.quantize(fmt, x).reshape(-1, nbytes)
    if fmt == oracle.Q5_K:
        nsub, length, levels, smax_code, qmax, walk = 8, 32, 31, 63, 31, q5_walk
        hdr = lambda b: (b[0:2], b[2:4])
    else:
        nsub, length, levels, smax_code, qmax, walk = 16, 16, 3, 15, 3, q2_walk
        hdr = lambda b: (b[80:82], b[82:84])
    for blk, xs in zip(blocks, x.reshape(-1, nsub, length)):
        d, dmin, sc, mc, q = walk(blk)
        s, m = affine_stats(xs, levels)
        db, mb = (int(h.view(np.uint16)[0]) for h in hdr(blk))
        assert nearest_binary16(db, Fraction(float(np.float32(s.max()) / np.float32(smax_code))))
        assert nearest_binary16(mb, Fraction(float(np.float32(m.max()) / np.float32(smax_code))))
        assert np.all(np.abs(s.astype(np.float64) / d - sc) <= 0.5 + 1e-6)
        assert np.all(np.abs(m.astype(np.float64) / dmin - mc) <= 0.5 + 1e-6)
        S = (np.float32(d) * sc.astype(np.float32)).astype(np.float64)
        Mn = (np.float32(dmin) * mc.astype(np.float32)).astype(np.float64)
        grid = S[:, None, None] * np.arange(qmax + 1)[None, None, :] - Mn[:, None, None]
        dist = np.abs(xs.astype(np.float64)[:, :, None] - grid)
        chosen = np.abs(xs.astype(np.float64) - (S[:, None] * q.reshape(nsub, length) - Mn[:, None]))
        slack = (S[:, None] + Mn[:, None]) * 2.0 ** -20
        assert np.all(chosen <= dist.min(axis=-1) + slack)


def test_q3_k_scales_and_codes_are_nearest():
    x = inputs.weights(6, 1024, 42, fp32=True).numpy()
    blocks = oracle.quantize(oracle.Q3_K, x).reshape(-1, 110)
    for blk, xs in zip(blocks, x.reshape(-1, 16, 16)):
        d, fields, q = q3_walk(blk)
        sc = fields - 32
        s = (np.abs(xs).max(axis=1).astype(np.float32) / np.float32(3)).astype(np.float32)
        db = int(blk[108:110].view(np.uint16)[0])
        assert nearest_binary16(db, Fraction(float(np.float32(s.max()) / np.float32(31))))
        assert np.all(np.abs(s.astype(np.float64) / d - sc) <= 0.5 + 1e-6)
        assert sc.min() >= 0 and sc.max() <= 31
        S = (np.float32(d) * sc.astype(np.float32)).astype(np.float64)
        grid = S[:, None, None] * (np.arange(8) - 4)[None, None, :]
        dist = np.abs(xs.astype(np.float64)[:, :, None] - grid)
        chosen = np.abs(xs.astype(np.float64) - S[:, None] * (q.reshape(16, 16) - 4))
        assert np.all(chosen <= dist.min(axis=-1) + S[:, None] * 2.0 ** -20)


# ------------------------------------------------------------ the rounding rule at exact half-steps
def test_q5_k_half_steps_round_away():
    # sub-block 0: q = 0 .. 31 span with S = 32 U (d = U, sc = 32 after
    # sub-block 1 fixes the superblock maximum at sc = 63); no negative values,
    # so Mn = 0; x = (k + 1/2) S gives (k + 1) away from zero
    x = np.zeros((8, 32), dtype=np.float32)
    x[1, 0] = 63 * 31 * U            # s_1 = 63 U -> d = U, sc_1 = 63
    x[0, 0] = 31 * 32 * U            # s_0 = 32 U -> sc_0 = 32, S_0 = 2^-5
    ks = [0, 1, 2, 5, 10, 29]
    for i, k in enumerate(ks):
        x[0, 1 + i] = (k + 0.5) * 32 * U
    x[2, 0] = 31 * 32.5 * U          # s_2 = 32.5 U -> sc_2 = 33 (even: 32)
    blk = oracle.quantize(oracle.Q5_K, x.reshape(1, 256)).reshape(176)
    d, dmin, sc, mc, q = q5_walk(blk)
    assert d == U and dmin == 0.0 and not mc.any()
    assert sc[0] == 32 and sc[1] == 63 and sc[2] == 33
    assert q.reshape(8, 32)[0, 1:1 + len(ks)].tolist() == [k + 1 for k in ks]


def test_q3_k_half_steps_round_away():
    x = np.zeros((16, 16), dtype=np.float32)
    x[0, 0] = 93 * U                 # s_0 = 31 U -> d = U, sc_0 = 31
    x[1, 0] = 48 * U                 # s_1 = 16 U -> sc_1 = 16, S_1 = 2^-6
    x[1, 1], x[1, 2] = 0.5 * 16 * U, 1.5 * 16 * U
    x[1, 3], x[1, 4] = -0.5 * 16 * U, -2.5 * 16 * U
    x[2, 0] = 3 * 10.5 * U           # s_2 = 10.5 U -> sc_2 = 11 (even: 10)
    blk = oracle.quantize(oracle.Q3_K, x.reshape(1, 256)).reshape(110)
    d, fields, q = q3_walk(blk)
    assert d == U and fields[0] == 63 and fields[1] == 48 and fields[2] == 32 + 11
    c = q.reshape(16, 16) - 4
    assert c[1, :5].tolist() == [3, 1, 2, -1, -3]


def test_q2_k_half_steps_round_away():
    x = np.zeros((16, 16), dtype=np.float32)
    x[0, 0] = 45 * U                 # s_0 = 15 U -> d = U, sc_0 = 15
    x[1, 0] = 3 * 8 * U              # s_1 = 8 U -> sc_1 = 8, S_1 = 2^-7
    x[1, 1], x[1, 2] = 0.5 * 8 * U, 1.5 * 8 * U
    x[2, 0] = 3 * 4.5 * U            # s_2 = 4.5 U -> sc_2 = 5 (even: 4)
    blk = oracle.quantize(oracle.Q2_K, x.reshape(1, 256)).reshape(84)
    d, dmin, sc, mc, q = q2_walk(blk)
    assert d == U and dmin == 0.0 and sc[0] == 15 and sc[1] == 8 and sc[2] == 5
    assert q.reshape(16, 16)[1, :3].tolist() == [3, 1, 2]


# ------------------------------------------------------------ degenerate superblocks and sources
@pytest.mark.parametrize("fmt", [oracle.Q5_K, oracle.Q3_K, oracle.Q2_K])
def test_zero_and_tiny_superblocks(fmt):
    z = oracle.quantize(fmt, np.zeros((2, 256), dtype=np.float32))
    assert not oracle.dequantize(fmt, z, 2, 256).any()
    tiny = np.full((1, 256), 1e-9, dtype=np.float32)  # scales underflow binary16
    assert not oracle.dequantize(fmt, oracle.quantize(fmt, tiny), 1, 256).any()
    if fmt == oracle.Q3_K:
        d, fields, q = q3_walk(z[0])
        assert d == 0.0 and np.all(fields == 32) and np.all(q == 4)


@pytest.mark.parametrize("fmt", [oracle.Q5_K, oracle.Q3_K, oracle.Q2_K])
def test_bf16_and_f32_sources_agree(fmt):
    w = inputs.weights(8, 1024, 43)
    assert np.array_equal(oracle.quantize(fmt, inputs.bf16_bits(w)), oracle.quantize(fmt, w.float().numpy()))
