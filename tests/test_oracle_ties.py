"""Pins for the oracle's rounding rule at exact half-steps.

The Q8_0 recipe this library follows rounds codes half away from zero (the
tiny Q8_0 linear workload: q = round-half-away(x / d)), and the Q4_K codes
(q, and the 6-bit scale and min codes sc_j, mc_j) use the same rule.  The
nearest-grid tests elsewhere accept either neighbour when the distances are
equal, so they cannot tell this rule from round-half-even.  Here every
quotient is built to land exactly on k + 1/2 (power-of-two scales, values
with few significant bits, so every fp32 step is exact) and the expected codes
are written out by hand: away from zero, which differs from the even
neighbour whenever k is even.
"""
import numpy as np

import oracle
from ggml_block_quantized_linear_b300 import inputs  # noqa: F401  (keeps the import order of the suite)
from test_oracle_q4_k import table_decode

# Q8_0: d0 = 2^-7, made the block scale by one value 127 * d0 per block; the
# other values are (h) * d0 with h a half-integer, so x / d = h exactly.
Q8_HALF_STEPS = [0.5, 2.5, 4.5, 10.5, 64.5, 126.5, -0.5, -2.5, -4.5, -10.5, -64.5, -126.5,
                 1.5, -1.5, 3.5, -3.5, 100.5, -100.5, 0.0, 8.5, -8.5, 32.5, -32.5, 50.5,
                 -50.5, 6.5, -6.5, 12.5, -12.5, 20.5, -20.5]


def away(h):
    return int(np.sign(h) * np.floor(abs(h) + 0.5))


def q8_0_tie_block():
    d0 = 2.0 ** -7
    x = np.array([127.0 * d0] + [h * d0 for h in Q8_HALF_STEPS], dtype=np.float32)
    assert x.size == 32
    want_q = [127] + [away(h) for h in Q8_HALF_STEPS]
    return x, want_q


def test_q8_0_half_steps_round_away_from_zero():
    x, want_q = q8_0_tie_block()
    rows = np.stack([x, -x])  # the mirrored block: -127 * d0 sets the same scale
    for src in (rows, inputs_bf16(rows)):
        packed = oracle.quantize(oracle.Q8_0, src).reshape(2, 34)
        for r, sign in ((0, 1), (1, -1)):
            # binary16 2^-7: exponent field 8, fraction 0 -> 0x2000, little-endian
            assert packed[r, 0] == 0x00 and packed[r, 1] == 0x20
            got = packed[r, 2:].view(np.int8).astype(int).tolist()
            assert got == [sign * w for w in want_q]
    # the even-neighbour rule would give 0 for 0.5, 2 for 2.5, -126 for -126.5
    assert want_q[1] == 1 and want_q[2] == 3 and want_q[12] == -127


def inputs_bf16(x32):
    """fp32 values that bf16 holds exactly, as bf16 bit patterns."""
    b = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32)
    assert np.all(b & 0xFFFF == 0)
    return (b >> 16).astype(np.uint16)


# Q4_K: one superblock whose scales come out as d = dmin = 2^-10.
U = 2.0 ** -10


def q4_k_tie_superblock():
    x = np.zeros((8, 32), dtype=np.float32)
    x[0, 0] = 945 * U           # s_0 = 945 U / 15 = 63 U: the largest s, so d = 63 U / 63 = U
    x[1, 0] = -63 * U           # m_1 = 63 U: the largest m, so dmin = U
    x[2, 0] = 615 * U / 2       # s_2 = 307.5 U / 15 = 20.5 U: sc_2 = 20.5 -> 21
    x[3, 0] = -12.5 * U         # m_3 = 12.5 U: mc_3 = 12.5 -> 13
    # sub-block 4: min 0 (Mn = 0), max 240 U -> s = 16 U, sc = 16, S = 2^-6;
    # values (k + 1/2) * 2^-6 give q = k + 1/2 exactly
    ks4 = [0, 2, 4, 6, 8, 10, 12, 14]
    x[4, 0] = 240 * U
    for i, k in enumerate(ks4):
        x[4, 1 + i] = (k + 0.5) * 16 * U
    # sub-block 5: min -4 U (m = 4 U, mc = 4, Mn = 4 U), max 116 U ->
    # s = 120 U / 15 = 8 U, sc = 8, S = 8 U; x = 8k U gives (x + Mn) / S = k + 1/2
    ks5 = [0, 2, 4, 6, 8, 10, 12, 14]
    x[5, 0] = -4 * U
    x[5, 1] = 116 * U
    for i, k in enumerate(ks5):
        x[5, 2 + i] = 8 * k * U
    # sub-blocks 6 and 7 stay zero
    return x.reshape(1, 256), ks4, ks5


def q4_k_codes(packed):
    """q[j][l] of one superblock: byte 32c + l holds sub-block 2c (low nibble)
    and 2c + 1 (high nibble)."""
    qb = packed[16:144]
    q = np.zeros((8, 32), dtype=int)
    for c in range(4):
        q[2 * c] = qb[32 * c:32 * c + 32] & 15
        q[2 * c + 1] = qb[32 * c:32 * c + 32] >> 4
    return q


def test_q4_k_half_steps_round_away():
    x, ks4, ks5 = q4_k_tie_superblock()
    packed = oracle.quantize(oracle.Q4_K, x).reshape(144)
    # d and dmin: binary16 2^-10 = exponent field 5 -> 0x1400
    assert packed[0:4].tolist() == [0x00, 0x14, 0x00, 0x14]
    sc, mc = table_decode(packed[4:16])
    sc, mc = [int(v) for v in sc], [int(v) for v in mc]
    assert sc[0] == 63 and mc[1] == 63
    assert sc[2] == 21          # 20.5 away from zero (even: 20)
    assert mc[3] == 13          # 12.5 away from zero (even: 12)
    assert sc[4] == 16 and mc[4] == 0
    assert sc[5] == 8 and mc[5] == 4
    assert sc[6] == sc[7] == mc[6] == mc[7] == 0
    q = q4_k_codes(packed)
    assert q[4, 0] == 15                                     # 240 U / 16 U = 15
    assert q[4, 1:9].tolist() == [k + 1 for k in ks4]        # k + 1/2 -> k + 1 (even: k)
    assert q[5, 0] == 0 and q[5, 1] == 15                    # (-4 + 4) / 8, (116 + 4) / 8
    assert q[5, 2:10].tolist() == [k + 1 for k in ks5]
    assert not q[6].any() and not q[7].any()


def test_q4_k_half_step_values_dequantize_on_the_upper_neighbour():
    # dequantized value of a half-step weight = S * (k + 1) - Mn: the upper
    # grid point, half a step above the input
    x, ks4, ks5 = q4_k_tie_superblock()
    packed = oracle.quantize(oracle.Q4_K, x)
    w = oracle.dequantize(oracle.Q4_K, packed, 1, 256).reshape(8, 32)
    x = x.reshape(8, 32)
    for i, k in enumerate(ks4):
        assert w[4, 1 + i] == (k + 1) * 16 * U
        assert w[4, 1 + i] - x[4, 1 + i] == 8 * U
    for i, k in enumerate(ks5):
        assert w[5, 2 + i] == 8 * (k + 1) * U - 4 * U
