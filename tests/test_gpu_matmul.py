"""GPU parity of qmm_matmul against the fp64 CPU oracle.

Tolerance per element: |y - y_ref| <= 1e-3 * sum_k |w^_k x_k| + 1e-6, with
y_ref and the sum computed by the oracle in fp64 over the exactly dequantized
weights.  Small shapes compare every output; the full decode / prefill shapes
compare sampled output features (all tokens) computed one by one.
"""
import numpy as np
import pytest
import torch

import oracle
import ggml_block_quantized_linear_b300 as q
from ggml_block_quantized_linear_b300 import inputs
from qmm_testutil import DEV, bf16_from_bits, check_matmul, to_dev_u8

pytestmark = pytest.mark.gpu
FMTS = [q.QMM_Q8_0, q.QMM_Q4_K]


def problem(fmt, n, k, m, seed):
    w = inputs.weights(n, k, seed)
    x = inputs.activations(m, k, seed)
    packed = oracle.quantize(fmt, inputs.bf16_bits(w))
    xb = inputs.bf16_bits(x)
    return packed, xb


def run(fmt, packed, xb, n):
    return q.qmm_matmul(fmt, to_dev_u8(packed), bf16_from_bits(xb), n)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("n,k", [(64, 256), (100, 512), (1024, 1792), (192, 4096), (333, 2304)])
@pytest.mark.parametrize("m", [1, 2, 4, 7, 8, 9, 16])
def test_decode_small_full(fmt, n, k, m):
    packed, xb = problem(fmt, n, k, m, 1000 + n + k + m)
    Y, A = oracle.matmul(fmt, packed, xb, n, k)
    check_matmul(run(fmt, packed, xb, n), Y, A, "fmt=%d n=%d k=%d m=%d" % (fmt, n, k, m))


# Shapes with at least one 16-row tile per SM take the persistent row-tile
# kernel (M <= 16, one or two 8-token MMA column tiles): one chunk per tile (seven idle consumer warps), a chunk
# count that is not a multiple of 8, more tiles than resident CTAs (CTAs
# loop over tiles), activations too many to hold at once (windows of K, with
# a one-chunk last window), and a ragged last tile; odd and even chunk
# counts (the 2-chunk copies then end on a half-filled or a full box).
# Windows (M * chunks > 256): 34 chunks in 32 + 2, 33 in 32 + 1, 56 in 48 + 8.
# With 1-2 tokens the kernel also takes grids of a quarter of the SMs
# (38 and 63 tiles, ragged).
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("n,k,m", [(2369, 256, 1), (2369, 256, 8), (9999, 1280, 2), (9999, 1280, 8),
                                   (3000, 4352, 5), (3000, 4352, 8), (12000, 4352, 8), (10000, 2304, 3),
                                   (2369, 512, 1), (10000, 2560, 3), (3000, 4608, 8), (12000, 4608, 1),
                                   (2400, 8704, 8), (2500, 8448, 8), (2400, 14336, 5),
                                   (2369, 256, 16), (9999, 1280, 12), (3000, 4608, 16), (2400, 4096, 9),
                                   (12000, 2304, 16), (600, 2304, 2), (1000, 4096, 1)])
def test_decode_row_tiles_full(fmt, n, k, m):
    packed, xb = problem(fmt, n, k, m, 2000 + n + k + m)
    Y, A = oracle.matmul(fmt, packed, xb, n, k)
    check_matmul(run(fmt, packed, xb, n), Y, A, "fmt=%d n=%d k=%d m=%d" % (fmt, n, k, m))


# More decode shapes checked in full and repeated bit for bit: ragged N, odd
# chunk counts (a half-filled last 2-chunk copy), fewer tiles than resident
# CTAs and a short last round of tiles, both decode kernels.
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("n,k,m", [(4000, 4096, 1), (4000, 4096, 4), (1100, 1280, 2), (3000, 2304, 4),
                                   (2500, 768, 1), (5000, 4096, 3), (1024, 4096, 1), (1024, 4096, 2),
                                   (2368, 3328, 8), (2600, 4096, 16), (7000, 512, 1), (300, 14336, 1)])
def test_decode_more_shapes_full(fmt, n, k, m):
    packed, xb = problem(fmt, n, k, m, 3000 + n + k + m)
    Y, A = oracle.matmul(fmt, packed, xb, n, k)
    w, x = to_dev_u8(packed), bf16_from_bits(xb)
    y = q.qmm_matmul(fmt, w, x, n)
    check_matmul(y, Y, A, "fmt=%d n=%d k=%d m=%d" % (fmt, n, k, m))
    for _ in range(2):
        assert torch.equal(q.qmm_matmul(fmt, w, x, n), y)
    assert q.qmm_device_error_take() == 0


@pytest.mark.parametrize("fmt", FMTS)
def test_tiny_linear_config(fmt):
    # fp32 W 256 x 512 quantized, X bf16 1 x 512
    w = inputs.weights(256, 512, inputs.seed_for(1), fp32=True)
    packed = oracle.quantize(fmt, w.numpy())
    xb = inputs.bf16_bits(inputs.activations(1, 512, inputs.seed_for(1)))
    Y, A = oracle.matmul(fmt, packed, xb, 256, 512)
    check_matmul(run(fmt, packed, xb, 256), Y, A)


def sample_rows(n, count, seed):
    rng = np.random.default_rng(seed)
    s = set(rng.choice(n, size=min(count, n), replace=False).tolist())
    s.update([0, n - 1, min(63, n - 1), min(64, n - 1)])
    return np.array(sorted(s), dtype=np.int64)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", inputs.DECODE_SHAPES)
@pytest.mark.parametrize("m", inputs.DECODE_MS)
def test_decode_full_shapes_sampled(fmt, shape, m):
    n, k = shape
    cfg = 2 if fmt == q.QMM_Q8_0 else 3
    si, mi = inputs.DECODE_SHAPES.index(shape), inputs.DECODE_MS.index(m)
    w = inputs.weights(n, k, inputs.seed_for(cfg, si))
    packed = oracle.quantize(fmt, inputs.bf16_bits(w))
    xb = inputs.bf16_bits(inputs.activations(m, k, inputs.seed_for(cfg, si, mi)))
    y = run(fmt, packed, xb, n).cpu()
    ns = sample_rows(n, 192, si * 10 + mi)
    Y, A = oracle.matmul_columns(fmt, packed, xb, k, ns)
    check_matmul(y[:, torch.from_numpy(ns)], Y, A, "fmt=%d %s m=%d" % (fmt, shape, m))


@pytest.mark.parametrize("fmt", FMTS)
def test_one_hot_and_zero(fmt):
    n, k = 130, 1024
    packed, _ = problem(fmt, n, k, 1, 5)
    cols = [0, 1, 255, 256, 700, 1023, 31, 32, 33, 512, 513, 1000, 100, 200, 300, 400]
    x = torch.zeros((len(cols), k), dtype=torch.bfloat16)
    for i, c in enumerate(cols):
        x[i, c] = 1.0
    xb = inputs.bf16_bits(x)
    Y, A = oracle.matmul(fmt, packed, xb, n, k)
    y = run(fmt, packed, xb, n)
    check_matmul(y, Y, A, "one-hot")
    if fmt == q.QMM_Q8_0:  # d * q survives the offset arithmetic exactly
        assert np.array_equal(y.cpu().double().numpy(), Y)
    zp = oracle.quantize(fmt, np.zeros((n, k), dtype=np.float32))
    xb2 = inputs.bf16_bits(inputs.activations(16, k, 3))
    assert not run(fmt, zp, xb2, n).cpu().any()


@pytest.mark.parametrize("fmt", FMTS)
def test_deterministic_and_stream(fmt):
    n, k, m = 4096, 4096, 4
    packed, xb = problem(fmt, n, k, m, 77)
    s = torch.cuda.Stream()
    w, x = to_dev_u8(packed), bf16_from_bits(xb)
    with torch.cuda.stream(s):
        a = q.qmm_matmul(fmt, w, x, n)
        b = q.qmm_matmul(fmt, w, x, n)
    s.synchronize()
    assert torch.equal(a, b)
    assert q.qmm_device_error_take() == 0


@pytest.mark.parametrize("fmt", FMTS)
def test_activation_range(fmt):
    n, k = 64, 512
    packed, _ = problem(fmt, n, k, 1, 11)
    rng = np.random.default_rng(4)
    x = torch.from_numpy(rng.normal(0, 1, (3, k)).astype(np.float32))
    x[0] *= 3000.0          # large but inside binary16 range
    x[1] *= 1e-3
    x[2, ::3] = 0.0
    xb = inputs.bf16_bits(x.to(torch.bfloat16))
    Y, A = oracle.matmul(fmt, packed, xb, n, k)
    check_matmul(run(fmt, packed, xb, n), Y, A, "range")


# ---------------------------------------------------------------- prefill GEMM
# Output grids filling under half of the SMs split K (each output tile is a
# few units whose partial tiles the last one to finish adds in order): 16 and
# 20 weight tiles x 2-3 token tiles; the last also has a Y size that is not a
# multiple of 4.
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("n,k,m", [(2048, 512, 513), (2560, 1024, 257), (2047, 512, 301)])
def test_prefill_split_k_full(fmt, n, k, m):
    packed, xb = problem(fmt, n, k, m, 3000 + n + k + m)
    Y, A = oracle.matmul(fmt, packed, xb, n, k)
    y = run(fmt, packed, xb, n)
    check_matmul(y, Y, A, "fmt=%d n=%d k=%d m=%d" % (fmt, n, k, m))
    assert torch.equal(y, run(fmt, packed, xb, n))  # parts added in a fixed order


# 256-token tiles with a ragged last token tile (1000 = 3 x 256 + 232;
# 1500 = 5 x 256 + 220; 1100 = 4 x 256 + 76): 128 and 96 tiles take K halves
# added onto a zeroed Y; 160 tiles (4096 x 1100) run whole, in two waves.
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("n,k,m", [(4096, 512, 1000), (2048, 1024, 1500), (4096, 512, 1100)])
def test_prefill_256_token_ragged_full(fmt, n, k, m):
    packed, xb = problem(fmt, n, k, m, 5000 + n + k + m)
    Y, A = oracle.matmul(fmt, packed, xb, n, k)
    y = run(fmt, packed, xb, n)
    check_matmul(y, Y, A, "fmt=%d n=%d k=%d m=%d" % (fmt, n, k, m))
    assert torch.equal(y, run(fmt, packed, xb, n))


# Stream-K (256-token tiles, four waves or more on the 148 SMs): each CTA
# runs an equal share of the (tile, packed group) pairs, and a tile cut
# between two CTAs is the sum of both parts on a zeroed Y.  600 tiles of 2
# groups and 608 of 3 (in the second N is ragged and not a multiple of 4, and
# M is ragged); all four formats of the tiled kernel, compared in full, and
# run twice.
@pytest.mark.parametrize("fmt", FMTS + [q.QMM_Q5_K, q.QMM_FP8_E4M3])
@pytest.mark.parametrize("n,k,m", [(9600, 512, 2048), (9602, 768, 1900)])
def test_prefill_stream_k_full(fmt, n, k, m):
    packed, xb = problem(fmt, n, k, m, 8000 + n + k + m)
    Y, A = oracle.matmul(fmt, packed, xb, n, k)
    y = run(fmt, packed, xb, n)
    check_matmul(y, Y, A, "fmt=%d n=%d k=%d m=%d" % (fmt, n, k, m))
    assert torch.equal(y, run(fmt, packed, xb, n))  # two parts on zero: either order, the same sum
    assert q.qmm_device_error_take() == 0


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("n,k", [(128, 256), (200, 512), (384, 1024), (130, 2304)])
@pytest.mark.parametrize("m", [17, 64, 255, 256, 300])
def test_prefill_small_full(fmt, n, k, m):
    packed, xb = problem(fmt, n, k, m, 3000 + n + k + m)
    Y, A = oracle.matmul(fmt, packed, xb, n, k)
    check_matmul(run(fmt, packed, xb, n), Y, A, "fmt=%d n=%d k=%d m=%d" % (fmt, n, k, m))


# Mid-size batches (continuous batching, 17 <= M < 256): the token tile is
# 32, 64, 128 or 256 (the smallest of 32 / 64 / 128 holding M, else 256) and
# K is split into as many parts as fill the SMs (up to one part per 256-wide
# group), the last part of each tile adding all parts in order.  Tile
# boundaries (32 / 33, 64 / 65, 128 / 129), one-group parts, uneven parts
# (groups not a multiple of the part count) and ragged N.
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("n,k", [(128, 256), (300, 1280), (1024, 4096), (130, 2304)])
@pytest.mark.parametrize("m", [17, 32, 33, 64, 65, 100, 128, 129, 200])
def test_mid_batch_full(fmt, n, k, m):
    packed, xb = problem(fmt, n, k, m, 4000 + n + k + m)
    Y, A = oracle.matmul(fmt, packed, xb, n, k)
    y = run(fmt, packed, xb, n)
    check_matmul(y, Y, A, "fmt=%d n=%d k=%d m=%d" % (fmt, n, k, m))
    assert torch.equal(y, run(fmt, packed, xb, n))  # same parts, same order


# Long rows (K >= 12288) at 9-16 tokens: FP8 and Q5_K from 9 tokens and
# Q8_0 from 12 take the tiled kernel, the others (and shorter rows) the
# decode kernels; both sides of each threshold, compared in full.
@pytest.mark.parametrize("fmt", FMTS + [q.QMM_Q5_K, q.QMM_FP8_E4M3])
@pytest.mark.parametrize("n,k,m", [(300, 14336, 8), (300, 14336, 9), (300, 14336, 11), (300, 12288, 12),
                                   (257, 14336, 16), (300, 11264, 16)])
def test_long_rows_decode_batches_full(fmt, n, k, m):
    packed, xb = problem(fmt, n, k, m, 9500 + n + k + m)
    Y, A = oracle.matmul(fmt, packed, xb, n, k)
    y = run(fmt, packed, xb, n)
    check_matmul(y, Y, A, "fmt=%d n=%d k=%d m=%d" % (fmt, n, k, m))
    assert torch.equal(y, run(fmt, packed, xb, n))
    assert q.qmm_device_error_take() == 0


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", inputs.DECODE_SHAPES)
@pytest.mark.parametrize("m", [17, 32, 64, 128])
def test_mid_batch_decode_shapes_sampled(fmt, shape, m):
    n, k = shape
    si = inputs.DECODE_SHAPES.index(shape)
    w = inputs.weights(n, k, inputs.seed_for(6, si))
    packed = oracle.quantize(fmt, inputs.bf16_bits(w))
    xb = inputs.bf16_bits(inputs.activations(m, k, inputs.seed_for(6, si, m)))
    y = run(fmt, packed, xb, n).cpu()
    ns = sample_rows(n, 40, 200 + si * 10 + m)
    Y, A = oracle.matmul_columns(fmt, packed, xb, k, ns)
    check_matmul(y[:, torch.from_numpy(ns)], Y, A, "fmt=%d %s m=%d" % (fmt, shape, m))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", inputs.PREFILL_SHAPES)
@pytest.mark.parametrize("m", inputs.PREFILL_MS)
def test_prefill_full_shapes_sampled(fmt, shape, m):
    n, k = shape
    si, mi = inputs.PREFILL_SHAPES.index(shape), inputs.PREFILL_MS.index(m)
    w = inputs.weights(n, k, inputs.seed_for(4, si))
    packed = oracle.quantize(fmt, inputs.bf16_bits(w))
    xb = inputs.bf16_bits(inputs.activations(m, k, inputs.seed_for(4, si, mi)))
    y = run(fmt, packed, xb, n).cpu()
    ns = sample_rows(n, 40, 100 + si * 10 + mi)
    Y, A = oracle.matmul_columns(fmt, packed, xb, k, ns)
    check_matmul(y[:, torch.from_numpy(ns)], Y, A, "fmt=%d %s m=%d" % (fmt, shape, m))


@pytest.mark.parametrize("fmt", FMTS)
def test_prefill_one_hot_and_determinism(fmt):
    n, k = 256, 1024
    packed, _ = problem(fmt, n, k, 1, 8)
    cols = list(range(0, 1024, 17))[:40]
    x = torch.zeros((len(cols), k), dtype=torch.bfloat16)
    for i, c in enumerate(cols):
        x[i, c] = 1.0
    xb = inputs.bf16_bits(x)
    Y, A = oracle.matmul(fmt, packed, xb, n, k)
    y1 = run(fmt, packed, xb, n)
    y2 = run(fmt, packed, xb, n)
    check_matmul(y1, Y, A, "one-hot prefill")
    assert torch.equal(y1, y2)
    assert q.qmm_device_error_take() == 0
