"""GPU parity of the K-quants Q5_K, Q3_K and Q2_K (the page's q5k / q3k / q2k).

ISQ bytes and dequantized weights bit-identical to the CPU oracle (bf16 and
fp32 sources, exact half-steps, inputs on the grid, degenerate superblocks,
rows whose superblocks are only 2- or 4-byte aligned), the matmul within the
per-element tolerance for decode and prefill batch sizes, the embedding rows
exact, and the sensitive-tensor policy's head type for each model type.
"""
import numpy as np
import pytest
import torch

import oracle
import ggml_block_quantized_linear_b300 as q
from ggml_block_quantized_linear_b300 import inputs
from qmm_testutil import DEV, bf16_from_bits, check_matmul, to_dev_u8

pytestmark = pytest.mark.gpu
FMTS = [q.QMM_Q5_K, q.QMM_Q3_K, q.QMM_Q2_K]
U = 2.0 ** -10


def cases():
    rng = np.random.default_rng(19)
    c = {}
    c["normal"] = inputs.weights(64, 1024, 71, fp32=True).numpy()
    c["odd_superblocks"] = inputs.weights(37, 768, 72, fp32=True).numpy()
    c["wide_range"] = (rng.normal(0, 1, (8, 512)) * np.exp2(rng.integers(-20, 8, (8, 512)))).astype(np.float32)
    c["zeros"] = np.zeros((2, 512), dtype=np.float32)
    c["tiny"] = (rng.normal(0, 1e-7, (4, 256))).astype(np.float32)
    c["constant"] = np.full((2, 512), -0.37, dtype=np.float32)
    c["positive"] = np.abs(inputs.weights(8, 512, 73, fp32=True).numpy())
    # exact half-steps of each quantizer (see the oracle pins)
    h5 = np.zeros((8, 32), dtype=np.float32)
    h5[1, 0], h5[0, 0], h5[2, 0] = 63 * 31 * U, 31 * 32 * U, 31 * 32.5 * U
    for i, k in enumerate([0, 1, 2, 5, 10, 29]):
        h5[0, 1 + i] = (k + 0.5) * 32 * U
    h3 = np.zeros((16, 16), dtype=np.float32)
    h3[0, 0], h3[1, 0], h3[2, 0] = 93 * U, 48 * U, 3 * 10.5 * U
    h3[1, 1:5] = [0.5 * 16 * U, 1.5 * 16 * U, -0.5 * 16 * U, -2.5 * 16 * U]
    h2 = np.zeros((16, 16), dtype=np.float32)
    h2[0, 0], h2[1, 0], h2[2, 0] = 45 * U, 24 * U, 13.5 * U
    h2[1, 1:3] = [0.5 * 8 * U, 1.5 * 8 * U]
    c["half_steps"] = np.concatenate([h5.reshape(1, 256), h3.reshape(1, 256), h2.reshape(1, 256)], axis=0)
    return c


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("name", sorted(cases()))
@pytest.mark.parametrize("src", ["f32", "bf16"])
def test_quantize_and_dequantize_bit_exact(fmt, name, src):
    x = cases()[name]
    if src == "bf16":
        t = torch.from_numpy(x).to(torch.bfloat16)
        want = oracle.quantize(fmt, inputs.bf16_bits(t))
        got = q.qmm_quantize(fmt, t.to(DEV)).cpu().numpy()
    else:
        want = oracle.quantize(fmt, x)
        got = q.qmm_quantize(fmt, torch.from_numpy(x).to(DEV)).cpu().numpy()
    assert np.array_equal(got.reshape(-1), want.reshape(-1))
    rows, cols = x.shape
    deq = q.qmm_dequantize(fmt, to_dev_u8(want), rows, cols).cpu().numpy()
    ref = oracle.dequantize(fmt, want, rows, cols)
    assert np.array_equal(deq.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("fmt", FMTS)
def test_decode_shape_bit_exact(fmt):
    w = inputs.weights(4096, 4096, 74)
    got = q.qmm_quantize(fmt, w.to(DEV)).cpu().numpy()
    assert np.array_equal(got, oracle.quantize(fmt, inputs.bf16_bits(w)))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("n,k", [(64, 256), (131, 768), (300, 4096), (77, 2304)])
@pytest.mark.parametrize("m", [1, 3, 8, 9, 16, 17, 40])
def test_matmul_full(fmt, n, k, m):
    w = inputs.weights(n, k, 75 + n + k)
    packed = oracle.quantize(fmt, inputs.bf16_bits(w))
    xb = inputs.bf16_bits(inputs.activations(m, k, 76 + m))
    Y, A = oracle.matmul(fmt, packed, xb, n, k)
    y = q.qmm_matmul(fmt, to_dev_u8(packed), bf16_from_bits(xb), n)
    check_matmul(y, Y, A, "fmt=%d n=%d k=%d m=%d" % (fmt, n, k, m))
    assert torch.equal(y, q.qmm_matmul(fmt, to_dev_u8(packed), bf16_from_bits(xb), n))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", inputs.DECODE_SHAPES)
def test_decode_shapes_sampled(fmt, shape):
    n, k = shape
    w = inputs.weights(n, k, 77, device=DEV)
    packed = q.qmm_quantize(fmt, w)
    for m in (1, 16):
        x = inputs.activations(m, k, 78 + m, device=DEV)
        y = q.qmm_matmul(fmt, packed, x, n)
        rng = np.random.default_rng(n + k + m)
        rows = np.unique(np.concatenate([rng.choice(n, 24, replace=False), [0, n - 1]])).astype(np.int64)
        ridx = torch.from_numpy(rows).to(DEV)
        want = oracle.quantize(fmt, inputs.bf16_bits(w[ridx]))
        assert np.array_equal(packed[ridx].cpu().numpy(), want)
        Y, A = oracle.matmul(fmt, want, inputs.bf16_bits(x), rows.size, k)
        check_matmul(y[:, ridx], Y, A, "fmt=%d %s m=%d" % (fmt, shape, m))
    assert q.qmm_device_error_take() == 0


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("V,D", [(300, 4096), (37, 768)])
def test_embedding_lookup(fmt, V, D):
    w = inputs.weights(V, D, 79)
    packed = oracle.quantize(fmt, inputs.bf16_bits(w))
    rng = np.random.default_rng(80)
    ids = np.concatenate([rng.integers(0, V, 50), [0, V - 1, 3, 3]]).astype(np.int64)
    want = oracle.gather(fmt, packed, V, D, ids)
    table = to_dev_u8(packed)
    dids = torch.from_numpy(ids).to(DEV)
    got = q.qmm_embedding(fmt, table, dids, D).cpu().numpy()
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    gotb = q.qmm_embedding(fmt, table, dids, D, dtype=torch.bfloat16).cpu()
    assert torch.equal(gotb.view(torch.int16), torch.from_numpy(want).to(torch.bfloat16).view(torch.int16))
    bad = torch.tensor([1, V], dtype=torch.int64, device=DEV)
    out = q.qmm_embedding(fmt, table, bad, D).cpu().numpy()
    assert q.qmm_device_error_take() == q.QMM_DEVERR_EMBEDDING_ID
    assert np.array_equal(out[0], want[np.where(ids == 1)[0][0]] if (ids == 1).any()
                          else oracle.gather(fmt, packed, V, D, np.array([1]))[0])
    assert not out[1].any()
    assert q.qmm_device_error_take() == 0


@pytest.mark.parametrize("model,head", [(q.QMM_Q2_K, q.QMM_Q6_K), (q.QMM_Q3_K, q.QMM_Q6_K),
                                        (q.QMM_Q5_K, q.QMM_Q8_0)])
def test_output_head_type_of_each_model(model, head):
    # the sensitive-tensor policy gives the head its type; the head at M = 1 in that type
    assert q.qmm_embedding_format(model) == head
    V, D = 3000, 4096
    w = inputs.weights(V, D, 81, device=DEV)
    packed = q.qmm_quantize(head, w)
    x = inputs.activations(1, D, 82, device=DEV)
    y = q.qmm_matmul(head, packed, x, V)
    rows = np.array([0, 5, 1499, 2999], dtype=np.int64)
    ridx = torch.from_numpy(rows).to(DEV)
    want = oracle.quantize(head, inputs.bf16_bits(w[ridx]))
    Y, A = oracle.matmul(head, want, inputs.bf16_bits(x), rows.size, D)
    check_matmul(y[:, ridx], Y, A, "head")


# One token on the TMA-fed kernel (rows a 16-byte multiple): ragged row tiles
# (N not a multiple of 8), several 8-superblock stages, a partial last stage
# (Q2_K, 12 superblocks), many tiles per CTA (N = 9000), and K = 14336.
@pytest.mark.parametrize("fmt,n,k", [(q.QMM_Q3_K, 300, 4096), (q.QMM_Q2_K, 300, 4096), (q.QMM_Q2_K, 77, 3072),
                                     (q.QMM_Q3_K, 1001, 14336), (q.QMM_Q2_K, 1001, 14336),
                                     (q.QMM_Q6_K, 301, 4096), (q.QMM_Q6_K, 203, 14336),
                                     (q.QMM_Q3_K, 9000, 2048), (q.QMM_Q6_K, 9000, 2048)])
def test_one_token_tma_path(fmt, n, k):
    w = inputs.weights(n, k, 83 + n + k)
    packed = oracle.quantize(fmt, inputs.bf16_bits(w))
    xb = inputs.bf16_bits(inputs.activations(1, k, 84))
    Y, A = oracle.matmul(fmt, packed, xb, n, k)
    y = q.qmm_matmul(fmt, to_dev_u8(packed), bf16_from_bits(xb), n)
    check_matmul(y, Y, A, "fmt=%d n=%d k=%d" % (fmt, n, k))
    # repeated and chained calls stay identical (persistent CTAs, dependent launches)
    y2 = q.qmm_matmul(fmt, to_dev_u8(packed), bf16_from_bits(xb), n)
    assert torch.equal(y, y2)
    assert q.qmm_device_error_take() == 0


# Rows that are not 16-byte multiples take the direct-load kernel (Q3_K and
# Q2_K with 12 superblocks: 1320 bytes; Q2_K's 1008 bytes are a multiple and
# take the TMA path); one token on the direct-load kernel forms each row's sum
# exactly as the TMA path does, which a TMA-path row of the same weights shows.
def test_one_token_fallback_and_same_order():
    n, k = 129, 3072
    w = inputs.weights(n, k, 85)
    xb = inputs.bf16_bits(inputs.activations(1, k, 86))
    for fmt in (q.QMM_Q3_K, q.QMM_Q2_K):
        packed = oracle.quantize(fmt, inputs.bf16_bits(w))
        Y, A = oracle.matmul(fmt, packed, xb, n, k)
        check_matmul(q.qmm_matmul(fmt, to_dev_u8(packed), bf16_from_bits(xb), n), Y, A, "fmt=%d" % fmt)
    # Q3_K rows of 16 superblocks (TMA path) against the same superblocks as the
    # first 16 of 20 (a 2200-byte row: direct loads) with zero activations beyond
    w2 = inputs.weights(n, 5120, 88)
    x2 = inputs.activations(1, 5120, 89)
    x2[:, 4096:] = 0
    p2 = q.qmm_quantize(q.QMM_Q3_K, w2.to(DEV))
    y_direct = q.qmm_matmul(q.QMM_Q3_K, p2, x2.to(DEV), n)
    p1 = q.qmm_quantize(q.QMM_Q3_K, w2[:, :4096].contiguous().to(DEV))
    y_tma = q.qmm_matmul(q.QMM_Q3_K, p1, x2[:, :4096].contiguous().to(DEV), n)
    assert torch.equal(y_direct, y_tma)


# One token with a K whose activations do not fit the TMA-fed kernel's
# shared memory (K * 2 bytes > 64 KB): the direct-load kernel takes it.
@pytest.mark.parametrize("fmt,k", [(q.QMM_Q6_K, 34816), (q.QMM_Q2_K, 33792), (q.QMM_Q3_K, 34816)])
def test_one_token_long_k(fmt, k):
    n = 64
    w = inputs.weights(n, k, 93)
    packed = oracle.quantize(fmt, inputs.bf16_bits(w))
    xb = inputs.bf16_bits(inputs.activations(1, k, 94))
    Y, A = oracle.matmul(fmt, packed, xb, n, k)
    y = q.qmm_matmul(fmt, to_dev_u8(packed), bf16_from_bits(xb), n)
    check_matmul(y, Y, A, "fmt=%d k=%d" % (fmt, k))
    assert q.qmm_device_error_take() == 0


# Q5_K prefill on the tiled tensor-core kernel at decode and prefill shapes
# (a K split at 512 tokens on 4096 x 4096, 2048 tokens filling the SMs, a
# 300-token ragged tile on K = 14336): sampled rows, every token.
@pytest.mark.parametrize("n,k,m", [(4096, 4096, 512), (14336, 4096, 2048), (4096, 14336, 300), (1024, 4096, 40)])
def test_q5_k_prefill_sampled(n, k, m):
    w = inputs.weights(n, k, 95 + m, device=DEV)
    packed = q.qmm_quantize(q.QMM_Q5_K, w)
    x = inputs.activations(m, k, 96 + m, device=DEV)
    y = q.qmm_matmul(q.QMM_Q5_K, packed, x, n)
    rng = np.random.default_rng(n + k + m)
    rows = np.unique(np.concatenate([rng.choice(n, 16, replace=False), [0, 127, 128, n - 1]])).astype(np.int64)
    ridx = torch.from_numpy(rows).to(DEV)
    want = oracle.quantize(q.QMM_Q5_K, inputs.bf16_bits(w[ridx]))
    assert np.array_equal(packed[ridx].cpu().numpy(), want)
    Y, A = oracle.matmul(q.QMM_Q5_K, want, inputs.bf16_bits(x), rows.size, k)
    check_matmul(y[:, ridx], Y, A, "Q5_K n=%d k=%d m=%d" % (n, k, m))
    assert torch.equal(y, q.qmm_matmul(q.QMM_Q5_K, packed, x, n))
    assert q.qmm_device_error_take() == 0
