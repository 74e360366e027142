"""GPU parity of FP8 E4M3 weights with a scale per row (W8A16).

ISQ codes, row scales and dequantized weights bit-identical to the CPU
oracle (IEEE division x / s, E4M3 rounding to nearest even with saturation),
including exact E4M3 midpoints, values past 448 before saturation, the
subnormal range, zero rows and odd counts of 256-wide chunks; the matmul
(decode kernel up to 16 tokens, tiled kernel above) within the per-element
tolerance of the other formats.
"""
import numpy as np
import pytest
import torch

import oracle
import ggml_block_quantized_linear_b300 as q
from ggml_block_quantized_linear_b300 import inputs
from qmm_testutil import DEV, bf16_from_bits, check_matmul, to_dev_u8

pytestmark = pytest.mark.gpu
F = q.QMM_FP8_E4M3


def cases():
    rng = np.random.default_rng(11)
    c = {}
    c["normal"] = inputs.weights(64, 1024, 71, fp32=True).numpy()
    c["odd_chunks"] = inputs.weights(37, 4352, 72, fp32=True).numpy()   # 17 chunks of 256
    c["one_chunk"] = inputs.weights(5, 256, 73, fp32=True).numpy()
    c["wide_range"] = (rng.normal(0, 1, (8, 512)) * np.exp2(rng.integers(-24, 8, (8, 512)))).astype(np.float32)
    c["zeros"] = np.zeros((2, 512), dtype=np.float32)
    c["constant"] = np.full((2, 512), -0.37, dtype=np.float32)
    # exact E4M3 midpoints: the row scale is s0 = 2^-8 (one value 448 s0)
    vals = oracle.e4m3_bits_to_f32(np.arange(0x7F, dtype=np.uint8))
    mids = ((vals[:-1].astype(np.float64) + vals[1:]) / 2)
    row = np.zeros(256, dtype=np.float64)
    row[:mids.size] = mids
    row[200] = 448.0
    row[201:201 + 20] = -mids[-20:]
    c["midpoints"] = (np.tile(row, (3, 2)) * 2.0 ** -8).astype(np.float32)
    # a scale that is not a power of two (amax 0.7): each E4M3 midpoint times s
    # and its float neighbours 1 and 2 ulps away, where x / s rounds next to a
    # rounding boundary of E4M3 (the quotient must be the IEEE one)
    sc = np.float32(np.float32(0.7) / np.float32(448.0))
    near = []
    for mval in mids:
        v = np.float32(mval * np.float64(sc))
        near += [v, np.nextafter(v, np.float32(1)), np.nextafter(v, np.float32(-1)),
                 np.nextafter(np.nextafter(v, np.float32(1)), np.float32(1)),
                 np.nextafter(np.nextafter(v, np.float32(-1)), np.float32(-1))]
    r2 = np.zeros(1024, dtype=np.float32)
    r2[0] = 0.7
    r2[1:1 + len(near)] = near
    c["near_midpoints"] = np.stack([r2, -r2, r2[::-1].copy()])
    return c


@pytest.mark.parametrize("name", sorted(cases()))
@pytest.mark.parametrize("src", ["f32", "bf16"])
def test_quantize_and_dequantize_bit_exact(name, src):
    x = cases()[name]
    if src == "bf16":
        t = torch.from_numpy(x).to(torch.bfloat16)
        want = oracle.quantize(oracle.FP8, inputs.bf16_bits(t))
        got = q.qmm_quantize(F, t.to(DEV)).cpu().numpy()
    else:
        want = oracle.quantize(oracle.FP8, x)
        got = q.qmm_quantize(F, torch.from_numpy(x).to(DEV)).cpu().numpy()
    assert np.array_equal(got, want)
    rows, cols = x.shape
    deq = q.qmm_dequantize(F, to_dev_u8(want), rows, cols).cpu().numpy()
    ref = oracle.dequantize(oracle.FP8, want, rows, cols)
    assert np.array_equal(deq.view(np.uint32), ref.view(np.uint32))


def problem(n, k, m, seed):
    w = inputs.weights(n, k, seed)
    packed = oracle.quantize(oracle.FP8, inputs.bf16_bits(w))
    xb = inputs.bf16_bits(inputs.activations(m, k, seed + 1))
    return packed, xb


@pytest.mark.parametrize("n,k", [(64, 256), (100, 512), (1024, 2304), (333, 4352), (2369, 1280)])
@pytest.mark.parametrize("m", [1, 3, 8, 9, 16, 17, 33, 100, 300])
def test_matmul_full(n, k, m):
    packed, xb = problem(n, k, m, 6000 + n + k + m)
    Y, A = oracle.matmul(oracle.FP8, packed, xb, n, k)
    y = q.qmm_matmul(F, to_dev_u8(packed), bf16_from_bits(xb), n)
    check_matmul(y, Y, A, "fp8 n=%d k=%d m=%d" % (n, k, m))
    assert torch.equal(y, q.qmm_matmul(F, to_dev_u8(packed), bf16_from_bits(xb), n))


@pytest.mark.parametrize("shape", inputs.DECODE_SHAPES)
@pytest.mark.parametrize("m", [1, 16, 64, 2048])
def test_matmul_full_shapes_sampled(shape, m):
    n, k = shape
    w = inputs.weights(n, k, 7000 + n + k, device=DEV)
    packed = q.qmm_quantize(F, w)
    x = inputs.activations(m, k, 7001 + m, device=DEV)
    y = q.qmm_matmul(F, packed, x, n)
    rows = np.array(sorted({0, 1, 63, 64, n // 2, n - 1}), dtype=np.int64)
    ridx = torch.from_numpy(rows).to(DEV)
    want = oracle.quantize(oracle.FP8, inputs.bf16_bits(w[ridx]))
    assert np.array_equal(packed[ridx].cpu().numpy(), want)
    Y, A = oracle.matmul(oracle.FP8, want, inputs.bf16_bits(x), rows.size, k)
    check_matmul(y[:, ridx], Y, A, "fp8 %s m=%d" % (shape, m))
    assert q.qmm_device_error_take() == 0


# ISQ rows staged in shared memory up to the largest row that fits twice
# (51200 bf16 values: 200 KB), and the direct kernel beyond (53248); fp32
# sources switch at half the length.
@pytest.mark.parametrize("rows,k,src", [(3, 51200, "bf16"), (3, 53248, "bf16"), (2, 25600, "f32"),
                                        (2, 26624, "f32")])
def test_quantize_long_rows(rows, k, src):
    x = inputs.weights(rows, k, 91 + k, fp32=True).numpy()
    if src == "bf16":
        t = torch.from_numpy(x).to(torch.bfloat16)
        want = oracle.quantize(oracle.FP8, inputs.bf16_bits(t))
        got = q.qmm_quantize(F, t.to(DEV)).cpu().numpy()
    else:
        want = oracle.quantize(oracle.FP8, x)
        got = q.qmm_quantize(F, torch.from_numpy(x).to(DEV)).cpu().numpy()
    assert np.array_equal(got, want)
    assert q.qmm_device_error_take() == 0
