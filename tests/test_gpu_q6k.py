"""GPU parity of the Q6_K format and of the quantized embedding lookup.

Q6_K (the type the pages' "Sensitive tensor precision" section gives the
token embeddings and output head of a Q4K model): ISQ bytes and dequantized
weights bit-identical to the CPU oracle, including exact half-steps,
on-grid inputs and superblocks that are only 2-byte aligned in a row
(K / 256 odd); the matmul within the per-element tolerance of the other
formats.  Embedding lookup, every format: fp32 rows bit-identical to the
oracle's dequantized rows, bf16 rows equal to those values rounded to
nearest even; an id outside the table writes zeros and records its code.
"""
import numpy as np
import pytest
import torch

import oracle
import ggml_block_quantized_linear_b300 as q
from ggml_block_quantized_linear_b300 import inputs
from qmm_testutil import DEV, bf16_from_bits, check_matmul, to_dev_u8

pytestmark = pytest.mark.gpu


def cases():
    rng = np.random.default_rng(9)
    c = {}
    c["normal"] = inputs.weights(64, 1024, 61, fp32=True).numpy()
    c["odd_superblocks"] = inputs.weights(37, 768, 62, fp32=True).numpy()  # 630-byte rows
    c["wide_range"] = (rng.normal(0, 1, (8, 512)) * np.exp2(rng.integers(-20, 8, (8, 512)))).astype(np.float32)
    c["zeros"] = np.zeros((2, 512), dtype=np.float32)
    c["tiny"] = (rng.normal(0, 1e-7, (4, 256))).astype(np.float32)
    c["constant"] = np.full((2, 512), -0.37, dtype=np.float32)
    ties = np.zeros((16, 16), dtype=np.float32)
    u = 2.0 ** -10
    ties[0, 0] = 3937 * u
    ties[1, 0] = 1271 * u / 2
    ties[2, 0] = 496 * u
    for i, k in enumerate([0, 2, 4, 10, 20, 30]):
        ties[2, 1 + i] = (k + 0.5) * 16 * u
        ties[2, 8 + i] = -(k + 0.5) * 16 * u
    c["half_steps"] = np.tile(ties.reshape(1, 256), (3, 2))
    d0 = 2.0 ** -9
    sc = rng.integers(1, 128, 16)
    sc[3] = 127
    cc = rng.integers(-31, 32, (16, 16))
    cc[:, 0] = 31
    c["on_grid"] = (d0 * sc[:, None] * cc).astype(np.float32).reshape(1, 256)
    return c


@pytest.mark.parametrize("name", sorted(cases()))
@pytest.mark.parametrize("src", ["f32", "bf16"])
def test_quantize_and_dequantize_bit_exact(name, src):
    x = cases()[name]
    if src == "bf16":
        t = torch.from_numpy(x).to(torch.bfloat16)
        want = oracle.quantize(oracle.Q6_K, inputs.bf16_bits(t))
        got = q.qmm_quantize(q.QMM_Q6_K, t.to(DEV)).cpu().numpy()
    else:
        want = oracle.quantize(oracle.Q6_K, x)
        got = q.qmm_quantize(q.QMM_Q6_K, torch.from_numpy(x).to(DEV)).cpu().numpy()
    assert np.array_equal(got.reshape(-1), want.reshape(-1))
    rows, cols = x.shape
    deq = q.qmm_dequantize(q.QMM_Q6_K, to_dev_u8(want), rows, cols).cpu().numpy()
    ref = oracle.dequantize(oracle.Q6_K, want, rows, cols)
    assert np.array_equal(deq.view(np.uint32), ref.view(np.uint32))


def test_decode_shape_bit_exact():
    w = inputs.weights(4096, 4096, 63)
    got = q.qmm_quantize(q.QMM_Q6_K, w.to(DEV)).cpu().numpy()
    assert np.array_equal(got, oracle.quantize(oracle.Q6_K, inputs.bf16_bits(w)))


@pytest.mark.parametrize("n,k", [(64, 256), (131, 768), (300, 4096), (77, 2304)])
@pytest.mark.parametrize("m", [1, 3, 8, 9, 16, 17, 40])
def test_matmul_full(n, k, m):
    w = inputs.weights(n, k, 64 + n + k)
    packed = oracle.quantize(oracle.Q6_K, inputs.bf16_bits(w))
    xb = inputs.bf16_bits(inputs.activations(m, k, 65 + m))
    Y, A = oracle.matmul(oracle.Q6_K, packed, xb, n, k)
    y = q.qmm_matmul(q.QMM_Q6_K, to_dev_u8(packed), bf16_from_bits(xb), n)
    check_matmul(y, Y, A, "q6_k n=%d k=%d m=%d" % (n, k, m))
    assert torch.equal(y, q.qmm_matmul(q.QMM_Q6_K, to_dev_u8(packed), bf16_from_bits(xb), n))


def test_output_head_of_a_q4_k_model():
    # the sensitive-tensor policy: a Q4_K model's output head is Q6_K; a
    # vocabulary-sized head at M = 1, sampled rows
    fmt = q.qmm_embedding_format(q.QMM_Q4_K)
    assert fmt == q.QMM_Q6_K
    V, D = 32000, 4096
    w = inputs.weights(V, D, 66, device=DEV)
    packed = q.qmm_quantize(fmt, w)
    x = inputs.activations(1, D, 67, device=DEV)
    y = q.qmm_matmul(fmt, packed, x, V)
    rows = np.array([0, 1, 777, 15999, 31998, 31999], dtype=np.int64)
    ridx = torch.from_numpy(rows).to(DEV)
    want = oracle.quantize(fmt, inputs.bf16_bits(w[ridx]))
    assert np.array_equal(packed[ridx].cpu().numpy(), want)
    Y, A = oracle.matmul(fmt, want, inputs.bf16_bits(x), rows.size, D)
    check_matmul(y[:, ridx], Y, A, "output head")


@pytest.mark.parametrize("fmt", [q.QMM_Q8_0, q.QMM_Q4_K, q.QMM_Q6_K, q.QMM_FP8_E4M3])
@pytest.mark.parametrize("V,D", [(1000, 4096), (37, 768)])
def test_embedding_lookup(fmt, V, D):
    w = inputs.weights(V, D, 68)
    packed = oracle.quantize(fmt, inputs.bf16_bits(w))
    rng = np.random.default_rng(69)
    ids = np.concatenate([rng.integers(0, V, 50), [0, V - 1, 3, 3]]).astype(np.int64)
    want = oracle.gather(fmt, packed, V, D, ids)
    table = to_dev_u8(packed)
    dids = torch.from_numpy(ids).to(DEV)
    got = q.qmm_embedding(fmt, table, dids, D).cpu().numpy()
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    gotb = q.qmm_embedding(fmt, table, dids, D, dtype=torch.bfloat16).cpu()
    wantb = torch.from_numpy(want).to(torch.bfloat16)
    assert torch.equal(gotb.view(torch.int16), wantb.view(torch.int16))
    assert q.qmm_device_error_take() == 0


def test_embedding_bad_id_writes_zeros_and_reports():
    V, D = 20, 512
    packed = oracle.quantize(q.QMM_Q8_0, inputs.bf16_bits(inputs.weights(V, D, 70)))
    ids = torch.tensor([1, V, -3, 2], dtype=torch.int64, device=DEV)
    out = q.qmm_embedding(q.QMM_Q8_0, to_dev_u8(packed), ids, D)
    assert q.qmm_device_error_take() == q.QMM_DEVERR_EMBEDDING_ID
    o = out.cpu().numpy()
    assert not o[1].any() and not o[2].any()
    full = oracle.dequantize(q.QMM_Q8_0, packed, V, D)
    assert np.array_equal(o[0], full[1]) and np.array_equal(o[3], full[2])
    assert q.qmm_device_error_take() == 0
