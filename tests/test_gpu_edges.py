"""GPU accuracy at the edges of binary16, in both matmul paths.

Both paths round each activation to binary16 once; the prefill path (M > 16)
also rounds each dequantized weight to binary16 once.  In binary16's normal
range that is a relative error of at most 2^-11, inside the per-element bound
1e-3 * sum|w^ x| + 1e-6.  Below 2^-14 the error is absolute, at most 2^-25,
and include/qmm.h states the bound with that term added:

    |y - y_exact| <= 1e-3 * sum|w^ x| + 1e-6 + 2^-25 * T,
    T = sum |x_k| over weights |w^_k| < 2^-14 (prefill only)
      + sum |w^_k| over activations |x_k| < 2^-14 (both paths).

These tests check the plain bound on large and small activations in range,
on weights just inside the normal range, and the stated bound on weights and
activations below it.
"""
import numpy as np
import pytest
import torch

import oracle
import ggml_block_quantized_linear_b300 as q
from ggml_block_quantized_linear_b300 import inputs
from qmm_testutil import bf16_from_bits, check_matmul, to_dev_u8

pytestmark = pytest.mark.gpu
FMTS = [q.QMM_Q8_0, q.QMM_Q4_K]
TINY = 2.0 ** -14


def bits_of(x32):
    return inputs.bf16_bits(torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(torch.bfloat16))


def extra_term(w_hat, xb, prefill):
    """2^-25 * T of the stated bound, [M x N] (w_hat fp32 [N x K], xb bf16 bits)."""
    x = (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    w = np.abs(w_hat.astype(np.float64))
    ax = np.abs(x)
    # zeros are exact in binary16 and add nothing
    t = ((ax < TINY) & (ax > 0)).astype(np.float64) @ w.T
    if prefill:
        t += ax @ ((w < TINY) & (w > 0)).astype(np.float64).T
    return 2.0 ** -25 * t


def check_stated(y_gpu, Y, A, E, what):
    y = y_gpu.detach().cpu().double().numpy()
    err = np.abs(y - Y)
    bound = 1e-3 * A + 1e-6 + E
    bad = err > bound
    assert not bad.any(), "%s: %d outside the stated bound; worst ratio %g" % (
        what, int(bad.sum()), float((err / bound).max()))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("m", [3, 300])
def test_activation_range_both_paths(fmt, m):
    n, k = 192, 1024
    w = inputs.weights(n, k, 21)
    packed = oracle.quantize(fmt, inputs.bf16_bits(w))
    rng = np.random.default_rng(5)
    x = rng.normal(0, 1, (m, k)).astype(np.float32)
    x[0::3] *= 3000.0        # large, inside binary16's range
    x[1::3] *= 1e-3          # small, still normal in binary16 (|x| >= 2^-14 mostly)
    x[2::3, ::3] = 0.0
    xb = bits_of(x)
    Y, A = oracle.matmul(fmt, packed, xb, n, k)
    y = q.qmm_matmul(fmt, to_dev_u8(packed), bf16_from_bits(xb), n)
    E = extra_term(oracle.dequantize(fmt, packed, n, k), xb, m > 16)
    check_stated(y, Y, A, E, "range m=%d" % m)
    # outputs that meet no value below 2^-14 (T = 0) meet the plain bound
    sel = E == 0
    err = np.abs(y.cpu().double().numpy() - Y)
    assert np.all(err[sel] <= 1e-3 * A[sel] + 1e-6)


def sparse_large_x(m, k, seed, magnitude=100.0, per_row=3):
    rng = np.random.default_rng(seed)
    x = np.zeros((m, k), dtype=np.float32)
    for r in range(m):
        cols = rng.choice(k, size=per_row, replace=False)
        x[r, cols] = magnitude * rng.choice([-1.0, 1.0], size=per_row)
    return x


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("m", [3, 40])
def test_weights_just_inside_binary16_normal_range(fmt, m):
    # weights ~ N(0, 1) * 2^-9: dequantized values mostly between 2^-14 and
    # 2^-6, so the prefill's binary16 weights keep their relative precision;
    # sparse activations of magnitude 100 then see single weights
    n, k = 256, 1024
    rng = np.random.default_rng(31)
    w = (rng.normal(0, 1, (n, k)) * 2.0 ** -9).astype(np.float32)
    packed = oracle.quantize(fmt, w)
    w_hat = oracle.dequantize(fmt, packed, n, k)
    xb = bits_of(sparse_large_x(m, k, 32))
    Y, A = oracle.matmul(fmt, packed, xb, n, k)
    y = q.qmm_matmul(fmt, to_dev_u8(packed), bf16_from_bits(xb), n)
    E = extra_term(w_hat, xb, m > 16)
    check_stated(y, Y, A, E, "normal-range weights")
    # where every weight the activations meet is normal (or zero), T = 0 and
    # the plain bound holds
    x = (xb.astype(np.uint32) << 16).view(np.float32)
    met = (np.abs(x) > 0).astype(np.float64) @ ((np.abs(w_hat) < TINY) & (w_hat != 0)).astype(np.float64).T
    yy = y.cpu().double().numpy()
    sel = met == 0
    assert sel.mean() > 0.5
    err = np.abs(yy - Y)
    assert np.all(err[sel] <= 1e-3 * A[sel] + 1e-6)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("m", [3, 40])
def test_tiny_weights_sparse_large_activations(fmt, m):
    # weights of scale ~1e-5 (below 2^-14 = 6.1e-5): in the prefill path each
    # rounds to a binary16 subnormal (absolute error <= 2^-25); the decode
    # path multiplies exact codes and keeps the plain bound
    n, k = 256, 1024
    rng = np.random.default_rng(41)
    w = (rng.normal(0, 1e-5, (n, k))).astype(np.float32)
    packed = oracle.quantize(fmt, w)
    w_hat = oracle.dequantize(fmt, packed, n, k)
    xb = bits_of(sparse_large_x(m, k, 42))
    Y, A = oracle.matmul(fmt, packed, xb, n, k)
    y = q.qmm_matmul(fmt, to_dev_u8(packed), bf16_from_bits(xb), n)
    if m <= 16:
        check_matmul(y, Y, A, "tiny weights, decode")
    else:
        check_stated(y, Y, A, extra_term(w_hat, xb, True), "tiny weights, prefill")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("m", [1, 8, 16, 17, 300])
def test_tiny_activations_both_paths(fmt, m):
    # correlated activations of magnitude ~1e-5 (binary16 subnormals)
    n, k = 200, 2048
    w = inputs.weights(n, k, 51)
    packed = oracle.quantize(fmt, inputs.bf16_bits(w))
    rng = np.random.default_rng(52)
    base = rng.normal(0, 1, k)
    x = ((base[None, :] + 0.1 * rng.normal(0, 1, (m, k))) * 1e-5).astype(np.float32)
    xb = bits_of(x)
    Y, A = oracle.matmul(fmt, packed, xb, n, k)
    y = q.qmm_matmul(fmt, to_dev_u8(packed), bf16_from_bits(xb), n)
    E = extra_term(oracle.dequantize(fmt, packed, n, k), xb, m > 16)
    check_stated(y, Y, A, E, "tiny activations m=%d" % m)
