"""Pins for the oracle's matmul Y = X W^T over exactly dequantized weights.

Checks: exact rational arithmetic (Python fractions) on tiny shapes, one-hot
activation rows that must return single dequantized weights exactly (which
also catches a transposed operand), zero weights, linearity, the column
sampler against the full product, and the tolerance scale A = sum |w x|.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from ggml_block_quantized_linear_b300 import inputs


def make(fmt, n, k, m, seed):
    w = inputs.weights(n, k, seed)
    x = inputs.activations(m, k, seed)
    packed = oracle.quantize(fmt, inputs.bf16_bits(w))
    return packed, inputs.bf16_bits(x), x.float().numpy()


@pytest.mark.parametrize("fmt,k", [(oracle.Q8_0, 64), (oracle.Q4_K, 256), (oracle.Q6_K, 256), (oracle.FP8, 256), (oracle.Q5_K, 256), (oracle.Q3_K, 256), (oracle.Q2_K, 256)])
def test_exact_rational_tiny(fmt, k):
    n, m = 5, 3
    packed, xb, xf = make(fmt, n, k, m, 31)
    wd = oracle.dequantize(fmt, packed, n, k)
    Y, A = oracle.matmul(fmt, packed, xb, n, k)
    for i in range(m):
        for j in range(n):
            exact = sum(Fraction(float(wd[j, t])) * Fraction(float(xf[i, t])) for t in range(k))
            absum = sum(abs(Fraction(float(wd[j, t])) * Fraction(float(xf[i, t]))) for t in range(k))
            assert abs(Fraction(Y[i, j]) - exact) <= Fraction(k) * Fraction(2.0 ** -52) * absum
            assert abs(Fraction(A[i, j]) - absum) <= Fraction(k) * Fraction(2.0 ** -52) * absum


@pytest.mark.parametrize("fmt", [oracle.Q8_0, oracle.Q4_K, oracle.Q6_K, oracle.FP8, oracle.Q5_K, oracle.Q3_K, oracle.Q2_K])
def test_one_hot_rows_select_weights(fmt):
    n, k = 6, 512
    packed, _, _ = make(fmt, n, k, 1, 32)
    wd = oracle.dequantize(fmt, packed, n, k)
    cols = [0, 1, 37, 255, 256, 511]
    x = torch.zeros((len(cols), k), dtype=torch.bfloat16)
    for i, c in enumerate(cols):
        x[i, c] = 1.0
    Y, _ = oracle.matmul(fmt, packed, inputs.bf16_bits(x), n, k)
    assert np.array_equal(Y, wd[:, cols].T.astype(np.float64))


@pytest.mark.parametrize("fmt", [oracle.Q8_0, oracle.Q4_K, oracle.Q6_K, oracle.FP8, oracle.Q5_K, oracle.Q3_K, oracle.Q2_K])
def test_zero_weights(fmt):
    n, k = 4, 256
    packed = oracle.quantize(fmt, np.zeros((n, k), dtype=np.float32))
    xb = inputs.bf16_bits(inputs.activations(2, k, 1))
    Y, A = oracle.matmul(fmt, packed, xb, n, k)
    assert not Y.any() and not A.any()


@pytest.mark.parametrize("fmt", [oracle.Q8_0, oracle.Q4_K, oracle.Q6_K, oracle.FP8, oracle.Q5_K, oracle.Q3_K, oracle.Q2_K])
def test_linearity(fmt):
    n, k = 8, 512
    packed, _, _ = make(fmt, n, k, 1, 33)
    rng = np.random.default_rng(5)
    # small integers: X1, X2 and X1 + X2 are exact in bf16
    x1 = torch.from_numpy(rng.integers(-8, 9, (3, k)).astype(np.float32)).to(torch.bfloat16)
    x2 = torch.from_numpy(rng.integers(-8, 9, (3, k)).astype(np.float32)).to(torch.bfloat16)
    Y1, A1 = oracle.matmul(fmt, packed, inputs.bf16_bits(x1), n, k)
    Y2, A2 = oracle.matmul(fmt, packed, inputs.bf16_bits(x2), n, k)
    Y12, _ = oracle.matmul(fmt, packed, inputs.bf16_bits(x1 + x2), n, k)
    assert np.all(np.abs(Y12 - (Y1 + Y2)) <= 4 * k * 2.0 ** -52 * (A1 + A2))
    # the sum really changes the output (guards against a dropped operand)
    assert np.abs(Y1).max() > 0 and np.abs(Y12 - Y1).max() > 0


@pytest.mark.parametrize("fmt", [oracle.Q8_0, oracle.Q4_K, oracle.Q6_K, oracle.FP8, oracle.Q5_K, oracle.Q3_K, oracle.Q2_K])
def test_columns_match_full_product(fmt):
    n, k, m = 40, 512, 3
    packed, xb, _ = make(fmt, n, k, m, 34)
    Y, A = oracle.matmul(fmt, packed, xb, n, k)
    ns = [39, 0, 17, 17, 5]
    Yc, Ac = oracle.matmul_columns(fmt, packed, xb, k, ns)
    assert np.array_equal(Yc, Y[:, ns]) and np.array_equal(Ac, A[:, ns])
    assert np.all(A >= np.abs(Y))


def test_thread_count_does_not_change_results():
    n, k, m = 64, 1024, 2
    packed, xb, _ = make(oracle.Q4_K, n, k, m, 35)
    oracle.set_threads(1)
    Y1, _ = oracle.matmul(oracle.Q4_K, packed, xb, n, k)
    oracle.set_threads(4)
    Y4, _ = oracle.matmul(oracle.Q4_K, packed, xb, n, k)
    oracle.set_threads(oracle.max_threads())
    assert np.array_equal(Y1, Y4)
