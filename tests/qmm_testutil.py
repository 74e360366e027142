"""Shared helpers of the GPU parity tests: device uploads and the matmul
tolerance check.  Expected values always come from the CPU oracle."""
import numpy as np
import torch

import oracle
import ggml_block_quantized_linear_b300 as q

DEV = "cuda:0"
FMT_NAMES = {q.QMM_Q8_0: "q8_0", q.QMM_Q4_K: "q4_k"}


def to_dev_u8(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def bf16_from_bits(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(DEV)


def check_matmul(y_gpu: torch.Tensor, Y: np.ndarray, A: np.ndarray, what: str = ""):
    """Per element: |y - y_ref| <= 1e-3 * sum|w x| + 1e-6 (y_ref, sum in fp64)."""
    y = y_gpu.detach().cpu().double().numpy()
    assert y.shape == Y.shape, (y.shape, Y.shape)
    assert np.isfinite(y).all(), what
    err = np.abs(y - Y)
    bound = 1e-3 * A + 1e-6
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err / bound), err.shape)
        raise AssertionError("%s: %d / %d outside tolerance; worst at %s: y=%r ref=%r err=%g bound=%g"
                             % (what, int(bad.sum()), bad.size, i, y[i], Y[i], err[i], bound[i]))
    return float((err / bound).max())
