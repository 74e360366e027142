"""qmm_matmul_prefill_static: the prefill matmul that allocates nothing.

Some callers cannot allocate device memory (a plugin handed raw pointers by
a host framework, an engine whose pool owns all device memory, a loop that
must not call cudaMalloc since it can synchronise the device).  This entry
point keeps its scratch in a fixed device array inside the library.  The test
calls it through the C ABI and checks it against the allocating entry point
(qmm_matmul with a torch-allocated workspace) within the tolerance of the
other matmul tests, on two calls in a row, then checks its size limits.
It sits in a file of its own that pytest collects last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import ggml_block_quantized_linear_b300 as q
from ggml_block_quantized_linear_b300 import inputs
from qmm_testutil import DEV, bf16_from_bits, check_matmul, to_dev_u8

pytestmark = pytest.mark.gpu


def static_fn():
    L = q.load()
    f = L.qmm_matmul_prefill_static
    f.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                  ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f


def call_static(fmt, w, x, y, m, n, k):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return static_fn()(fmt, w.data_ptr(), x.data_ptr(), y.data_ptr(), m, n, k, stream)


@pytest.mark.parametrize("fmt", [q.QMM_Q8_0, q.QMM_Q4_K])
def test_static_scratch_matches_allocating_entry_point(fmt):
    for (n, k, m, seed) in [(384, 1024, 300, 1), (256, 2304, 64, 2)]:
        w = inputs.weights(n, k, seed)
        xt = inputs.activations(m, k, seed)
        packed = oracle.quantize(fmt, inputs.bf16_bits(w))
        xb = inputs.bf16_bits(xt)
        Y, A = oracle.matmul(fmt, packed, xb, n, k)
        wd, xd = to_dev_u8(packed), bf16_from_bits(xb)
        ref = q.qmm_matmul(fmt, wd, xd, n)  # allocating entry point
        torch.cuda.synchronize()
        for _ in range(2):  # two calls in a row share the static scratch
            y = torch.full((m, n), float("nan"), dtype=torch.float32, device=DEV)
            assert call_static(fmt, wd, xd, y, m, n, k) == q.QMM_OK
            torch.cuda.synchronize()
            check_matmul(y, Y, A, "static scratch vs oracle")
            bound = 1e-3 * A + 1e-6
            diff = np.abs(y.cpu().double().numpy() - ref.cpu().double().numpy())
            assert np.all(diff <= bound)
    assert q.qmm_device_error_take() == 0


def test_static_scratch_limits():
    fn = static_fn()
    dummy = torch.empty(16, dtype=torch.uint8, device=DEV)
    p = dummy.data_ptr()
    s0 = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # M * K * 2 bytes beyond the 64 MiB array: rejected before any launch
    assert fn(q.QMM_Q8_0, p, p, p, 4096, 64, 16384 + 256, s0) == q.QMM_ERR_WORKSPACE
    # decode sizes need no scratch and are left to qmm_matmul
    assert fn(q.QMM_Q8_0, p, p, p, 16, 64, 256, s0) == q.QMM_ERR_UNSUPPORTED
    assert fn(q.QMM_Q4_K, p, p, p, 32, 64, 300, s0) == q.QMM_ERR_SHAPE
    assert fn(q.QMM_Q4_K, 0, p, p, 32, 64, 256, s0) == q.QMM_ERR_INVALID_ARG
