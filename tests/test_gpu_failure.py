"""The failure path of the kernels' bounded waits, exercised on the GPU
without a fault: the library's self-test kernel waits on an mbarrier that
nothing ever arrives on, gives up after a few microseconds, records its code
in the device error word and returns.  The host reads the code, the context
stays usable, and a normal call afterwards is correct and records nothing."""
import numpy as np
import pytest

import oracle
import ggml_block_quantized_linear_b300 as q
from ggml_block_quantized_linear_b300 import inputs
from qmm_testutil import bf16_from_bits, check_matmul, to_dev_u8

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_cleared():
    assert q.qmm_device_error_take() == 0
    q.qmm_selftest_bounded_wait(20000)          # 20 us limit
    assert q.qmm_device_error_take() == q.QMM_DEVERR_SELFTEST_TIMEOUT
    assert q.qmm_device_error_take() == 0       # taking the code clears it
    # the first code recorded is kept until taken
    q.qmm_selftest_bounded_wait(5000)
    q.qmm_selftest_bounded_wait(5000)
    assert q.qmm_device_error_take() == q.QMM_DEVERR_SELFTEST_TIMEOUT
    # a normal call afterwards
    n, k = 256, 1024
    for fmt in (q.QMM_Q8_0, q.QMM_Q4_K):
        packed = oracle.quantize(fmt, inputs.bf16_bits(inputs.weights(n, k, 61)))
        for m in (1, 40):
            xb = inputs.bf16_bits(inputs.activations(m, k, 62))
            Y, A = oracle.matmul(fmt, packed, xb, n, k)
            check_matmul(q.qmm_matmul(fmt, to_dev_u8(packed), bf16_from_bits(xb), n), Y, A)
    assert q.qmm_device_error_take() == 0


def test_selftest_rejects_limits_out_of_range():
    for bad in (0, -1, 100000001):
        with pytest.raises(q.QmmError) as e:
            q.qmm_selftest_bounded_wait(bad)
        assert e.value.status == q.QMM_ERR_INVALID_ARG
    assert q.qmm_device_error_take() == 0
