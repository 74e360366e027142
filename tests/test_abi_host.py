"""Host-only checks of the C ABI (no kernel is launched): the library builds
and loads, exports every function include/qmm.h declares, and rejects bad
arguments with the documented status before touching the GPU."""
import ctypes
import os
import re

import pytest

import ggml_block_quantized_linear_b300 as q
from ggml_block_quantized_linear_b300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return q.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "qmm.h")).read()
    return re.findall(r"QMM_API\s+[\w\s\*]+?\b(qmm_\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = set(declared_functions())
    assert {"qmm_quantize", "qmm_dequantize", "qmm_matmul", "qmm_packed_bytes",
            "qmm_matmul_workspace_bytes", "qmm_status_string"} <= names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert q.qmm_version().startswith("qmm ")


def test_packed_bytes(lib):
    assert q.qmm_packed_bytes(q.QMM_Q8_0, 4096, 4096) == 17825792
    assert q.qmm_packed_bytes(q.QMM_Q4_K, 4096, 4096) == 9437184
    assert q.qmm_packed_bytes(q.QMM_Q8_0, 14336, 4096) == 62390272
    assert q.qmm_packed_bytes(q.QMM_Q4_K, 14336, 4096) == 33030144
    assert q.qmm_packed_bytes(q.QMM_Q8_0, 1, 48) == 0       # not a block multiple
    assert q.qmm_packed_bytes(q.QMM_Q4_K, 1, 512 + 32) == 0
    assert q.qmm_packed_bytes(7, 1, 256) == 0
    assert q.qmm_packed_bytes(q.QMM_Q8_0, -1, 256) == 0
    assert q.qmm_packed_bytes(q.QMM_Q8_0, 0, 256) == 0


def test_status_strings(lib):
    for s in range(-7, 1):
        assert len(q.qmm_status_string(s)) > 0
    assert q.qmm_status_string(99) == "unknown status"


FAKE = ctypes.c_void_p(0x1000)        # never dereferenced: every case fails first
MISALIGNED = ctypes.c_void_p(0x1008)
NULL = ctypes.c_void_p(0)
S0 = ctypes.c_void_p(0)


def test_quantize_argument_errors(lib):
    L = lib
    assert L.qmm_quantize(7, 0, FAKE, FAKE, 4, 256, S0) == q.QMM_ERR_INVALID_ARG
    assert L.qmm_quantize(8, 3, FAKE, FAKE, 4, 256, S0) == q.QMM_ERR_INVALID_ARG
    assert L.qmm_quantize(8, 0, FAKE, FAKE, -1, 256, S0) == q.QMM_ERR_INVALID_ARG
    assert L.qmm_quantize(8, 0, FAKE, FAKE, 4, 0, S0) == q.QMM_ERR_SHAPE
    assert L.qmm_quantize(8, 0, FAKE, FAKE, 4, 288, S0) == q.QMM_ERR_SHAPE
    assert L.qmm_quantize(4, 0, FAKE, FAKE, 4, 128, S0) == q.QMM_ERR_SHAPE
    assert L.qmm_quantize(8, 0, NULL, FAKE, 4, 256, S0) == q.QMM_ERR_INVALID_ARG
    assert L.qmm_quantize(8, 0, FAKE, NULL, 4, 256, S0) == q.QMM_ERR_INVALID_ARG
    assert L.qmm_quantize(4, 1, MISALIGNED, FAKE, 4, 256, S0) == q.QMM_ERR_ALIGNMENT
    assert L.qmm_quantize(4, 1, FAKE, MISALIGNED, 4, 256, S0) == q.QMM_ERR_ALIGNMENT
    assert L.qmm_quantize(8, 0, NULL, NULL, 0, 256, S0) == q.QMM_OK  # empty: nothing to do


def test_dequantize_argument_errors(lib):
    L = lib
    assert L.qmm_dequantize(7, FAKE, FAKE, 4, 256, S0) == q.QMM_ERR_INVALID_ARG
    assert L.qmm_dequantize(8, FAKE, FAKE, 4, 100, S0) == q.QMM_ERR_SHAPE
    assert L.qmm_dequantize(8, NULL, FAKE, 4, 256, S0) == q.QMM_ERR_INVALID_ARG
    assert L.qmm_dequantize(4, FAKE, MISALIGNED, 4, 256, S0) == q.QMM_ERR_ALIGNMENT
    assert L.qmm_dequantize(4, NULL, NULL, 0, 256, S0) == q.QMM_OK


def test_matmul_argument_errors(lib):
    L = lib
    assert L.qmm_matmul(1, FAKE, FAKE, FAKE, 1, 64, 256, NULL, 0, S0) == q.QMM_ERR_INVALID_ARG
    assert L.qmm_matmul(8, FAKE, FAKE, FAKE, -1, 64, 256, NULL, 0, S0) == q.QMM_ERR_INVALID_ARG
    assert L.qmm_matmul(8, FAKE, FAKE, FAKE, 1, 64, 200, NULL, 0, S0) == q.QMM_ERR_SHAPE
    assert L.qmm_matmul(4, FAKE, FAKE, FAKE, 1, 64, 0, NULL, 0, S0) == q.QMM_ERR_SHAPE
    assert L.qmm_matmul(8, NULL, FAKE, FAKE, 1, 64, 256, NULL, 0, S0) == q.QMM_ERR_INVALID_ARG
    assert L.qmm_matmul(8, FAKE, NULL, FAKE, 1, 64, 256, NULL, 0, S0) == q.QMM_ERR_INVALID_ARG
    assert L.qmm_matmul(8, FAKE, FAKE, NULL, 1, 64, 256, NULL, 0, S0) == q.QMM_ERR_INVALID_ARG
    assert L.qmm_matmul(8, MISALIGNED, FAKE, FAKE, 1, 64, 256, NULL, 0, S0) == q.QMM_ERR_ALIGNMENT
    assert L.qmm_matmul(8, FAKE, MISALIGNED, FAKE, 1, 64, 256, NULL, 0, S0) == q.QMM_ERR_ALIGNMENT
    assert L.qmm_matmul(8, FAKE, FAKE, MISALIGNED, 1, 64, 256, NULL, 0, S0) == q.QMM_ERR_ALIGNMENT
    assert L.qmm_matmul(8, NULL, NULL, NULL, 0, 64, 256, NULL, 0, S0) == q.QMM_OK
    assert L.qmm_matmul(8, NULL, NULL, NULL, 3, 0, 256, NULL, 0, S0) == q.QMM_OK


def test_workspace_query(lib):
    for fmt in (q.QMM_Q8_0, q.QMM_Q4_K):
        for M in (1, 4, 16):  # decode shapes reduce in distributed shared memory
            assert q.qmm_matmul_workspace_bytes(fmt, M, 4096, 4096) == 0
        assert q.qmm_matmul_workspace_bytes(fmt, 512, 4096, 100) == 0  # invalid K
        # tiled path (148 SMs when no GPU is visible): a binary16 copy of the
        # activations; with a K split of tiles under 256 tokens, the partial
        # tiles and one ticket per tile follow (256-byte aligned regions)
        # 512 x 4096: 256-token tiles, K halves added onto a zeroed Y
        assert q.qmm_matmul_workspace_bytes(fmt, 512, 4096, 4096) == 512 * 4096 * 2
        # 2048 x 14336: 112 x 8 tiles, stream-K onto a zeroed Y (no partial tiles)
        assert q.qmm_matmul_workspace_bytes(fmt, 2048, 14336, 4096) == 2048 * 4096 * 2
        # 32 tokens: a 32-token tile; 8 weight tiles, K in min(16, 148 // 8, 8) = 8 parts
        assert q.qmm_matmul_workspace_bytes(fmt, 32, 1024, 4096) == 32 * 4096 * 2 + 8 * 8 * 32 * 128 * 4 + 256
    # long rows (K >= 12288) at decode batch sizes: FP8 and Q5_K from 9 tokens,
    # Q8_0 from 12 run the tiled kernel (workspace); Q4_K and shorter rows do not
    F8 = q.QMM_FP8_E4M3
    assert q.qmm_matmul_workspace_bytes(F8, 8, 4096, 14336) == 0
    assert q.qmm_matmul_workspace_bytes(F8, 9, 4096, 14336) > 9 * 14336 * 2
    assert q.qmm_matmul_workspace_bytes(q.QMM_Q5_K, 9, 4096, 12288) > 0
    assert q.qmm_matmul_workspace_bytes(q.QMM_Q8_0, 11, 4096, 14336) == 0
    assert q.qmm_matmul_workspace_bytes(q.QMM_Q8_0, 12, 4096, 14336) > 0
    assert q.qmm_matmul_workspace_bytes(q.QMM_Q4_K, 16, 4096, 14336) == 0
    assert q.qmm_matmul_workspace_bytes(F8, 16, 4096, 11264) == 0
    L = lib
    assert L.qmm_matmul(8, FAKE, FAKE, FAKE, 32, 64, 256, NULL, 0, S0) == q.QMM_ERR_WORKSPACE
    assert L.qmm_matmul(4, FAKE, FAKE, FAKE, 32, 64, 256, FAKE, 100, S0) == q.QMM_ERR_WORKSPACE
    assert L.qmm_matmul(4, FAKE, FAKE, FAKE, 32, 64, 256, MISALIGNED, 1 << 20, S0) == q.QMM_ERR_ALIGNMENT


def test_q6_k_sizes_and_policy(lib):
    import json
    assert q.qmm_packed_bytes(q.QMM_Q6_K, 4096, 4096) == 4096 * 16 * 210
    assert q.qmm_packed_bytes(q.QMM_Q6_K, 3, 768) == 3 * 3 * 210
    assert q.qmm_packed_bytes(q.QMM_Q6_K, 1, 256 + 32) == 0
    assert q.qmm_matmul_workspace_bytes(q.QMM_Q6_K, 512, 4096, 4096) == 0
    # the pages' sensitive-tensor table, read from the golden file
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "paper_widths.json")))
    names = {"Q2K": q.QMM_Q2_K, "Q3K": q.QMM_Q3_K, "Q4K": q.QMM_Q4_K, "Q5K": q.QMM_Q5_K, "Q6K": q.QMM_Q6_K,
             "Q8_0": q.QMM_Q8_0}
    for model, emb in g["sensitive_tensor_type"].items():
        assert q.qmm_embedding_format(names[model]) == names[emb]
    assert q.qmm_embedding_format(7) == 0
    assert q.qmm_embedding_format(q.QMM_FP8_E4M3) == 0


def test_k_quant_sizes(lib):
    # Q5_K 176, Q3_K 110, Q2_K 84 bytes per 256 weights.  Q5_K prefill runs the
    # tiled kernel (the binary16 copy of X as workspace, the static entry
    # serves it); Q3_K / Q2_K need no workspace and the static entry leaves
    # them to qmm_matmul
    L = lib
    for fmt, nb in ((q.QMM_Q5_K, 176), (q.QMM_Q3_K, 110), (q.QMM_Q2_K, 84)):
        assert q.qmm_packed_bytes(fmt, 4096, 4096) == 4096 * 16 * nb
        assert q.qmm_packed_bytes(fmt, 3, 768) == 3 * 3 * nb
        assert q.qmm_packed_bytes(fmt, 1, 256 + 32) == 0
        assert q.qmm_matmul_workspace_bytes(fmt, 16, 4096, 4096) == 0
        assert L.qmm_quantize(fmt, 0, FAKE, FAKE, 4, 200, S0) == q.QMM_ERR_SHAPE
        assert L.qmm_quantize(fmt, 0, MISALIGNED, FAKE, 4, 256, S0) == q.QMM_ERR_ALIGNMENT
        assert L.qmm_dequantize(fmt, NULL, FAKE, 4, 256, S0) == q.QMM_ERR_INVALID_ARG
        assert L.qmm_matmul(fmt, FAKE, FAKE, NULL, 1, 64, 256, NULL, 0, S0) == q.QMM_ERR_INVALID_ARG
    assert q.qmm_matmul_workspace_bytes(q.QMM_Q5_K, 512, 4096, 4096) == 512 * 4096 * 2
    assert L.qmm_matmul(q.QMM_Q5_K, FAKE, FAKE, FAKE, 32, 64, 256, NULL, 0, S0) == q.QMM_ERR_WORKSPACE
    assert L.qmm_matmul_prefill_static(q.QMM_Q5_K, NULL, FAKE, FAKE, 512, 64, 256, S0) == q.QMM_ERR_INVALID_ARG
    for fmt in (q.QMM_Q3_K, q.QMM_Q2_K):
        assert q.qmm_matmul_workspace_bytes(fmt, 512, 4096, 4096) == 0
        assert L.qmm_matmul_prefill_static(fmt, FAKE, FAKE, FAKE, 512, 64, 256, S0) == q.QMM_ERR_UNSUPPORTED


def test_fp8_sizes(lib):
    assert q.qmm_packed_bytes(q.QMM_FP8_E4M3, 4096, 4096) == 4096 * (4096 + 16)
    assert q.qmm_packed_bytes(q.QMM_FP8_E4M3, 3, 256) == 3 * 272
    assert q.qmm_packed_bytes(q.QMM_FP8_E4M3, 1, 288) == 0
    assert q.qmm_matmul_workspace_bytes(q.QMM_FP8_E4M3, 512, 4096, 4096) == 512 * 4096 * 2


def test_embedding_argument_errors(lib):
    L = lib
    ids8 = ctypes.c_void_p(0x1000)
    ids_mis = ctypes.c_void_p(0x1004)
    assert L.qmm_embedding(7, FAKE, ids8, 4, 10, 256, FAKE, 0, S0) == q.QMM_ERR_INVALID_ARG
    assert L.qmm_embedding(8, FAKE, ids8, 4, 10, 256, FAKE, 2, S0) == q.QMM_ERR_INVALID_ARG
    assert L.qmm_embedding(8, FAKE, ids8, -1, 10, 256, FAKE, 0, S0) == q.QMM_ERR_INVALID_ARG
    assert L.qmm_embedding(8, FAKE, ids8, 4, 10, 300, FAKE, 0, S0) == q.QMM_ERR_SHAPE
    assert L.qmm_embedding(6, FAKE, ids8, 4, 0, 256, FAKE, 0, S0) == q.QMM_ERR_INVALID_ARG
    assert L.qmm_embedding(6, NULL, ids8, 4, 10, 256, FAKE, 0, S0) == q.QMM_ERR_INVALID_ARG
    assert L.qmm_embedding(4, FAKE, ids_mis, 4, 10, 256, FAKE, 1, S0) == q.QMM_ERR_ALIGNMENT
    assert L.qmm_embedding(4, MISALIGNED, ids8, 4, 10, 256, FAKE, 1, S0) == q.QMM_ERR_ALIGNMENT
    assert L.qmm_embedding(4, NULL, NULL, 0, 10, 256, NULL, 1, S0) == q.QMM_OK  # no tokens


def test_selftest_limit_checked_on_the_host(lib):
    for bad in (0, -5, 100000001):
        assert lib.qmm_selftest_bounded_wait(bad, S0) == q.QMM_ERR_INVALID_ARG


def test_static_prefill_argument_errors(lib):
    f = lib.qmm_matmul_prefill_static
    # M * K * 2 bytes of scratch beyond the fixed 64 MiB array
    assert f(8, FAKE, FAKE, FAKE, 4096, 64, 16384 + 256, S0) == q.QMM_ERR_WORKSPACE
    assert f(8, FAKE, FAKE, FAKE, 16, 64, 256, S0) == q.QMM_ERR_UNSUPPORTED
    assert f(4, FAKE, FAKE, FAKE, 32, 64, 300, S0) == q.QMM_ERR_SHAPE
    assert f(4, NULL, FAKE, FAKE, 32, 64, 256, S0) == q.QMM_ERR_INVALID_ARG
    assert f(4, FAKE, MISALIGNED, FAKE, 32, 64, 256, S0) == q.QMM_ERR_ALIGNMENT
    assert f(6, FAKE, FAKE, FAKE, 32, 64, 256, S0) == q.QMM_ERR_UNSUPPORTED  # Q6_K needs no scratch


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError):
        q.load(str(tmp_path / "nope.so"))
