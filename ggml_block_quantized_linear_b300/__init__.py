"""B300-native GGML block-quantized linear layers (Q8_0, Q4_K).

A thin ctypes binding over ``libqmm.so`` (``include/qmm.h``).  The functions
keep the C names and only marshal arguments: torch tensors supply device
memory and the current CUDA stream; every step of the computation runs in the
library's sm_103a kernels.  There is no fallback: if ``libqmm.so`` is missing
or a call fails, an exception is raised.

    packed = qmm_quantize(QMM_Q4_K, w_bf16)            # ISQ, uint8 [N, K/256*144]
    w_hat  = qmm_dequantize(QMM_Q4_K, packed, N, K)    # fp32 [N, K]
    y      = qmm_matmul(QMM_Q4_K, packed, x_bf16, N)   # fp32 [M, N]
"""
from __future__ import annotations

import ctypes
import os
import threading

QMM_Q8_0 = 8
QMM_Q4_K = 4
QMM_Q6_K = 6
QMM_Q5_K = 5
QMM_Q3_K = 3
QMM_Q2_K = 2
QMM_FP8_E4M3 = 80
QMM_OUT_F32 = 0
QMM_OUT_BF16 = 1
QMM_SRC_BF16 = 0
QMM_SRC_F32 = 1

QMM_OK = 0
QMM_ERR_INVALID_ARG = -1
QMM_ERR_UNSUPPORTED = -2
QMM_ERR_SHAPE = -3
QMM_ERR_ALIGNMENT = -4
QMM_ERR_WORKSPACE = -5
QMM_ERR_CUDA = -6
QMM_ERR_DEVICE = -7

FORMATS = {"q8_0": QMM_Q8_0, "q4_k": QMM_Q4_K, "q6_k": QMM_Q6_K, "q5_k": QMM_Q5_K, "q3_k": QMM_Q3_K,
           "q2_k": QMM_Q2_K, "fp8": QMM_FP8_E4M3}
BLOCK = {QMM_Q8_0: (32, 34), QMM_Q4_K: (256, 144), QMM_Q6_K: (256, 210), QMM_Q5_K: (256, 176),
         QMM_Q3_K: (256, 110), QMM_Q2_K: (256, 84)}

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqmm.so")
_lib = None
_lock = threading.Lock()


class QmmError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__("%s failed: %s (%d)" % (fn, qmm_status_string(status), status))


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libqmm.so (build it first with ``python -m
    ggml_block_quantized_linear_b300.build``).  Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError("libqmm.so not found at %s: build it with "
                               "`python -m ggml_block_quantized_linear_b300.build`" % p)
        L = ctypes.CDLL(p)
        i64, vp, sz = ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
        L.qmm_packed_bytes.argtypes = [ctypes.c_int, i64, i64]
        L.qmm_packed_bytes.restype = sz
        L.qmm_quantize.argtypes = [ctypes.c_int, ctypes.c_int, vp, vp, i64, i64, vp]
        L.qmm_quantize.restype = ctypes.c_int
        L.qmm_dequantize.argtypes = [ctypes.c_int, vp, vp, i64, i64, vp]
        L.qmm_dequantize.restype = ctypes.c_int
        L.qmm_matmul_workspace_bytes.argtypes = [ctypes.c_int, i64, i64, i64]
        L.qmm_matmul_workspace_bytes.restype = sz
        L.qmm_matmul.argtypes = [ctypes.c_int, vp, vp, vp, i64, i64, i64, vp, sz, vp]
        L.qmm_matmul.restype = ctypes.c_int
        L.qmm_status_string.argtypes = [ctypes.c_int]
        L.qmm_status_string.restype = ctypes.c_char_p
        L.qmm_device_error_take.argtypes = []
        L.qmm_device_error_take.restype = ctypes.c_int
        L.qmm_version.argtypes = []
        L.qmm_version.restype = ctypes.c_char_p
        L.qmm_embedding.argtypes = [ctypes.c_int, vp, vp, i64, i64, i64, vp, ctypes.c_int, vp]
        L.qmm_embedding.restype = ctypes.c_int
        L.qmm_embedding_format.argtypes = [ctypes.c_int]
        L.qmm_embedding_format.restype = ctypes.c_int
        L.qmm_selftest_bounded_wait.argtypes = [i64, vp]
        L.qmm_selftest_bounded_wait.restype = ctypes.c_int
        L.qmm_matmul_prefill_static.argtypes = [ctypes.c_int, vp, vp, vp, i64, i64, i64, vp]
        L.qmm_matmul_prefill_static.restype = ctypes.c_int
        if path is None:
            _lib = L
        return L


def _stream_ptr(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn: str, status: int) -> None:
    if status != QMM_OK:
        raise QmmError(fn, status)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def qmm_status_string(status: int) -> str:
    return load().qmm_status_string(int(status)).decode()


def qmm_version() -> str:
    return load().qmm_version().decode()


def qmm_packed_bytes(fmt: int, rows: int, cols: int) -> int:
    return int(load().qmm_packed_bytes(int(fmt), int(rows), int(cols)))


def qmm_matmul_workspace_bytes(fmt: int, M: int, N: int, K: int) -> int:
    return int(load().qmm_matmul_workspace_bytes(int(fmt), int(M), int(N), int(K)))


def qmm_device_error_take() -> int:
    return int(load().qmm_device_error_take())


QMM_DEVERR_EMBEDDING_ID = 301
QMM_DEVERR_SELFTEST_TIMEOUT = 901


def qmm_embedding_format(model_fmt: int) -> int:
    return int(load().qmm_embedding_format(int(model_fmt)))


def qmm_embedding(fmt: int, table, ids, D: int, out=None, dtype=None, stream=None):
    """Embedding lookup: the dequantized rows ``ids`` (int64 CUDA tensor) of
    the packed table (uint8 [V, row_bytes]) as fp32 (default) or bf16."""
    import torch
    if table.dtype != torch.uint8 or table.dim() != 2 or not table.is_contiguous():
        raise ValueError("qmm_embedding: table must be a contiguous 2-D uint8 tensor")
    if ids.dtype != torch.int64 or not ids.is_contiguous():
        raise ValueError("qmm_embedding: ids must be a contiguous int64 tensor")
    dtype = dtype or (out.dtype if out is not None else torch.float32)
    if dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("qmm_embedding: output must be fp32 or bf16")
    T = ids.numel()
    if out is None:
        out = torch.empty((T, D), dtype=dtype, device=table.device)
    od = QMM_OUT_BF16 if dtype == torch.bfloat16 else QMM_OUT_F32
    _check("qmm_embedding", load().qmm_embedding(int(fmt), _ptr(table), _ptr(ids), T, table.shape[0],
                                                 int(D), _ptr(out), od, _stream_ptr(stream)))
    return out


def qmm_selftest_bounded_wait(limit_ns: int, stream=None) -> None:
    """Launch the bounded-wait self-test kernel (see include/qmm.h)."""
    _check("qmm_selftest_bounded_wait",
           load().qmm_selftest_bounded_wait(int(limit_ns), _stream_ptr(stream)))


def qmm_quantize(fmt: int, src, out=None, stream=None):
    """ISQ of a 2-D bf16 (or fp32) CUDA tensor into a uint8 [rows, row_bytes]
    tensor (``out`` if given)."""
    import torch
    if src.dtype == torch.bfloat16:
        st = QMM_SRC_BF16
    elif src.dtype == torch.float32:
        st = QMM_SRC_F32
    else:
        raise TypeError("qmm_quantize: source must be bf16 or fp32")
    if src.dim() != 2 or not src.is_contiguous():
        raise ValueError("qmm_quantize: source must be a contiguous 2-D tensor")
    rows, cols = src.shape
    nbytes = qmm_packed_bytes(fmt, rows, cols)
    if out is None:
        out = torch.empty((rows, nbytes // rows if rows else 0), dtype=torch.uint8, device=src.device)
    elif out.numel() != nbytes or out.dtype != torch.uint8 or not out.is_contiguous():
        raise ValueError("qmm_quantize: out must be a contiguous uint8 tensor of %d bytes" % nbytes)
    _check("qmm_quantize", load().qmm_quantize(int(fmt), st, _ptr(src), _ptr(out), rows, cols,
                                               _stream_ptr(stream)))
    return out


def qmm_dequantize(fmt: int, packed, rows: int, cols: int, out=None, stream=None):
    import torch
    if packed.dtype != torch.uint8 or not packed.is_contiguous():
        raise ValueError("qmm_dequantize: packed must be a contiguous uint8 tensor")
    if out is None:
        out = torch.empty((rows, cols), dtype=torch.float32, device=packed.device)
    _check("qmm_dequantize", load().qmm_dequantize(int(fmt), _ptr(packed), _ptr(out), int(rows),
                                                   int(cols), _stream_ptr(stream)))
    return out


def qmm_matmul(fmt: int, packed, x, N: int, out=None, workspace=None, stream=None):
    """Y[M, N] (fp32) = X[M, K] (bf16) times the transpose of the packed
    W[N, K].  A workspace of ``qmm_matmul_workspace_bytes`` bytes is
    allocated with torch if the problem needs one and none is given."""
    import torch
    if x.dtype != torch.bfloat16 or x.dim() != 2 or not x.is_contiguous():
        raise ValueError("qmm_matmul: x must be a contiguous 2-D bf16 tensor")
    if packed.dtype != torch.uint8 or not packed.is_contiguous():
        raise ValueError("qmm_matmul: packed must be a contiguous uint8 tensor")
    M, K = x.shape
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    need = qmm_matmul_workspace_bytes(fmt, M, N, K)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("qmm_matmul", load().qmm_matmul(int(fmt), _ptr(packed), _ptr(x), _ptr(out), M, int(N),
                                           K, _ptr(workspace), wbytes, _stream_ptr(stream)))
    return out
