"""CPU oracle for the GGML block-quantized linear layer (Q8_0, Q2_K-Q6_K, FP8).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package. The CUDA library never calls it and shares no code with it.

The arithmetic lives in ``qmm_oracle.c`` (plain C11, no FMA contraction,
fp64 matmul accumulation). This module only compiles it with gcc and
marshals numpy arrays to it with ctypes. The header of ``qmm_oracle.c`` gives
the formulas and the byte layouts, with their sources.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

Q8_0 = 8
Q4_K = 4
Q6_K = 6
Q5_K = 5
Q3_K = 3
Q2_K = 2
FP8 = 80
SRC_BF16 = 0
SRC_F32 = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

BLOCK = {Q8_0: (32, 34), Q4_K: (256, 144), Q6_K: (256, 210), Q5_K: (256, 176), Q3_K: (256, 110),
         Q2_K: (256, 84)}
FP8_ROW_PAD = 16  # FP8 rows: K codes, the fp32 row scale, 12 zero bytes


def build(force: bool = False) -> str:
    """Compile ``qmm_oracle.c`` into ``oracle/_build/liboracle.so``."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fopenmp", "-fPIC", "-shared", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            i64, vp = ctypes.c_int64, ctypes.c_void_p
            L.orc_f32_to_f16.argtypes = [ctypes.c_float]
            L.orc_f32_to_f16.restype = ctypes.c_uint16
            L.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
            L.orc_f16_to_f32.restype = ctypes.c_float
            L.orc_f32_to_f16_array.argtypes = [vp, vp, i64]
            L.orc_f16_to_f32_array.argtypes = [vp, vp, i64]
            L.orc_packed_bytes.argtypes = [ctypes.c_int, i64, i64]
            L.orc_packed_bytes.restype = i64
            L.orc_quantize.argtypes = [ctypes.c_int, ctypes.c_int, vp, vp, i64, i64]
            L.orc_quantize.restype = ctypes.c_int
            L.orc_dequantize.argtypes = [ctypes.c_int, vp, vp, i64, i64]
            L.orc_dequantize.restype = ctypes.c_int
            L.orc_matmul.argtypes = [ctypes.c_int, vp, vp, vp, vp, i64, i64, i64]
            L.orc_matmul.restype = ctypes.c_int
            L.orc_matmul_columns.argtypes = [ctypes.c_int, vp, vp, i64, i64, vp, i64, vp, vp]
            L.orc_matmul_columns.restype = ctypes.c_int
            L.orc_f32_to_e4m3_array.argtypes = [vp, vp, i64]
            L.orc_e4m3_to_f32_array.argtypes = [vp, vp, i64]
            L.orc_gather.argtypes = [ctypes.c_int, vp, i64, i64, vp, i64, vp]
            L.orc_gather.restype = ctypes.c_int
            L.orc_q6_k_position.argtypes = [ctypes.c_int, vp]
            L.orc_q3_k_position.argtypes = [ctypes.c_int, vp]
            L.orc_q3_k_get_field.argtypes = [vp, ctypes.c_int]
            L.orc_q3_k_get_field.restype = ctypes.c_int
            L.orc_q4_k_pack_scales.argtypes = [vp, vp, vp]
            L.orc_q4_k_unpack_scales.argtypes = [vp, vp, vp]
            L.orc_set_threads.argtypes = [ctypes.c_int]
            L.orc_max_threads.restype = ctypes.c_int
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> ctypes.c_void_p:
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


def set_threads(n: int) -> None:
    lib().orc_set_threads(int(n))


def max_threads() -> int:
    return int(lib().orc_max_threads())


def f32_to_f16_bits(values) -> np.ndarray:
    """binary16 encoding (round to nearest, ties to even) of float32 values."""
    v = np.ascontiguousarray(np.asarray(values, dtype=np.float32).ravel())
    out = np.zeros(v.size, dtype=np.uint16)
    lib().orc_f32_to_f16_array(_ptr(v), _ptr(out), v.size)
    return out


def f16_bits_to_f32(bits) -> np.ndarray:
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16).ravel())
    out = np.zeros(b.size, dtype=np.float32)
    lib().orc_f16_to_f32_array(_ptr(b), _ptr(out), b.size)
    return out


def packed_bytes(fmt: int, rows: int, cols: int) -> int:
    return int(lib().orc_packed_bytes(fmt, rows, cols))


def quantize(fmt: int, src: np.ndarray, src_kind: int | None = None) -> np.ndarray:
    """Pack ``src`` [rows x cols] into ``fmt``.

    ``src`` is either uint16 (bf16 bit patterns) or float32. Returns uint8
    [rows, row_bytes].
    """
    src = np.ascontiguousarray(src)
    if src_kind is None:
        src_kind = SRC_BF16 if src.dtype == np.uint16 else SRC_F32
    if src_kind == SRC_BF16:
        assert src.dtype == np.uint16
    else:
        assert src.dtype == np.float32
    rows, cols = src.shape
    nbytes = packed_bytes(fmt, rows, cols)
    if nbytes < 0:
        raise ValueError("cols must be a multiple of the block size")
    dst = np.zeros((rows, nbytes // rows if rows else 0), dtype=np.uint8)
    rc = lib().orc_quantize(fmt, src_kind, _ptr(src), _ptr(dst), rows, cols)
    if rc != 0:
        raise ValueError("orc_quantize failed: %d" % rc)
    return dst


def dequantize(fmt: int, packed: np.ndarray, rows: int, cols: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    assert packed.size == packed_bytes(fmt, rows, cols)
    out = np.zeros((rows, cols), dtype=np.float32)
    rc = lib().orc_dequantize(fmt, _ptr(packed), _ptr(out), rows, cols)
    if rc != 0:
        raise ValueError("orc_dequantize failed: %d" % rc)
    return out


def matmul(fmt: int, packed: np.ndarray, x_bf16: np.ndarray, N: int, K: int):
    """Returns (Y, A), both float64 [M x N]: Y = X W^T over the dequantized
    weights, A = sum |w x| (scale of the tolerance)."""
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    M = x.shape[0]
    assert x.shape[1] == K
    Y = np.zeros((M, N), dtype=np.float64)
    A = np.zeros((M, N), dtype=np.float64)
    rc = lib().orc_matmul(fmt, _ptr(packed), _ptr(x), _ptr(Y), _ptr(A), M, N, K)
    if rc != 0:
        raise ValueError("orc_matmul failed: %d" % rc)
    return Y, A


def matmul_columns(fmt: int, packed: np.ndarray, x_bf16: np.ndarray, K: int, ns):
    """Y and A for the output features ``ns`` only: float64 [M x len(ns)]."""
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    M = x.shape[0]
    Y = np.zeros((M, ns.size), dtype=np.float64)
    A = np.zeros((M, ns.size), dtype=np.float64)
    rc = lib().orc_matmul_columns(fmt, _ptr(packed), _ptr(x), M, K, _ptr(ns), ns.size,
                                  _ptr(Y), _ptr(A))
    if rc != 0:
        raise ValueError("orc_matmul_columns failed: %d" % rc)
    return Y, A


def pack_scales_q4_k(sc, mc) -> np.ndarray:
    sc = np.ascontiguousarray(sc, dtype=np.int32)
    mc = np.ascontiguousarray(mc, dtype=np.int32)
    out = np.zeros(12, dtype=np.uint8)
    lib().orc_q4_k_pack_scales(_ptr(sc), _ptr(mc), _ptr(out))
    return out


def unpack_scales_q4_k(s12):
    s12 = np.ascontiguousarray(s12, dtype=np.uint8)
    sc = np.zeros(8, dtype=np.int32)
    mc = np.zeros(8, dtype=np.int32)
    lib().orc_q4_k_unpack_scales(_ptr(s12), _ptr(sc), _ptr(mc))
    return sc, mc


def gather(fmt: int, packed: np.ndarray, V: int, D: int, ids) -> np.ndarray:
    """Embedding lookup: the dequantized rows ``ids`` of the packed [V x D]
    table, float32 [len(ids) x D]."""
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    ids = np.ascontiguousarray(ids, dtype=np.int64)
    out = np.zeros((ids.size, D), dtype=np.float32)
    rc = lib().orc_gather(fmt, _ptr(packed), V, D, _ptr(ids), ids.size, _ptr(out))
    if rc != 0:
        raise ValueError("orc_gather failed: %d" % rc)
    return out


def q6_k_position(w: int):
    """(ql byte, high nibble?, qh byte, bit shift) of weight w of a Q6_K superblock."""
    pos = np.zeros(4, dtype=np.int32)
    lib().orc_q6_k_position(int(w), _ptr(pos))
    return tuple(int(v) for v in pos)


def q3_k_position(w: int):
    """(qs byte, bit shift, hmask byte, bit) of weight w of a Q3_K superblock."""
    pos = np.zeros(4, dtype=np.int32)
    lib().orc_q3_k_position(int(w), _ptr(pos))
    return tuple(int(v) for v in pos)


def q3_k_scale_field(scale_bytes, j: int) -> int:
    """The 6-bit field j (0..15) of a Q3_K superblock's 12 scale bytes."""
    b = np.ascontiguousarray(np.asarray(scale_bytes, dtype=np.uint8))
    assert b.size == 12
    return int(lib().orc_q3_k_get_field(_ptr(b), int(j)))


def f32_to_e4m3_bits(values) -> np.ndarray:
    """E4M3 encoding (round to nearest even, saturating at +-448) of float32 values."""
    v = np.ascontiguousarray(np.asarray(values, dtype=np.float32).ravel())
    out = np.zeros(v.size, dtype=np.uint8)
    lib().orc_f32_to_e4m3_array(_ptr(v), _ptr(out), v.size)
    return out


def e4m3_bits_to_f32(bits) -> np.ndarray:
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint8).ravel())
    out = np.zeros(b.size, dtype=np.float32)
    lib().orc_e4m3_to_f32_array(_ptr(b), _ptr(out), b.size)
    return out
