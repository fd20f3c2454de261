"""CPU oracle for block-quantized mul_mat -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package. It never touches a GPU, shares no code with the CUDA library and
imports nothing from it. The arithmetic lives in ``gq_oracle.c`` (plain C, fp64
accumulation, single thread); this module only marshals numpy arrays into it.

Every function follows the pages as cited in ``gq_oracle.c``:
  - quantize: "A Complete Guide to llama.cpp and Customization with C++", section 2.2
    (Delta = max |w| / 7, codes in [-8, 7]) and the Q4_0 layout of "Development Guide for
    Small AI Models (TinyLLaMA, etc.) Using C++", section 6.1 (fp16 scale + 16 code bytes).
  - Q4_K super-blocks: named by the pages (the same two guides, sections 6 and 2.2) without
    a layout; the oracle follows the published GGUF Q4_K block format (gq_oracle.c) and
    its own plain min/max quantizer.
  - dequantize / mul_mat: "Development Guide ...", section 6.2 (load, unpack, dequantize,
    FMA) and "No Python! Building an AI Inference Engine Exclusively in C++", sections 6
    and 7.2 (C = A B; Y = X W^T in the cuBLAS call's layout).
  - mul_mat_q8x: "A Complete Guide to llama.cpp ...", section 2.2 (x quantized like the
    weights; y ~= Delta Delta_x sum q q_x with an integer sum per block).
  - mul_mat_rmsnorm: "Development Guide ...", section 4.1 (RMSNorm(x) = x / sqrt(mean(x^2)
    + eps) * gamma) ahead of the product.
  - mul_mat_swiglu: "Development Guide ...", section 4.4 (Swish(x W_gate) * (x W_up),
    Swish(z) = z / (1 + e^-z)).

Parity status: every function here is pinned by ``tests/test_oracle_pins.py`` (IEEE fp16
conversion against numpy, closed-form blocks, exact-rational brute force, one-hot rows).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

TYPE_Q4_0 = 2
TYPE_Q8_0 = 8
TYPE_Q4_K = 12
_TYPES = {"q4_0": TYPE_Q4_0, "q8_0": TYPE_Q8_0, "q4_k": TYPE_Q4_K, TYPE_Q4_0: TYPE_Q4_0,
          TYPE_Q8_0: TYPE_Q8_0, TYPE_Q4_K: TYPE_Q4_K}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gq_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
# IEEE arithmetic only: no fast-math, no contraction of a*b+c into fma.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile gq_oracle.c into liboracle.so next to it (gcc, a second or two)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        # GQ_ORACLE_SO names another build of gq_oracle.c; the mutation test uses it to
        # run the pins against copies with a mistake planted in them.
        lib = ctypes.CDLL(os.environ.get("GQ_ORACLE_SO") or build())
        c_int64, c_int, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        lib.oracle_fp16_from_f32.argtypes = [ctypes.c_float]
        lib.oracle_fp16_from_f32.restype = ctypes.c_uint16
        lib.oracle_f32_from_fp16.argtypes = [ctypes.c_uint16]
        lib.oracle_f32_from_fp16.restype = ctypes.c_float
        lib.oracle_fp16_from_f32_array.argtypes = [vp, c_int64, vp]
        lib.oracle_fp16_from_f32_array.restype = None
        lib.oracle_f32_from_fp16_array.argtypes = [vp, c_int64, vp]
        lib.oracle_f32_from_fp16_array.restype = None
        lib.oracle_block_bytes.argtypes = [c_int]
        lib.oracle_block_bytes.restype = c_int64
        lib.oracle_row_bytes.argtypes = [c_int, c_int64]
        lib.oracle_row_bytes.restype = c_int64
        lib.oracle_quantize.argtypes = [c_int, vp, c_int64, c_int64, vp]
        lib.oracle_quantize.restype = c_int
        lib.oracle_dequantize.argtypes = [c_int, vp, c_int64, c_int64, vp]
        lib.oracle_dequantize.restype = c_int
        lib.oracle_mul_mat.argtypes = [c_int, vp, c_int64, c_int64, vp, c_int64, vp, vp]
        lib.oracle_mul_mat.restype = c_int
        lib.oracle_mul_mat_q8x.argtypes = [c_int, vp, c_int64, c_int64, vp, c_int64, vp, vp]
        lib.oracle_mul_mat_q8x.restype = c_int
        lib.oracle_mul_mat_rmsnorm.argtypes = [c_int, vp, c_int64, c_int64, vp, vp,
                                               ctypes.c_double, c_int64, vp, vp, vp]
        lib.oracle_mul_mat_rmsnorm.restype = c_int
        lib.oracle_mul_mat_swiglu.argtypes = [c_int, vp, vp, c_int64, c_int64, vp, c_int64,
                                              vp, vp]
        lib.oracle_mul_mat_swiglu.restype = c_int
        _lib = lib
    return _lib


def _type(t) -> int:
    try:
        return _TYPES[t]
    except KeyError:
        raise ValueError(f"unknown block type {t!r}") from None


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def block_bytes(t) -> int:
    """Bytes per block: 18 for Q4_0 and 34 for Q8_0 (32 weights), 144 for Q4_K (256)."""
    return int(_load().oracle_block_bytes(_type(t)))


def block_weights(t) -> int:
    return 256 if _type(t) == TYPE_Q4_K else 32


def row_bytes(t, K: int) -> int:
    """Bytes of one row of K weights (K a multiple of block_weights(t))."""
    rb = int(_load().oracle_row_bytes(_type(t), K))
    if rb < 0:
        raise ValueError(f"K = {K} is not a multiple of the {t} block")
    return rb


def fp16_from_f32(x) -> np.ndarray:
    """IEEE binary32 -> binary16 bit patterns (uint16), round to nearest even."""
    x = _f32(x)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_fp16_from_f32_array(x.ctypes.data, x.size, out.ctypes.data)
    return out


def f32_from_fp16(h) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float32)
    _load().oracle_f32_from_fp16_array(h.ctypes.data, h.size, out.ctypes.data)
    return out


def quantize(t, W) -> np.ndarray:
    """W (M x K fp32) -> uint8 array of shape (M, K/32 * block_bytes)."""
    W = _f32(W)
    M, K = W.shape
    out = np.empty((M, row_bytes(t, K)), dtype=np.uint8)
    rc = _load().oracle_quantize(_type(t), W.ctypes.data, M, K, out.ctypes.data)
    if rc:
        raise ValueError("oracle_quantize rejected its arguments")
    return out


def dequantize(t, blocks, M: int, K: int) -> np.ndarray:
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    if blocks.size != M * row_bytes(t, K):
        raise ValueError("block buffer size does not match M, K")
    out = np.empty((M, K), dtype=np.float32)
    rc = _load().oracle_dequantize(_type(t), blocks.ctypes.data, M, K, out.ctypes.data)
    if rc:
        raise ValueError("oracle_dequantize rejected its arguments")
    return out


def mul_mat(t, blocks, M: int, K: int, X) -> np.ndarray:
    """Y (N x M fp32) = X (N x K fp32) . What^T, accumulated in fp64 on one CPU thread."""
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    X = _f32(X)
    if X.ndim == 1:
        X = X.reshape(1, -1)
    N = X.shape[0]
    if X.shape[1] != K or blocks.size != M * row_bytes(t, K):
        raise ValueError("shape mismatch")
    Y = np.empty((N, M), dtype=np.float32)
    wrow = np.empty(max(K, 1), dtype=np.float32)
    rc = _load().oracle_mul_mat(_type(t), blocks.ctypes.data, M, K, X.ctypes.data, N,
                                Y.ctypes.data, wrow.ctypes.data)
    if rc:
        raise ValueError("oracle_mul_mat rejected its arguments")
    return Y


def mul_mat_q8x(t, blocks, M: int, K: int, X) -> np.ndarray:
    """Y (N x M fp32) with X quantized per 32-block like Q8_0 and each block's dot product
    an exact integer sum ("A Complete Guide to llama.cpp ...", section 2.2):
    Y[n][m] = sum_b Delta_w * Delta_x * sum_i q_i q_x,i, in fp64 on one CPU thread."""
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    X = _f32(X)
    if X.ndim == 1:
        X = X.reshape(1, -1)
    N = X.shape[0]
    if X.shape[1] != K or blocks.size != M * row_bytes(t, K):
        raise ValueError("shape mismatch")
    Y = np.empty((N, M), dtype=np.float32)
    xq = np.empty(max(1, N * (K // 32) * 34), dtype=np.uint8)
    rc = _load().oracle_mul_mat_q8x(_type(t), blocks.ctypes.data, M, K, X.ctypes.data, N,
                                    Y.ctypes.data, xq.ctypes.data)
    if rc:
        raise ValueError("oracle_mul_mat_q8x rejected its arguments")
    return Y


def mul_mat_q8x_rows(t, blocks, M: int, K: int, X, rows) -> np.ndarray:
    """mul_mat_q8x on the selected rows only (for sampled checks of large problems)."""
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(M, row_bytes(t, K))
    rows = np.asarray(rows, dtype=np.int64)
    return mul_mat_q8x(t, np.ascontiguousarray(blocks[rows]), len(rows), K, X)


def mul_mat_rows(t, blocks, M: int, K: int, X, rows) -> np.ndarray:
    """Y[:, rows] only: the oracle run on the selected rows' blocks (row-major, so each
    row is one contiguous byte range). Used to check sampled outputs of large problems."""
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(M, row_bytes(t, K))
    rows = np.asarray(rows, dtype=np.int64)
    sub = np.ascontiguousarray(blocks[rows])
    return mul_mat(t, sub, len(rows), K, X)


def mul_mat_rmsnorm(t, blocks, M: int, K: int, X, gamma, eps: float) -> np.ndarray:
    """Y (N x M fp32) = RMSNorm(X) . What^T, RMSNorm(x) = x / sqrt(mean(x^2) + eps) * gamma
    ("Development Guide for Small AI Models (TinyLLaMA, etc.) Using C++", section 4.1),
    the normalized row and the sum in fp64, one rounding at the end."""
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    X = _f32(X)
    if X.ndim == 1:
        X = X.reshape(1, -1)
    gamma = _f32(gamma).reshape(-1)
    N = X.shape[0]
    if X.shape[1] != K or gamma.size != K or blocks.size != M * row_bytes(t, K):
        raise ValueError("shape mismatch")
    Y = np.empty((N, M), dtype=np.float32)
    wrow = np.empty(max(K, 1), dtype=np.float32)
    xhat = np.empty(max(K, 1), dtype=np.float64)
    rc = _load().oracle_mul_mat_rmsnorm(_type(t), blocks.ctypes.data, M, K, X.ctypes.data,
                                        gamma.ctypes.data, float(eps), N, Y.ctypes.data,
                                        wrow.ctypes.data, xhat.ctypes.data)
    if rc:
        raise ValueError("oracle_mul_mat_rmsnorm rejected its arguments")
    return Y


def mul_mat_swiglu(t, gate, up, M: int, K: int, X) -> np.ndarray:
    """H (N x M fp32) = Swish(X . Wgate_hat^T) * (X . Wup_hat^T), Swish(z) = z / (1 + e^-z)
    ("Development Guide ...", section 4.4), both sums, Swish and the product in fp64."""
    gate = np.ascontiguousarray(gate, dtype=np.uint8)
    up = np.ascontiguousarray(up, dtype=np.uint8)
    X = _f32(X)
    if X.ndim == 1:
        X = X.reshape(1, -1)
    N = X.shape[0]
    if X.shape[1] != K or gate.size != M * row_bytes(t, K) or up.size != gate.size:
        raise ValueError("shape mismatch")
    H = np.empty((N, M), dtype=np.float32)
    wrow = np.empty(max(2 * K, 1), dtype=np.float32)
    rc = _load().oracle_mul_mat_swiglu(_type(t), gate.ctypes.data, up.ctypes.data, M, K,
                                       X.ctypes.data, N, H.ctypes.data, wrow.ctypes.data)
    if rc:
        raise ValueError("oracle_mul_mat_swiglu rejected its arguments")
    return H


def _rows_of(t, blocks, M: int, K: int, rows) -> np.ndarray:
    b = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(M, row_bytes(t, K))
    return np.ascontiguousarray(b[np.asarray(rows, dtype=np.int64)])


def mul_mat_rmsnorm_rows(t, blocks, M: int, K: int, X, gamma, eps: float, rows) -> np.ndarray:
    """mul_mat_rmsnorm on the selected rows only (sampled checks of large problems)."""
    return mul_mat_rmsnorm(t, _rows_of(t, blocks, M, K, rows), len(rows), K, X, gamma, eps)


def mul_mat_swiglu_rows(t, gate, up, M: int, K: int, X, rows) -> np.ndarray:
    """mul_mat_swiglu on the selected rows only."""
    return mul_mat_swiglu(t, _rows_of(t, gate, M, K, rows), _rows_of(t, up, M, K, rows),
                          len(rows), K, X)
