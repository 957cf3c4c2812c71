"""Python wrapper of the fp64 CPU oracle (oracle.c).

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library and never reads the library's device layout.

Formats (canonical layouts, see oracle.c):
  FMT_SIGN1_G128: (bits uint32 [N, K/32], scales fp16-bits uint16 [N, K/128])
  FMT_AFFINE2:    (codes uint32 [N, K/16], scales uint16 [N, K/g], biases uint16 [N, K/g])
  FMT_Q4_0:       (blocks uint8 [N, K/32, 18])
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

FMT_SIGN1_G128 = 0
FMT_AFFINE2 = 1
FMT_Q4_0 = 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (no fused multiply-add) into _build/liboracle.so."""
    if force or not os.path.exists(_OUT) or os.path.getmtime(_OUT) < os.path.getmtime(_SRC):
        os.makedirs(os.path.dirname(_OUT), exist_ok=True)
        tmp = _OUT + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
             "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _OUT)
    return _OUT


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        L = ctypes.c_int64
        lib.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.orc_f16_to_f64.restype = ctypes.c_double
        lib.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_to_f64.restype = ctypes.c_double
        lib.orc_f64_to_f16.argtypes = [ctypes.c_double]
        lib.orc_f64_to_f16.restype = ctypes.c_uint16
        lib.orc_f64_to_bf16.argtypes = [ctypes.c_double]
        lib.orc_f64_to_bf16.restype = ctypes.c_uint16
        for name in ("orc_f64_to_f16_array", "orc_f64_to_bf16_array", "orc_f16_to_f64_array",
                     "orc_bf16_to_f64_array"):
            getattr(lib, name).argtypes = [P, L, P]
            getattr(lib, name).restype = None
        lib.orc_unpack.argtypes = [I, P, P, P, I, I, I, P]
        lib.orc_unpack.restype = None
        lib.orc_dequant_f16.argtypes = [I, P, P, P, I, I, P, L, P]
        lib.orc_dequant_f16.restype = None
        lib.orc_gemm.argtypes = [P, P, I, I, I, P]
        lib.orc_gemm.restype = None
        lib.orc_verify.argtypes = [I, P, P, P, I, P, I, I, P, L, P, P]
        lib.orc_verify.restype = None
        lib.orc_fwht128.argtypes = [P, I, P, P]
        lib.orc_fwht128.restype = None
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --- scalar / array conversions ------------------------------------------------

def f16_to_f64(h) -> np.ndarray:
    h = _c(h, np.uint16)
    out = np.empty(h.shape, np.float64)
    _load().orc_f16_to_f64_array(_ptr(h), h.size, _ptr(out))
    return out


def bf16_to_f64(h) -> np.ndarray:
    h = _c(h, np.uint16)
    out = np.empty(h.shape, np.float64)
    _load().orc_bf16_to_f64_array(_ptr(h), h.size, _ptr(out))
    return out


def f64_to_f16(v) -> np.ndarray:
    v = _c(v, np.float64)
    out = np.empty(v.shape, np.uint16)
    _load().orc_f64_to_f16_array(_ptr(v), v.size, _ptr(out))
    return out


def f64_to_bf16(v) -> np.ndarray:
    v = _c(v, np.float64)
    out = np.empty(v.shape, np.uint16)
    _load().orc_f64_to_bf16_array(_ptr(v), v.size, _ptr(out))
    return out


def x_to_f64(xbits, dtype: str) -> np.ndarray:
    """Activation bit patterns (uint16) of dtype 'f16' or 'bf16' -> exact fp64."""
    return f16_to_f64(xbits) if dtype == "f16" else bf16_to_f64(xbits)


def round_x(v, dtype: str) -> np.ndarray:
    """fp64 -> bit patterns of dtype 'f16' or 'bf16' (round to nearest even)."""
    return f64_to_f16(v) if dtype == "f16" else f64_to_bf16(v)


# --- weights -------------------------------------------------------------------

def _parts(fmt, parts, K, N, group):
    if fmt == FMT_SIGN1_G128:
        bits, scales = parts
        bits = _c(bits, np.uint32)
        scales = _c(scales, np.uint16)
        assert bits.size == N * (K // 32) and scales.size == N * (K // 128)
        return bits, scales, None
    if fmt == FMT_AFFINE2:
        codes, scales, biases = parts
        codes = _c(codes, np.uint32)
        scales = _c(scales, np.uint16)
        biases = _c(biases, np.uint16)
        assert codes.size == N * (K // 16)
        assert scales.size == N * (K // group) and biases.size == N * (K // group)
        return codes, scales, biases
    (blocks,) = parts
    blocks = _c(blocks, np.uint8)
    assert blocks.size == N * (K // 32) * 18
    return blocks, None, None


def unpack(fmt, parts, K, N, group=128) -> np.ndarray:
    """Dense exact weights W[K, N] (fp64)."""
    p0, p1, p2 = _parts(fmt, parts, K, N, group)
    W = np.empty((K, N), np.float64)
    _load().orc_unpack(fmt, _ptr(p0), _ptr(p1), _ptr(p2), K, N, group, _ptr(W))
    return W


def dequant_f16(fmt, parts, K, N, group=128, cols=None) -> np.ndarray:
    """fp16 bit patterns of RNE(w) for the given columns, as uint16 [K, len(cols)]."""
    p0, p1, p2 = _parts(fmt, parts, K, N, group)
    cols = np.arange(N, dtype=np.int64) if cols is None else _c(cols, np.int64)
    out = np.empty((K, cols.size), np.uint16)
    _load().orc_dequant_f16(fmt, _ptr(p0), _ptr(p1), _ptr(p2), K, group, _ptr(cols), cols.size,
                            _ptr(out))
    return out


def gemm(X, W) -> np.ndarray:
    """Naive fp64 triple loop Y = X . W."""
    X = _c(X, np.float64)
    W = _c(W, np.float64)
    M, K = X.shape
    K2, N = W.shape
    assert K == K2
    Y = np.empty((M, N), np.float64)
    _load().orc_gemm(_ptr(X), _ptr(W), M, K, N, _ptr(Y))
    return Y


def verify(fmt, parts, X, K, N, group=128, cols=None):
    """Packed verify matmul.  X: fp64 [M, K].  Returns (Y, A), each [M, len(cols)]:
    Y = X . W[:, cols] and A = sum_k |X[m,k] W[k,n]| (the tolerance scale)."""
    p0, p1, p2 = _parts(fmt, parts, K, N, group)
    X = _c(X, np.float64)
    M = X.shape[0]
    assert X.shape[1] == K
    cols = np.arange(N, dtype=np.int64) if cols is None else _c(cols, np.int64)
    Y = np.empty((M, cols.size), np.float64)
    A = np.empty((M, cols.size), np.float64)
    _load().orc_verify(fmt, _ptr(p0), _ptr(p1), _ptr(p2), group, _ptr(X), M, K, _ptr(cols),
                       cols.size, _ptr(Y), _ptr(A))
    return Y, A


def fwht128(x, signs=None) -> np.ndarray:
    """Blockwise normalized Sylvester Walsh-Hadamard rotation of each row (fp64)."""
    x = _c(x, np.float64)
    shape = x.shape
    L = shape[-1]
    assert L % 128 == 0
    x2 = x.reshape(-1, L)
    s = None if signs is None else _c(signs, np.uint32)
    out = np.empty_like(x2)
    for r in range(x2.shape[0]):
        row = np.ascontiguousarray(x2[r])
        o = np.empty(L, np.float64)
        _load().orc_fwht128(_ptr(row), L, _ptr(s), _ptr(o))
        out[r] = o
    return out.reshape(shape)


def argmax_rows(Y) -> np.ndarray:
    """Greedy choice per row (dflash-mlx-bonsai2 README, "What it does to the
    numbers": greedy decoding, acceptance by the argmax): the first column
    holding the row's largest value; -0 equals +0 and a NaN counts as the
    largest (the first NaN wins)."""
    Y = np.asarray(Y, np.float64)
    out = np.empty(Y.shape[0], np.int64)
    for m in range(Y.shape[0]):
        row = Y[m]
        nan = np.flatnonzero(np.isnan(row))
        out[m] = nan[0] if nan.size else int(np.argmax(row))
    return out
