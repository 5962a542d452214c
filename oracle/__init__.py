"""CPU oracle for the NWC entropy-coded matrix format (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package. The product library never calls it.

``oracle.c`` is a plain C restatement of the format and of the plain
matrix-vector definition; this module compiles it with gcc (``build()``) and
wraps it with ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None

BF16, FP8 = 0, 1


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so (plain -O2, no vector flags)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", _LIB, _SRC, "-lm"])
    return _LIB


def _L():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        u64, p = ctypes.c_uint64, ctypes.c_void_p
        lib.orc_encode.argtypes = [p, p, u64, u64, ctypes.c_int, ctypes.POINTER(p), ctypes.POINTER(u64)]
        lib.orc_free.argtypes = [p]
        lib.orc_info.argtypes = [p, u64, p, p]
        lib.orc_decode.argtypes = [p, u64, p, p]
        lib.orc_quantize_fp8.argtypes = [p, u64, u64, p, p]
        lib.orc_dequantize_fp8.argtypes = [p, p, u64, u64, p]
        lib.orc_e4m3_from_f32.argtypes = [ctypes.c_float]
        lib.orc_e4m3_from_f32.restype = ctypes.c_uint8
        lib.orc_gemv_rows.argtypes = [p, u64, p, p, u64, p]
        lib.orc_abs_dot_rows.argtypes = [p, u64, p, p, u64, p]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def encode(e: np.ndarray, elem: int = BF16, scales: np.ndarray | None = None) -> bytes:
    """Encode an (N, K) matrix: BF16 bit patterns (uint16) or fp8 bytes (uint8)
    with fp32 row scales. Returns the blob."""
    e = np.ascontiguousarray(e)
    n, k = e.shape
    e16 = np.ascontiguousarray(e.astype(np.uint16))
    sc = None
    if elem == FP8:
        sc = np.ascontiguousarray(np.asarray(scales, dtype=np.float32))
        assert sc.shape == (n,)
    out = ctypes.c_void_p()
    nbytes = ctypes.c_uint64()
    rc = _L().orc_encode(_ptr(e16), _ptr(sc) if sc is not None else None, n, k, elem,
                         ctypes.byref(out), ctypes.byref(nbytes))
    if rc != 0:
        raise ValueError(f"oracle encode failed ({rc})")
    blob = ctypes.string_at(out, nbytes.value)
    _L().orc_free(out)
    return blob


def info(blob: bytes) -> dict:
    out = np.zeros(6, np.uint64)
    ranks = np.zeros(16, np.uint8)
    b = np.frombuffer(blob, np.uint8)
    if _L().orc_info(_ptr(b), len(blob), _ptr(out), _ptr(ranks)) != 0:
        raise ValueError("malformed blob")
    elem, nr, n, k, nb, total = (int(v) for v in out)
    return dict(elem=elem, n_ranked=nr, N=n, K=k, n_blocks=nb, total=total, rank_exp=ranks[:nr].tolist())


def decode(blob: bytes):
    """Blob -> (N, K) uint16 BF16 bits (or uint8 fp8 bytes) and fp32 scales (fp8) or None."""
    h = info(blob)
    b = np.frombuffer(blob, np.uint8)
    e = np.zeros((h["N"], h["K"]), np.uint16)
    sc = np.zeros(h["N"], np.float32) if h["elem"] == FP8 else None
    rc = _L().orc_decode(_ptr(b), len(blob), _ptr(e), _ptr(sc) if sc is not None else None)
    if rc != 0:
        raise ValueError("malformed blob")
    if h["elem"] == FP8:
        return e.astype(np.uint8), sc
    return e, None


def quantize_fp8(w_bits: np.ndarray):
    """Per-row e4m3 quantization of BF16 bits: (q uint8 (N, K), scales fp32 (N,))."""
    w = np.ascontiguousarray(w_bits, dtype=np.uint16)
    n, k = w.shape
    q = np.zeros((n, k), np.uint8)
    s = np.zeros(n, np.float32)
    if _L().orc_quantize_fp8(_ptr(w), n, k, _ptr(q), _ptr(s)) != 0:
        raise ValueError("non-finite weight")
    return q, s


def dequantize_fp8(q: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """BF16 bits (uint16 (N, K)) of the FP32 products e4m3(q) * s_n, rounded to nearest even."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = np.ascontiguousarray(scales, dtype=np.float32)
    n, k = q.shape
    out = np.zeros((n, k), np.uint16)
    _L().orc_dequantize_fp8(_ptr(q), _ptr(s), n, k, _ptr(out))
    return out


def e4m3_from_f32(x: float) -> int:
    return int(_L().orc_e4m3_from_f32(float(x)))


def gemv(blob: bytes, x_bits: np.ndarray, rows=None) -> np.ndarray:
    """FP64 y = W x for the listed rows (all rows if None)."""
    h = info(blob)
    b = np.frombuffer(blob, np.uint8)
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    assert x.shape == (h["K"],)
    if rows is None:
        r = None
        n = h["N"]
    else:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n = len(r)
    y = np.zeros(n, np.float64)
    if _L().orc_gemv_rows(_ptr(b), len(blob), _ptr(x), _ptr(r) if r is not None else None, n, _ptr(y)) != 0:
        raise ValueError("malformed blob or row")
    return y


def abs_dot(blob: bytes, x_bits: np.ndarray, rows=None) -> np.ndarray:
    """FP64 sum_k |w x| per listed row (the tolerance scale)."""
    h = info(blob)
    b = np.frombuffer(blob, np.uint8)
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    if rows is None:
        r, n = None, h["N"]
    else:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n = len(r)
    out = np.zeros(n, np.float64)
    if _L().orc_abs_dot_rows(_ptr(b), len(blob), _ptr(x), _ptr(r) if r is not None else None, n, _ptr(out)) != 0:
        raise ValueError("malformed blob or row")
    return out
