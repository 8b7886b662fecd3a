"""CPU oracle for the all-gather matmul -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path never calls it.

The arithmetic lives in ``oracle.c`` (a triple loop with explicit
concatenation, float32 accumulation in ascending k, round-to-nearest-even cast
to the 16-bit output type, bf16 or fp16); this module only builds it with gcc
and marshals arrays through ctypes.  Every pin of the oracle is in
``tests/test_oracle.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile ``oracle.c`` into a shared library with gcc and OpenMP."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", src, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def load(path: Optional[str] = None):
    """Load (building if needed) the oracle library and declare its symbols."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    if path is None:
        build()
    lib = ctypes.CDLL(path or _LIB)
    i64, u16p = ctypes.c_int64, ctypes.POINTER(ctypes.c_uint16)
    lib.oracle_agmm.argtypes = [
        ctypes.c_int, i64, i64, i64, ctypes.c_int,
        ctypes.POINTER(u16p), u16p, i64, i64, ctypes.c_int,
        ctypes.POINTER(ctypes.c_float), u16p, ctypes.POINTER(ctypes.c_double), ctypes.c_int,
    ]
    lib.oracle_agmm.restype = ctypes.c_int
    lib.oracle_agmm_typed.argtypes = lib.oracle_agmm.argtypes + [ctypes.c_int]
    lib.oracle_agmm_typed.restype = ctypes.c_int
    lib.oracle_f32_to_f16.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_f16.restype = ctypes.c_uint16
    lib.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_to_f32.restype = ctypes.c_float
    lib.oracle_f32_array_to_f16.argtypes = [ctypes.POINTER(ctypes.c_float), u16p, i64]
    lib.oracle_f16_array_to_f32.argtypes = [u16p, ctypes.POINTER(ctypes.c_float), i64]
    lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
    lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f32.restype = ctypes.c_float
    lib.oracle_f32_array_to_bf16.argtypes = [ctypes.POINTER(ctypes.c_float), u16p, i64]
    lib.oracle_bf16_array_to_f32.argtypes = [u16p, ctypes.POINTER(ctypes.c_float), i64]
    lib.oracle_max_threads.restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


ELEM = {"bf16": 0, "f16": 1}


def as_bits(t, dtype: str = "bf16") -> np.ndarray:
    """A contiguous uint16 array of 16-bit patterns from a torch bf16 / fp16
    tensor (matching ``dtype``) or a numpy uint16 array."""
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint16
        return np.ascontiguousarray(t)
    import torch  # local: the oracle itself does not depend on torch

    want = torch.bfloat16 if dtype == "bf16" else torch.float16
    assert t.dtype == want, (t.dtype, dtype)
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def as_bf16_bits(t) -> np.ndarray:
    """A contiguous uint16 array of bf16 bit patterns from a torch bf16 tensor
    or a numpy uint16 array."""
    return as_bits(t, "bf16")


def _infer_dtype(t) -> str:
    if isinstance(t, np.ndarray):
        return "bf16"
    import torch

    return "f16" if t.dtype == torch.float16 else "bf16"


def f16_bits_to_f32(bits: np.ndarray, lib=None) -> np.ndarray:
    """fp16 bit patterns -> float32 through the oracle's own decoder."""
    lib = lib or load()
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float32)
    lib.oracle_f16_array_to_f32(b.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)),
                                out.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), b.size)
    return out


def f32_to_f16_bits(a: np.ndarray, lib=None) -> np.ndarray:
    lib = lib or load()
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.uint16)
    lib.oracle_f32_array_to_f16(a.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                                out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)), a.size)
    return out


def bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 (exact)."""
    return (np.ascontiguousarray(bits).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(a: np.ndarray, lib=None) -> np.ndarray:
    lib = lib or load()
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.uint16)
    lib.oracle_f32_array_to_bf16(a.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                                 out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)), a.size)
    return out


def agmm(xs: Sequence, y, rhs_transpose: bool, row_begin: int = 0, row_end: Optional[int] = None,
         acc: str = "f32", nthreads: int = 0, lib=None, dtype: Optional[str] = None):
    """O = concat(xs) @ (y or y.T), rows [row_begin, row_end).

    ``xs``: P shards ``[m_per_device, k]`` (torch bf16 / fp16 or uint16 bits);
    ``y``: ``[k, n]`` or, with ``rhs_transpose``, ``[n, k]``, same type.
    ``dtype`` ("bf16" or "f16") is taken from the torch tensors when omitted.

    acc="f32" returns ``(out_f32, out_bits)``: float32 sums and their
    rounding to the 16-bit type.  acc="f64" returns the double-precision sums.
    """
    lib = lib or load()
    dtype = dtype or _infer_dtype(xs[0])
    if dtype not in ELEM:
        raise ValueError(f"unknown dtype {dtype!r}")
    elem = ELEM[dtype]
    xb = [as_bits(x, dtype) for x in xs]
    yb = as_bits(y, dtype)
    P = len(xb)
    m_pd, k = xb[0].shape
    for x in xb:
        if x.shape != (m_pd, k):
            raise ValueError("all shards must have the same shape")
    if rhs_transpose:
        n, ky = yb.shape
    else:
        ky, n = yb.shape
    if ky != k:
        raise ValueError("contracting dimension mismatch")
    M = P * m_pd
    if row_end is None:
        row_end = M
    if not (0 <= row_begin <= row_end <= M):
        raise ValueError(f"row range [{row_begin}, {row_end}) outside [0, {M})")
    rows = row_end - row_begin
    u16p = ctypes.POINTER(ctypes.c_uint16)
    ptrs = (u16p * P)(*[x.ctypes.data_as(u16p) for x in xb])
    if acc == "f64":
        out64 = np.empty((rows, n), dtype=np.float64)
        rc = lib.oracle_agmm_typed(P, m_pd, k, n, int(bool(rhs_transpose)), ptrs, yb.ctypes.data_as(u16p),
                                   row_begin, row_end, 1, None, None,
                                   out64.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), nthreads, elem)
        if rc != 0:
            raise RuntimeError(f"oracle_agmm failed: {rc}")
        return out64
    out32 = np.empty((rows, n), dtype=np.float32)
    out16 = np.empty((rows, n), dtype=np.uint16)
    rc = lib.oracle_agmm_typed(P, m_pd, k, n, int(bool(rhs_transpose)), ptrs, yb.ctypes.data_as(u16p),
                               row_begin, row_end, 0, out32.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                               out16.ctypes.data_as(u16p), None, nthreads, elem)
    if rc != 0:
        raise RuntimeError(f"oracle_agmm failed: {rc}")
    return out32, out16


def max_threads(lib=None) -> int:
    return (lib or load()).oracle_max_threads()


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
