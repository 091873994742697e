"""CPU oracle for the streaming path: TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. The CUDA library and its Python binding never
import it, and the two share no code: the oracle is plain C++ (``oracle.cpp``)
compiled on its own, wrapped here with ctypes over numpy arrays.

Every function is pinned by ``tests/test_oracle_pins.py`` against values fixed
by the pages or by mathematics rather than against itself.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

__all__ = ["Oracle", "load"]

_f32p = ctypes.POINTER(ctypes.c_float)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_f32p)


def _f32(a) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a


class Oracle:
    """ctypes wrapper around one compiled copy of ``oracle.cpp``."""

    def __init__(self, lib_path: str | None = None):
        if lib_path is None:
            lib_path = _build.build()
        self.path = lib_path
        lib = ctypes.CDLL(lib_path)
        lib.orc_scale.argtypes = [_f32p, _f32p, ctypes.c_int64, ctypes.c_float]
        lib.orc_scale.restype = None
        lib.orc_row_roll.argtypes = [_f32p, _f32p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]
        lib.orc_row_roll.restype = ctypes.c_int
        lib.orc_poly.argtypes = [_f32p, _f32p, ctypes.c_int64, _f32p, ctypes.c_int]
        lib.orc_poly.restype = ctypes.c_int
        lib.orc_cluster_exchange.argtypes = [_f32p, _f32p, ctypes.c_int64, ctypes.c_int, ctypes.c_int64]
        lib.orc_cluster_exchange.restype = ctypes.c_int
        lib.orc_cluster_exchange_ex.argtypes = [_f32p, _f32p, ctypes.c_int64, ctypes.c_int, ctypes.c_int64,
                                                ctypes.c_int64]
        lib.orc_cluster_exchange_ex.restype = ctypes.c_int
        lib.orc_cluster_all_to_all.argtypes = [_f32p, _f32p, ctypes.c_int64, ctypes.c_int, ctypes.c_int64]
        lib.orc_cluster_all_to_all.restype = ctypes.c_int
        lib.orc_masked_copy.argtypes = [_f32p, _f32p, ctypes.c_int64, ctypes.c_void_p]
        lib.orc_masked_copy.restype = ctypes.c_int
        self._lib = lib

    def scale(self, x, alpha: float) -> np.ndarray:
        x = _f32(x).ravel()
        y = np.empty_like(x)
        self._lib.orc_scale(_ptr(x), _ptr(y), x.size, ctypes.c_float(alpha))
        return y

    def row_roll(self, A, shift: int) -> np.ndarray:
        A = _f32(A)
        if A.ndim != 2:
            raise ValueError("row_roll expects a 2-D matrix")
        rows, cols = A.shape
        B = np.empty_like(A)
        rc = self._lib.orc_row_roll(_ptr(A), _ptr(B), rows, cols, int(shift))
        if rc != 0:
            raise ValueError("orc_row_roll rejected the shape")
        return B

    def poly(self, x, coeffs) -> np.ndarray:
        x = _f32(x).ravel()
        c = _f32(coeffs).ravel()
        if c.size < 1:
            raise ValueError("need at least one coefficient")
        y = np.empty_like(x)
        rc = self._lib.orc_poly(_ptr(x), _ptr(y), x.size, _ptr(c), c.size - 1)
        if rc != 0:
            raise ValueError("orc_poly rejected the degree")
        return y

    def cluster_exchange(self, x, cluster_size: int, chunk_bytes: int) -> np.ndarray:
        x = _f32(x).ravel()
        y = np.empty_like(x)
        rc = self._lib.orc_cluster_exchange(_ptr(x), _ptr(y), x.size, int(cluster_size), int(chunk_bytes))
        if rc != 0:
            raise ValueError("orc_cluster_exchange rejected the sizes")
        return y


    def cluster_exchange_ex(self, x, cluster_size: int, chunk_bytes: int, shift: int) -> np.ndarray:
        x = _f32(x).ravel()
        y = np.empty_like(x)
        rc = self._lib.orc_cluster_exchange_ex(_ptr(x), _ptr(y), x.size, int(cluster_size), int(chunk_bytes),
                                               int(shift))
        if rc != 0:
            raise ValueError("orc_cluster_exchange_ex rejected the sizes")
        return y


    def cluster_all_to_all(self, x, cluster_size: int, chunk_bytes: int) -> np.ndarray:
        x = _f32(x).ravel()
        y = np.empty_like(x)
        rc = self._lib.orc_cluster_all_to_all(_ptr(x), _ptr(y), x.size, int(cluster_size), int(chunk_bytes))
        if rc != 0:
            raise ValueError("orc_cluster_all_to_all rejected the sizes")
        return y

    def masked_copy(self, x, out_before, codes) -> np.ndarray:
        """out = out_before with chunk k replaced per codes[k] (int8, one per 16 bytes)."""
        x = _f32(x).ravel()
        y = _f32(out_before).ravel().copy()
        c = np.ascontiguousarray(codes, dtype=np.int8).ravel()
        if x.size % 4 or y.size != x.size or c.size != x.size // 4:
            raise ValueError("masked_copy needs whole 16-byte chunks and one code per chunk")
        rc = self._lib.orc_masked_copy(_ptr(x), _ptr(y), c.size, c.ctypes.data)
        if rc != 0:
            raise ValueError("orc_masked_copy rejected a code")
        return y


_default: Oracle | None = None


def load() -> Oracle:
    """The oracle built from ``oracle/oracle.cpp`` (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default
