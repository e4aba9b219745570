"""fp64 CPU oracle for masked scaled dot-product attention (test infrastructure).

NOT part of the product path.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg may import this package.  It shares no code
with the CUDA library and imports nothing from it.

``attn_oracle.c`` is the plain definition (see its header for the passages it
follows and the readings taken where the pages are silent); ``brute.py`` is a
second, independent statement of the same formula for tiny sizes.  Both are
pinned by ``tests/test_oracle_pins.py`` against the pages' worked examples,
closed forms, invariants and a library routine.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "attn_oracle.c")
LIBRARY = os.path.join(_HERE, "liboracle.so")

MASK_KEY_PADDING = 1
MASK_CAUSAL = 2
MASK_WINDOW = 4


def compile_oracle(source: str = SOURCE, output: str = LIBRARY, openmp: bool = True) -> str:
    """Compile the C oracle into a shared library with gcc (portable flags only)."""
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", source, "-o", output, "-lm"]
    if openmp:
        try:
            subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                           capture_output=True, text=True)
            return output
        except subprocess.CalledProcessError:
            pass  # no libgomp: build a single-threaded oracle instead
    subprocess.run(base, check=True, capture_output=True, text=True)
    return output


def _stale(lib: str, src: str) -> bool:
    return not os.path.exists(lib) or os.path.getmtime(lib) < os.path.getmtime(src)


class Oracle:
    """ctypes handle on one compiled oracle library."""

    def __init__(self, path: str):
        self.path = path
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        i32p = ctypes.POINTER(ctypes.c_int32)
        i64p = ctypes.POINTER(ctypes.c_int64)
        i64 = ctypes.c_int64
        lib.oracle_attn_fwd.argtypes = [dp, dp, dp, i32p, ctypes.c_int, ctypes.c_double,
                                        i64, i64, i64, i64, i64, dp]
        lib.oracle_attn_fwd.restype = ctypes.c_int
        lib.oracle_attn_rows.argtypes = [dp, dp, dp, i32p, ctypes.c_int, ctypes.c_double,
                                         i64, i64, i64, i64, i64, i64p, i64, dp]
        lib.oracle_attn_rows.restype = ctypes.c_int
        lib.oracle_bf16_to_f64.argtypes = [ctypes.POINTER(ctypes.c_uint16), dp, i64]
        lib.oracle_bf16_to_f64.restype = None
        lib.oracle_f32_to_f64.argtypes = [ctypes.POINTER(ctypes.c_float), dp, i64]
        lib.oracle_f32_to_f64.restype = None
        lib.oracle_attn_fwd_w.argtypes = [dp, dp, dp, i32p, ctypes.c_int, i64, ctypes.c_double,
                                          i64, i64, i64, i64, i64, dp]
        lib.oracle_attn_fwd_w.restype = ctypes.c_int
        lib.oracle_attn_rows_w.argtypes = [dp, dp, dp, i32p, ctypes.c_int, i64, ctypes.c_double,
                                           i64, i64, i64, i64, i64, i64p, i64, dp]
        lib.oracle_attn_rows_w.restype = ctypes.c_int
        lib.oracle_attn_lse_w.argtypes = [dp, dp, i32p, ctypes.c_int, i64, ctypes.c_double,
                                          i64, i64, i64, i64, i64, dp]
        lib.oracle_attn_lse_w.restype = ctypes.c_int
        lib.oracle_attn_lse.argtypes = [dp, dp, i32p, ctypes.c_int, ctypes.c_double,
                                        i64, i64, i64, i64, i64, dp]
        lib.oracle_attn_lse.restype = ctypes.c_int
        lib.oracle_attn_bwd.argtypes = [dp, dp, dp, dp, i32p, ctypes.c_int, ctypes.c_double,
                                        i64, i64, i64, i64, i64, i64p, i64, dp, dp, dp]
        lib.oracle_attn_bwd.restype = ctypes.c_int
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        lib.oracle_set_num_threads.restype = None
        self._lib = lib

    # -- input widening ---------------------------------------------------
    def widen(self, x: np.ndarray) -> np.ndarray:
        """bf16 bit patterns (uint16) or float32/float64 -> float64, exactly."""
        x = np.ascontiguousarray(x)
        out = np.empty(x.shape, dtype=np.float64)
        dp = ctypes.POINTER(ctypes.c_double)
        if x.dtype == np.uint16:
            self._lib.oracle_bf16_to_f64(x.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)),
                                         out.ctypes.data_as(dp), x.size)
        elif x.dtype == np.float32:
            self._lib.oracle_f32_to_f64(x.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                                        out.ctypes.data_as(dp), x.size)
        elif x.dtype == np.float64:
            out[...] = x
        else:
            raise TypeError(f"oracle inputs must be uint16 (bf16 bits), float32 or float64, got {x.dtype}")
        return out

    def num_threads(self) -> int:
        return int(self._lib.oracle_num_threads())

    def set_num_threads(self, n: int) -> None:
        """Threads the row loops use from now on (timing only; results do not depend on it)."""
        self._lib.oracle_set_num_threads(int(n))

    @staticmethod
    def _dims(q, k, v):
        if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
            raise ValueError("q, k, v must be [B, h, len, d]")
        B, h, m, d = q.shape
        if k.shape[:2] != (B, h) or v.shape != k.shape or k.shape[3] != d:
            raise ValueError(f"shape mismatch q{q.shape} k{k.shape} v{v.shape}")
        return B, h, m, k.shape[2], d

    def attn_fwd(self, q, k, v, key_lengths: Optional[np.ndarray], mask_kind: int,
                 scale: float, window: Optional[int] = None) -> np.ndarray:
        """Every output row, float64 [B, h, m, d].  window: half-width of the restricted-
        attention window (used when mask_kind has MASK_WINDOW)."""
        q, k, v = self.widen(q), self.widen(k), self.widen(v)
        B, h, m, n, d = self._dims(q, k, v)
        lens = None if key_lengths is None else np.ascontiguousarray(key_lengths, dtype=np.int32)
        out = np.empty((B, h, m, d), dtype=np.float64)
        dp = ctypes.POINTER(ctypes.c_double)
        lp = None if lens is None else lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
        if window is not None:
            rc = self._lib.oracle_attn_fwd_w(q.ctypes.data_as(dp), k.ctypes.data_as(dp), v.ctypes.data_as(dp),
                                             lp, int(mask_kind), int(window), float(scale), B, h, m, n, d,
                                             out.ctypes.data_as(dp))
            if rc != 0:
                raise RuntimeError("oracle_attn_fwd_w failed")
            return out
        rc = self._lib.oracle_attn_fwd(
            q.ctypes.data_as(dp), k.ctypes.data_as(dp), v.ctypes.data_as(dp), lp,
            int(mask_kind), float(scale), B, h, m, n, d, out.ctypes.data_as(dp))
        if rc != 0:
            raise RuntimeError("oracle_attn_fwd failed")
        return out

    def attn_rows(self, q, k, v, key_lengths: Optional[np.ndarray], mask_kind: int,
                  scale: float, rows: np.ndarray, widened: bool = False,
                  window: Optional[int] = None) -> np.ndarray:
        """Selected output rows (linear ids ((b*h+head)*m+i)), float64 [len(rows), d]."""
        if not widened:
            q, k, v = self.widen(q), self.widen(k), self.widen(v)
        B, h, m, n, d = self._dims(q, k, v)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        lens = None if key_lengths is None else np.ascontiguousarray(key_lengths, dtype=np.int32)
        out = np.empty((rows.size, d), dtype=np.float64)
        dp = ctypes.POINTER(ctypes.c_double)
        lp = None if lens is None else lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
        rp = rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
        if window is not None:
            rc = self._lib.oracle_attn_rows_w(q.ctypes.data_as(dp), k.ctypes.data_as(dp), v.ctypes.data_as(dp),
                                              lp, int(mask_kind), int(window), float(scale), B, h, m, n, d,
                                              rp, rows.size, out.ctypes.data_as(dp))
        else:
            rc = self._lib.oracle_attn_rows(
                q.ctypes.data_as(dp), k.ctypes.data_as(dp), v.ctypes.data_as(dp), lp,
                int(mask_kind), float(scale), B, h, m, n, d, rp, rows.size, out.ctypes.data_as(dp))
        if rc != 0:
            raise RuntimeError("oracle_attn_rows failed")
        return out

    def attn_lse(self, q, k, key_lengths: Optional[np.ndarray], mask_kind: int, scale: float,
                 window: Optional[int] = None) -> np.ndarray:
        """Natural log of each row's softmax normaliser, float64 [B, h, m] (-inf: no allowed key)."""
        q, k = self.widen(q), self.widen(k)
        B, h, m, n, d = self._dims(q, k, k)
        lens = None if key_lengths is None else np.ascontiguousarray(key_lengths, dtype=np.int32)
        out = np.empty((B, h, m), dtype=np.float64)
        dp = ctypes.POINTER(ctypes.c_double)
        lp = None if lens is None else lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
        if window is not None:
            rc = self._lib.oracle_attn_lse_w(q.ctypes.data_as(dp), k.ctypes.data_as(dp), lp, int(mask_kind),
                                             int(window), float(scale), B, h, m, n, d, out.ctypes.data_as(dp))
            if rc != 0:
                raise RuntimeError("oracle_attn_lse_w failed")
            return out
        rc = self._lib.oracle_attn_lse(
            q.ctypes.data_as(dp), k.ctypes.data_as(dp), lp,
            int(mask_kind), float(scale), B, h, m, n, d, out.ctypes.data_as(dp))
        if rc != 0:
            raise RuntimeError("oracle_attn_lse failed")
        return out

    def attn_bwd(self, q, k, v, do, key_lengths: Optional[np.ndarray], mask_kind: int, scale: float,
                 heads: Optional[np.ndarray] = None):
        """Gradients (dQ, dK, dV) of sum(dO * out), float64, shaped like q, k, v.

        heads: linear (batch * h + head) ids to compute; the others stay NaN.
        """
        q, k, v, do = self.widen(q), self.widen(k), self.widen(v), self.widen(do)
        B, h, m, n, d = self._dims(q, k, v)
        if do.shape != q.shape:
            raise ValueError(f"dO{do.shape} must match q{q.shape}")
        lens = None if key_lengths is None else np.ascontiguousarray(key_lengths, dtype=np.int32)
        dq = np.full(q.shape, np.nan)
        dk = np.full(k.shape, np.nan)
        dv = np.full(v.shape, np.nan)
        hl = None if heads is None else np.ascontiguousarray(heads, dtype=np.int64)
        dp = ctypes.POINTER(ctypes.c_double)
        rc = self._lib.oracle_attn_bwd(
            q.ctypes.data_as(dp), k.ctypes.data_as(dp), v.ctypes.data_as(dp), do.ctypes.data_as(dp),
            None if lens is None else lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
            int(mask_kind), float(scale), B, h, m, n, d,
            None if hl is None else hl.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
            0 if hl is None else hl.size,
            dq.ctypes.data_as(dp), dk.ctypes.data_as(dp), dv.ctypes.data_as(dp))
        if rc != 0:
            raise RuntimeError("oracle_attn_bwd failed")
        return dq, dk, dv


_default: Optional[Oracle] = None


def load(path: Optional[str] = None) -> Oracle:
    """The compiled oracle (building it on first use if it is missing or stale)."""
    global _default
    if path is not None:
        return Oracle(path)
    if _default is None:
        if _stale(LIBRARY, SOURCE):
            compile_oracle()
        _default = Oracle(LIBRARY)
    return _default
