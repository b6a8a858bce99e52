"""Row-wise softmax oracle (double precision, single-threaded CPU).

TEST INFRASTRUCTURE ONLY.  Only tests/, ``__graft_entry__.smoke()`` and
bench.py's ``cpu_baseline`` / ``--impl reference`` leg may import this module.
The library (``row_wise_softmax_gb300``) never imports it and shares no code
with it; the C source ``softmax_oracle.c`` includes nothing from the CUDA path.

The functions restate the pages' softmax (the "Level 1: Softmax" formula of
the cs336 lecture 6 notes and the fused-softmax example of "Triton: write
CUDA-grade GPU operators in Python"), the online (m, l) recurrence of
"Triton GPU programming deep dive" section 3.3, the scaled and causally
masked softmax of attention scores (the same page, sections 3.1 and 3.3),
and the tiled row sum of the
lecture notes' "Level 2".  See ``softmax_oracle.c`` for each function's
citation.  Every function is pinned in tests/test_oracle_pins.py.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "softmax_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

F32 = 0
BF16 = 1
F16 = 2

# -ffp-contract=off: no fused multiply-add contraction, so x86 and Arm hosts
# produce the same doubles.  No fast-math: rint() must round ties to even.
_CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle with gcc into ``out`` (default: oracle/liboracle.so)."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + ".tmp%d" % os.getpid()
    subprocess.run(["gcc", *_CFLAGS, src, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out)
    return out


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i64, dbl, vp = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        lib.oracle_softmax_rows.argtypes = [vp, vp, i64, i64, i64, i64, ctypes.c_int, i64]
        lib.oracle_softmax_rows.restype = ctypes.c_int
        lib.oracle_softmax_rows_ex.argtypes = [vp, vp, i64, i64, i64, i64, ctypes.c_int, i64,
                                               dbl, ctypes.c_int, i64, i64]
        lib.oracle_softmax_rows_ex.restype = ctypes.c_int
        lib.oracle_double_to_bf16.argtypes = [dbl]
        lib.oracle_double_to_bf16.restype = ctypes.c_uint16
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = dbl
        lib.oracle_double_to_bf16_array.argtypes = [vp, vp, i64]
        lib.oracle_bf16_to_double_array.argtypes = [vp, vp, i64]
        lib.oracle_double_to_f16.argtypes = [dbl]
        lib.oracle_double_to_f16.restype = ctypes.c_uint16
        lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_double.restype = dbl
        lib.oracle_double_to_f16_array.argtypes = [vp, vp, i64]
        lib.oracle_f16_to_double_array.argtypes = [vp, vp, i64]
        lib.oracle_softmax_backward_rows.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64,
                                                     ctypes.c_int]
        lib.oracle_softmax_backward_rows.restype = ctypes.c_int
        lib.oracle_softmax_strided.argtypes = [vp, vp, i64, i64, i64, i64, ctypes.c_int]
        lib.oracle_softmax_strided.restype = ctypes.c_int
        lib.oracle_tiled_row_sum.argtypes = [vp, i64, i64, i64, vp]
        lib.oracle_tiled_row_sum.restype = dbl
        self._lib = lib

    def softmax_rows(self, buf: np.ndarray, n_rows: int, n_cols: int,
                     in_row_stride: int | None = None, dtype: int = F32,
                     tile: int = 0, scale: float = 1.0, causal: bool = False,
                     causal_period: int = 0, causal_offset: int = 0) -> np.ndarray:
        """Softmax of each row of a strided row matrix, in double.

        ``buf`` is the flat input buffer: float32 values (dtype F32), or bf16
        (dtype BF16) or fp16 (dtype F16) bit patterns as uint16.  Row r starts at element
        ``r * in_row_stride``.  Returns a dense float64 array [n_rows, n_cols].
        ``tile > 0`` uses the online (m, l) recurrence with that tile width.
        ``scale`` multiplies the inputs (exactly, in double) before the
        softmax; ``causal`` keeps column c of row r iff c <= (r mod
        causal_period) + causal_offset (period <= 0: n_rows), the rest -inf.
        """
        if in_row_stride is None:
            in_row_stride = n_cols
        want = np.float32 if dtype == F32 else np.uint16
        buf = np.ascontiguousarray(buf).reshape(-1)
        if buf.dtype != want:
            raise TypeError("oracle: buffer dtype %s, expected %s" % (buf.dtype, want))
        if n_rows > 0 and n_cols > 0 and buf.size < (n_rows - 1) * in_row_stride + n_cols:
            raise ValueError("oracle: buffer too small for the strided rows")
        out = np.empty((n_rows, n_cols), dtype=np.float64)
        if scale == 1.0 and not causal:
            rc = self._lib.oracle_softmax_rows(buf.ctypes.data, out.ctypes.data, n_rows, n_cols,
                                               in_row_stride, n_cols, dtype, tile)
        else:
            rc = self._lib.oracle_softmax_rows_ex(buf.ctypes.data, out.ctypes.data, n_rows,
                                                  n_cols, in_row_stride, n_cols, dtype, tile,
                                                  float(np.float32(scale)), 1 if causal else 0,
                                                  causal_period, causal_offset)
        if rc != 0:
            raise ValueError("oracle_softmax_rows rejected its arguments")
        return out

    def to_bf16(self, values: np.ndarray) -> np.ndarray:
        """Round doubles to bf16 (ties to even); returns uint16 bit patterns."""
        v = np.ascontiguousarray(values, dtype=np.float64)
        out = np.empty(v.shape, dtype=np.uint16)
        self._lib.oracle_double_to_bf16_array(v.ctypes.data, out.ctypes.data, v.size)
        return out

    def softmax_backward_rows(self, y: np.ndarray, dy: np.ndarray, n_rows: int, n_cols: int,
                              y_row_stride: int | None = None, dy_row_stride: int | None = None,
                              dtype: int = F32) -> np.ndarray:
        """dx = y * (dy - sum(y * dy)) per row, in double, from flat y and dy
        buffers (float32 values, or 16-bit patterns as uint16); returns a dense
        float64 array [n_rows, n_cols]."""
        ys = n_cols if y_row_stride is None else y_row_stride
        gs = n_cols if dy_row_stride is None else dy_row_stride
        want = np.float32 if dtype == F32 else np.uint16
        y = np.ascontiguousarray(y).reshape(-1)
        dy = np.ascontiguousarray(dy).reshape(-1)
        for b, st in ((y, ys), (dy, gs)):
            if b.dtype != want:
                raise TypeError("oracle: buffer dtype %s, expected %s" % (b.dtype, want))
            if n_rows > 0 and n_cols > 0 and b.size < (n_rows - 1) * st + n_cols:
                raise ValueError("oracle: buffer too small for the strided rows")
        out = np.empty((n_rows, n_cols), dtype=np.float64)
        rc = self._lib.oracle_softmax_backward_rows(y.ctypes.data, dy.ctypes.data, out.ctypes.data,
                                                    n_rows, n_cols, ys, gs, n_cols, dtype)
        if rc != 0:
            raise ValueError("oracle_softmax_backward_rows rejected its arguments")
        return out

    def softmax_strided(self, buf: np.ndarray, n_rows: int, n_cols: int, in_row_stride: int,
                        in_col_stride: int, dtype: int = F32) -> np.ndarray:
        """Softmax over rows whose element c of row r is buf[r * in_row_stride +
        c * in_col_stride] (non-negative strides); dense float64 [n_rows, n_cols]."""
        want = np.float32 if dtype == F32 else np.uint16
        buf = np.ascontiguousarray(buf).reshape(-1)
        if buf.dtype != want:
            raise TypeError("oracle: buffer dtype %s, expected %s" % (buf.dtype, want))
        if in_row_stride < 0 or in_col_stride < 0:
            raise ValueError("oracle: strides must be non-negative")
        if n_rows > 0 and n_cols > 0 and \
                buf.size <= (n_rows - 1) * in_row_stride + (n_cols - 1) * in_col_stride:
            raise ValueError("oracle: buffer too small for the strided rows")
        out = np.empty((n_rows, n_cols), dtype=np.float64)
        rc = self._lib.oracle_softmax_strided(buf.ctypes.data, out.ctypes.data, n_rows, n_cols,
                                              in_row_stride, in_col_stride, dtype)
        if rc != 0:
            raise ValueError("oracle_softmax_strided rejected its arguments")
        return out

    def to_f16(self, values: np.ndarray) -> np.ndarray:
        """Round doubles to fp16 (ties to even); returns uint16 bit patterns."""
        v = np.ascontiguousarray(values, dtype=np.float64)
        out = np.empty(v.shape, dtype=np.uint16)
        self._lib.oracle_double_to_f16_array(v.ctypes.data, out.ctypes.data, v.size)
        return out

    def f16_to_double(self, bits: np.ndarray) -> np.ndarray:
        b = np.ascontiguousarray(bits, dtype=np.uint16)
        out = np.empty(b.shape, dtype=np.float64)
        self._lib.oracle_f16_to_double_array(b.ctypes.data, out.ctypes.data, b.size)
        return out

    def bf16_to_double(self, bits: np.ndarray) -> np.ndarray:
        b = np.ascontiguousarray(bits, dtype=np.uint16)
        out = np.empty(b.shape, dtype=np.float64)
        self._lib.oracle_bf16_to_double_array(b.ctypes.data, out.ctypes.data, b.size)
        return out

    def tiled_row_sum(self, x: np.ndarray, block: int, snapshot_tiles: int):
        """Returns (row sum, lane accumulators after ``snapshot_tiles`` tiles)."""
        xv = np.ascontiguousarray(x, dtype=np.float64)
        acc = np.zeros(block, dtype=np.float64)
        s = self._lib.oracle_tiled_row_sum(xv.ctypes.data, xv.size, block,
                                           snapshot_tiles, acc.ctypes.data)
        return s, acc


_default: Oracle | None = None


def load() -> Oracle:
    """Build (if needed) and load the oracle library."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def softmax_rows(*args, **kwargs) -> np.ndarray:
    return load().softmax_rows(*args, **kwargs)


def to_bf16(values: np.ndarray) -> np.ndarray:
    return load().to_bf16(values)


def bf16_to_double(bits: np.ndarray) -> np.ndarray:
    return load().bf16_to_double(bits)


def to_f16(values: np.ndarray) -> np.ndarray:
    return load().to_f16(values)


def f16_to_double(bits: np.ndarray) -> np.ndarray:
    return load().f16_to_double(bits)


def softmax_backward_rows(*args, **kwargs) -> np.ndarray:
    return load().softmax_backward_rows(*args, **kwargs)


def softmax_strided(*args, **kwargs) -> np.ndarray:
    return load().softmax_strided(*args, **kwargs)
