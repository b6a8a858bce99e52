"""Comparison of the CUDA path's outputs with the oracle's, element by element.

Tolerances (fixed here, used by every parity test):
  fp32 output: max |y - y*| <= 2e-6 and max over rows |sum_j y_j - 1| <= 1e-5,
               the row sum taken in double over the fp32 outputs;
  bf16 output: at most 1 bf16 ulp from y* rounded to bf16 (round to nearest
               even), measured as the distance of the two values in the
               ordered-integer view of bf16 bit patterns.  One ulp allows for
               the double rounding double -> fp32 -> bf16 at near-ties.
  fp16 output: the same, with binary16 in place of bf16.
  all:        where the oracle gives exactly 0 (a -inf input in a finite row)
               the output is exactly +0; where the oracle gives NaN (a row
               with NaN, +inf, or only -inf) the output is NaN.
"""
from __future__ import annotations

import numpy as np

import oracle
import workloads as wl

F32_ABS_TOL = 2e-6
F32_ROWSUM_TOL = 1e-5
BF16_ULP_TOL = 1


def decode16(bits: np.ndarray, dtype: int) -> np.ndarray:
    return oracle.bf16_to_double(bits) if dtype == wl.BF16 else oracle.f16_to_double(bits)


def bf16_ordered(bits: np.ndarray) -> np.ndarray:
    """Map bf16 (or fp16: the same sign-magnitude layout) bit patterns to
    integers that order like their values (+0 == -0)."""
    b = bits.astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def torch_dtype(dtype: int):
    import torch
    return {wl.F32: torch.float32, wl.BF16: torch.bfloat16, wl.F16: torch.float16}[dtype]


def device_input(w: wl.Workload):
    import torch
    if w.dtype == wl.F32:
        return torch.from_numpy(w.data).cuda()
    return torch.from_numpy(w.data.view(np.int16)).cuda().view(torch_dtype(w.dtype))


def empty_output(w: wl.Workload, fill=None):
    import torch
    t = torch.empty(max(w.out_elems, 1), dtype=torch_dtype(w.dtype), device="cuda")
    if fill is not None:
        t.fill_(fill)
    return t


def host_output(t, w: wl.Workload) -> np.ndarray:
    """Dense [n_rows, n_cols] view of a strided device output (float32, or uint16 bf16 bits)."""
    import torch
    flat = t.cpu()
    if w.dtype != wl.F32:
        flat = flat.view(torch.int16).numpy().view(np.uint16)
    else:
        flat = flat.numpy()
    if w.n_rows == 0 or w.n_cols == 0:
        return flat[:0].reshape(w.n_rows, w.n_cols) if flat.size else np.zeros((w.n_rows, w.n_cols))
    idx = (np.arange(w.n_rows)[:, None] * w.out_row_stride + np.arange(w.n_cols)[None, :])
    return flat[idx]


def expected(w: wl.Workload, rows: np.ndarray | None = None) -> np.ndarray:
    """Oracle output (double) for all rows, or for the listed rows only."""
    if rows is None:
        return oracle.softmax_rows(w.data, w.n_rows, w.n_cols, w.in_row_stride, w.dtype)
    stride = w.in_row_stride
    parts = [w.data[r * stride: r * stride + w.n_cols] for r in rows]
    buf = np.concatenate(parts) if parts else w.data[:0]
    return oracle.softmax_rows(buf, len(rows), w.n_cols, w.n_cols, w.dtype)


def compare(got: np.ndarray, want: np.ndarray, dtype: int, what: str = "") -> dict:
    """Assert the tolerances above; returns the measured errors."""
    assert got.shape == want.shape, (got.shape, want.shape)
    nan_rows = np.isnan(want).any(axis=1)
    stats = {"rows": int(want.shape[0]), "nan_rows": int(nan_rows.sum())}
    if nan_rows.any():
        g = got[nan_rows]
        if dtype == wl.F32:
            gv = g.astype(np.float64)
        else:
            gv = decode16(g, dtype)
        assert np.all(np.isnan(gv)), "%s: rows the formula makes NaN are not all NaN" % what
    ok = ~nan_rows
    g, w = got[ok], want[ok]
    if g.size == 0:
        return stats
    zero = w == 0.0
    if dtype == wl.F32:
        gd = g.astype(np.float64)
        err = np.abs(gd - w)
        assert not np.isnan(gd).any(), "%s: NaN output in a finite row" % what
        stats["max_abs_err"] = float(err.max())
        rs = np.abs(gd.sum(axis=1) - 1.0)
        stats["max_rowsum_err"] = float(rs.max())
        assert stats["max_abs_err"] <= F32_ABS_TOL, "%s: max abs err %.3g at %s" % (
            what, stats["max_abs_err"], np.unravel_index(np.argmax(err), err.shape))
        assert stats["max_rowsum_err"] <= F32_ROWSUM_TOL, "%s: row sum err %.3g" % (
            what, stats["max_rowsum_err"])
        assert np.all(g.view(np.uint32)[zero] == 0), "%s: masked output not +0" % what
    else:
        wb = oracle.to_bf16(w) if dtype == wl.BF16 else oracle.to_f16(w)
        d = np.abs(bf16_ordered(g) - bf16_ordered(wb))
        stats["max_ulp"] = int(d.max())
        stats["ulp_gt0"] = int((d > 0).sum())
        gd = decode16(g, dtype)
        stats["max_rowsum_err"] = float(np.abs(gd.sum(axis=1) - 1.0).max())
        assert stats["max_ulp"] <= BF16_ULP_TOL, "%s: %d ulp (16-bit) at %s" % (
            what, stats["max_ulp"], np.unravel_index(np.argmax(d), d.shape))
        assert np.all(g[zero] == 0), "%s: masked output not +0" % what
    return stats
