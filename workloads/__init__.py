"""Seeded synthetic inputs for the row-wise softmax workloads.

This module only draws numbers: it holds none of the softmax arithmetic and
imports neither the oracle nor the CUDA library.  Tests, bench.py and the
smoke check all take their inputs from here, so the oracle and the CUDA path
see the same bytes.

Five workloads, named by what they are (rows x cols, dtype):

  small_f32   128 x 1000 fp32, contiguous, N(0, 1)                 seed 1
  masked_f32  4096 x 4096 fp32, contiguous, N(0, 3^2); 41 distinct
              columns per row (1% of 4096, rounded) are -inf; one row
              is constant 0.5 with no -inf                          seed 2
  causal_bf16 32768 x 1024 bf16 in/out, N(0, 1) * 8 rounded to bf16;
              row r keeps columns c <= r mod 1024, the rest are -inf seed 3
  short_f32   262144 x 127 fp32, input row stride 128 (padded), output
              contiguous (stride 127), U[-80, 80]; the padding column
              holds NaN, which a correct kernel never reads         seed 4
  long_f32    256 x 262144 fp32, contiguous, N(0, 1) with one +50.0
              per row at a seeded column                            seed 5

Every generator takes ``n_rows`` so that tests can draw a smaller case of the
same recipe (same columns, strides, distributions and structure).  For the
causal workload the mask pattern depends on the row index, so a reduced case
keeps rows 0..n_rows-1 of the full pattern; ``row_offset`` selects a later
window of rows.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

F32 = 0
BF16 = 1
F16 = 2


@dataclass
class Workload:
    name: str
    n_rows: int
    n_cols: int
    in_row_stride: int
    out_row_stride: int
    dtype: int                 # F32 or BF16
    data: np.ndarray           # flat input buffer: float32, or uint16 bf16 bits
    seed: int

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == F32 else 2

    @property
    def algorithmic_bytes(self) -> int:
        """One read and one write of every element: n_rows*n_cols*(in+out size)."""
        return self.n_rows * self.n_cols * 2 * self.elem_bytes

    @property
    def out_elems(self) -> int:
        if self.n_rows == 0:
            return 0
        return (self.n_rows - 1) * self.out_row_stride + self.n_cols


FULL_ROWS = {
    "small_f32": 128,
    "masked_f32": 4096,
    "causal_bf16": 32768,
    "short_f32": 262144,
    "long_f32": 256,
}
COLS = {
    "small_f32": 1000,
    "masked_f32": 4096,
    "causal_bf16": 1024,
    "short_f32": 127,
    "long_f32": 262144,
}
SEEDS = {"small_f32": 1, "masked_f32": 2, "causal_bf16": 3, "short_f32": 4, "long_f32": 5}
NAMES = tuple(FULL_ROWS)
# Further workloads (not among the five configurations): fp16 I/O at the
# causal size.
EXTRA_NAMES = ("causal_f16",)


def _f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round binary32 values to bf16 (round to nearest even) with torch."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def _f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to binary16 (numpy, ties to even); uint16 bit patterns."""
    with np.errstate(over="ignore"):
        return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def causal_f16(n_rows: int = 32768) -> Workload:
    """The causal workload's recipe (row r keeps columns c <= r mod n_cols, the
    rest -inf) with binary16 values: fp16 I/O at the causal size."""
    n_cols = COLS["causal_bf16"]
    rng = np.random.default_rng(SEEDS["causal_bf16"])
    x = rng.standard_normal((n_rows, n_cols), dtype=np.float32) * np.float32(8.0)
    r = np.arange(n_rows)[:, None] % n_cols
    c = np.arange(n_cols)[None, :]
    x = np.where(c > r, np.float32(-np.inf), x).astype(np.float32)
    return Workload("causal_f16", n_rows, n_cols, n_cols, n_cols, F16,
                    _f32_to_f16_bits(x).reshape(-1), 3)


def small_f32(n_rows: int = 128) -> Workload:
    n_cols = COLS["small_f32"]
    rng = np.random.default_rng(SEEDS["small_f32"])
    x = rng.standard_normal((n_rows, n_cols), dtype=np.float32)
    return Workload("small_f32", n_rows, n_cols, n_cols, n_cols, F32, x.reshape(-1), 1)


def masked_f32(n_rows: int = 4096) -> Workload:
    n_cols = COLS["masked_f32"]
    rng = np.random.default_rng(SEEDS["masked_f32"])
    x = (rng.standard_normal((n_rows, n_cols), dtype=np.float32) * np.float32(3.0))
    n_masked = int(round(0.01 * n_cols))            # 41 of 4096
    # 41 distinct columns per row: the first 41 of a random permutation.
    keys = rng.random((n_rows, n_cols), dtype=np.float32)
    cols = np.argpartition(keys, n_masked, axis=1)[:, :n_masked]
    np.put_along_axis(x, cols, -np.inf, axis=1)
    const_row = int(rng.integers(0, n_rows))
    x[const_row, :] = np.float32(0.5)
    w = Workload("masked_f32", n_rows, n_cols, n_cols, n_cols, F32, x.reshape(-1), 2)
    w.const_row = const_row
    return w


def causal_bf16(n_rows: int = 32768, row_offset: int = 0) -> Workload:
    n_cols = COLS["causal_bf16"]
    rng = np.random.default_rng(SEEDS["causal_bf16"])
    if row_offset:
        rng.standard_normal((row_offset, n_cols), dtype=np.float32)   # skip ahead
    x = rng.standard_normal((n_rows, n_cols), dtype=np.float32) * np.float32(8.0)
    r = (np.arange(n_rows) + row_offset)[:, None] % n_cols
    c = np.arange(n_cols)[None, :]
    x = np.where(c > r, np.float32(-np.inf), x).astype(np.float32)
    bits = _f32_to_bf16_bits(x)
    w = Workload("causal_bf16", n_rows, n_cols, n_cols, n_cols, BF16, bits.reshape(-1), 3)
    w.row_offset = row_offset
    return w


def short_f32(n_rows: int = 262144) -> Workload:
    n_cols, stride = COLS["short_f32"], 128
    rng = np.random.default_rng(SEEDS["short_f32"])
    x = np.full((n_rows, stride), np.nan, dtype=np.float32)   # padding column = NaN
    x[:, :n_cols] = rng.uniform(-80.0, 80.0, size=(n_rows, n_cols)).astype(np.float32)
    return Workload("short_f32", n_rows, n_cols, stride, n_cols, F32, x.reshape(-1), 4)


def long_f32(n_rows: int = 256) -> Workload:
    n_cols = COLS["long_f32"]
    rng = np.random.default_rng(SEEDS["long_f32"])
    x = rng.standard_normal((n_rows, n_cols), dtype=np.float32)
    spikes = rng.integers(0, n_cols, size=n_rows)
    x[np.arange(n_rows), spikes] = np.float32(50.0)
    w = Workload("long_f32", n_rows, n_cols, n_cols, n_cols, F32, x.reshape(-1), 5)
    w.spike_cols = spikes
    return w


GENERATORS = {
    "small_f32": small_f32,
    "masked_f32": masked_f32,
    "causal_bf16": causal_bf16,
    "short_f32": short_f32,
    "long_f32": long_f32,
    "causal_f16": causal_f16,
}


def make(name: str, n_rows: int | None = None) -> Workload:
    """The named workload at full size, or its first ``n_rows`` rows' recipe."""
    gen = GENERATORS[name]
    return gen() if n_rows is None else gen(n_rows)


def random_rows(n_rows: int, n_cols: int, dtype: int = F32, seed: int = 0,
                in_row_stride: int | None = None, scale: float = 1.0,
                pad_value: float = np.nan) -> Workload:
    """Generic N(0, scale^2) rows for shape sweeps; padding holds ``pad_value``."""
    stride = n_cols if in_row_stride is None else in_row_stride
    rng = np.random.default_rng(seed)
    x = np.full((max(n_rows, 0), max(stride, 0)), pad_value, dtype=np.float32)
    if n_rows > 0 and n_cols > 0:
        x[:, :n_cols] = rng.standard_normal((n_rows, n_cols), dtype=np.float32) * np.float32(scale)
    flat = x.reshape(-1)
    if n_rows > 0:
        flat = flat[: (n_rows - 1) * stride + n_cols]        # exact strided extent
    if dtype == BF16:
        flat = _f32_to_bf16_bits(flat)
    elif dtype == F16:
        flat = _f32_to_f16_bits(flat)
    return Workload("random", n_rows, n_cols, stride, n_cols, dtype, np.ascontiguousarray(flat), seed)


def backward_pair(n_rows: int = 4096, n_cols: int = 4096, dtype: int = F32, seed: int = 6):
    """Inputs of the softmax backward at a given size: y ~ U[0, 2/n_cols) per
    element (rows of probabilities in scale, without being a softmax output)
    and dy ~ N(0, 1); flat, dense buffers of the dtype (uint16 bits for 16-bit)."""
    rng = np.random.default_rng(seed)
    y = (rng.random((n_rows, n_cols), dtype=np.float32) * np.float32(2.0 / n_cols)).reshape(-1)
    g = rng.standard_normal(n_rows * n_cols, dtype=np.float32)
    if dtype == BF16:
        return _f32_to_bf16_bits(y), _f32_to_bf16_bits(g)
    if dtype == F16:
        return _f32_to_f16_bits(y), _f32_to_f16_bits(g)
    return y, g


def attention_inputs(bh: int, n_q: int, n_k: int, d: int, dtype: int = BF16, seed: int = 7,
                     scale: float = 1.0):
    """Q [bh, n_q, d], K and V [bh, n_k, d] with N(0, scale^2) entries, as
    16-bit bit patterns (uint16) of the dtype."""
    rng = np.random.default_rng(seed)
    out = []
    for n in (n_q, n_k, n_k):
        x = (rng.standard_normal((bh, n, d), dtype=np.float32) * np.float32(scale)).reshape(-1)
        bits = _f32_to_bf16_bits(x) if dtype == BF16 else _f32_to_f16_bits(x)
        out.append(np.ascontiguousarray(bits).reshape(bh, n, d))
    return out
