"""The seeded inputs have the structure their recipes state."""
import numpy as np

import workloads as wl


def test_small_f32_shape_and_seed():
    a, b = wl.small_f32(16), wl.small_f32(16)
    assert a.data.dtype == np.float32 and a.data.size == 16 * 1000
    assert np.array_equal(a.data, b.data)                # seeded
    assert abs(float(a.data.std()) - 1.0) < 0.05


def test_masked_f32_structure():
    w = wl.masked_f32(256)
    x = w.data.reshape(256, 4096)
    n_inf = np.isneginf(x).sum(axis=1)
    assert n_inf[w.const_row] == 0 and np.all(x[w.const_row] == 0.5)
    others = np.delete(n_inf, w.const_row)
    assert np.all(others == 41)                          # 1% of 4096, distinct columns
    finite = x[np.isfinite(x)]
    assert 2.8 < float(finite.std()) < 3.2


def test_causal_bf16_mask_pattern():
    w = wl.causal_bf16(2100)
    bits = w.data.reshape(2100, 1024)
    neg_inf = bits == 0xFF80
    r = np.arange(2100)[:, None] % 1024
    c = np.arange(1024)[None, :]
    assert np.array_equal(neg_inf, c > r)
    w2 = wl.causal_bf16(4, row_offset=1023)              # window of later rows
    assert np.array_equal(w2.data.reshape(4, 1024)[0] == 0xFF80, np.zeros(1024, bool))


def test_short_f32_padding_and_range():
    w = wl.short_f32(1000)
    x = w.data.reshape(1000, 128)
    assert w.in_row_stride == 128 and w.out_row_stride == 127
    assert np.all(np.isnan(x[:, 127]))
    v = x[:, :127]
    assert v.min() >= -80 and v.max() <= 80


def test_long_f32_spike():
    w = wl.long_f32(3)
    x = w.data.reshape(3, 262144)
    assert np.all(x[np.arange(3), w.spike_cols] == 50.0)
    assert np.all(np.argmax(x, axis=1) == w.spike_cols)


def test_random_rows_exact_extent():
    w = wl.random_rows(5, 7, in_row_stride=9)
    assert w.data.size == 4 * 9 + 7
    wb = wl.random_rows(3, 4, dtype=wl.BF16)
    assert wb.data.dtype == np.uint16 and wb.data.size == 12
    wh = wl.random_rows(3, 4, dtype=wl.F16)
    assert wh.data.dtype == np.uint16 and wh.data.size == 12


def test_causal_f16_recipe():
    w = wl.causal_f16(2100)
    x = w.data.view(np.float16).reshape(2100, 1024).astype(np.float64)
    r = np.arange(2100)[:, None] % 1024
    c = np.arange(1024)[None, :]
    assert np.all(np.isneginf(x[c > r])) and np.all(np.isfinite(x[c <= r]))
    # Same draws as the bf16 recipe, rounded to binary16 instead of bfloat16.
    b = wl.causal_bf16(2100)
    xb = b.data.view(np.uint16).astype(np.uint32) << 16
    xb = xb.view(np.float32).reshape(2100, 1024).astype(np.float64)
    keep = c <= r
    assert np.max(np.abs(x[keep] - xb[keep]) / (np.abs(xb[keep]) + 1e-3)) < 2 ** -7
