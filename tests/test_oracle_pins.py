"""Pins for the oracle: checks against things other than the oracle itself.

Each test fixes the oracle to a closed form, an invariant, a high-precision
brute force (mpmath), a library routine (torch CPU in double), or the pages'
worked example, so that a dropped term, a wrong sign or index, or a wrong
stride in oracle/softmax_oracle.c fails at least one of them.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import BF16, F16, F32

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- bf16 codec

def test_bf16_decode_exhaustive(oracle_lib):
    torch = pytest.importorskip("torch")
    bits = np.arange(1 << 16, dtype=np.uint16)
    got = oracle_lib.bf16_to_double(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def _positive_bf16_table():
    """Exact values of all finite non-negative bf16 patterns, ascending."""
    pats = np.arange(0, 0x7F80, dtype=np.uint32)
    f32 = (pats << 16).astype(np.uint32).view(np.float32)
    return pats, [Fraction(float(v)) for v in f32]


_TABLE = None


def _nearest_even_bf16(v: float) -> int:
    """Brute-force RNE: bracket |v| among all bf16 values with exact fractions."""
    global _TABLE
    if _TABLE is None:
        _TABLE = _positive_bf16_table()
    pats, vals = _TABLE
    if math.isnan(v):
        return 0x7FC0 | (0x8000 if math.copysign(1.0, v) < 0 else 0)
    sign = 0x8000 if math.copysign(1.0, v) < 0 else 0
    a = Fraction(abs(v)) if math.isfinite(v) else None
    top = vals[-1]
    next_binade = Fraction(2) ** 128
    if a is None or a >= (top + next_binade) / 2:
        return sign | 0x7F80
    lo, hi = 0, len(vals) - 1
    if a >= top:
        return sign | int(pats[-1])
    while hi - lo > 1:                      # vals[lo] <= a < vals[hi]
        mid = (lo + hi) // 2
        if vals[mid] <= a:
            lo = mid
        else:
            hi = mid
    dlo, dhi = a - vals[lo], vals[hi] - a
    if dlo < dhi:
        pick = lo
    elif dhi < dlo:
        pick = hi
    else:
        pick = lo if (int(pats[lo]) & 1) == 0 else hi
    return sign | int(pats[pick])


def test_bf16_round_bruteforce(oracle_lib):
    rng = np.random.default_rng(11)
    vals = list(rng.standard_normal(400) * np.exp2(rng.integers(-140, 130, 400)))
    # Exact ties between neighbouring bf16 values, and their double neighbours.
    for p in list(rng.integers(0, 0x7F7F, 200)) + [0, 1, 0x7F, 0x80, 0x7F7E]:
        a = float(((np.uint32(p) << 16).astype(np.uint32)).view(np.float32))
        b = float(((np.uint32(p + 1) << 16).astype(np.uint32)).view(np.float32))
        mid = (a + b) / 2.0                 # exact in double
        vals += [mid, np.nextafter(mid, 0.0), np.nextafter(mid, np.inf), -mid]
    top = float(((np.uint32(0x7F7F) << 16).astype(np.uint32)).view(np.float32))
    over = (top + 2.0 ** 128) / 2.0
    vals += [0.0, -0.0, np.inf, -np.inf, top, over, np.nextafter(over, 0.0), 1e-300,
             2.0 ** -134, np.nextafter(2.0 ** -134, 1.0), 2.0 ** -133, 1.0, 1.0 / 3.0]
    vals = np.array(vals, dtype=np.float64)
    got = oracle_lib.to_bf16(vals)
    want = np.array([_nearest_even_bf16(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, want), vals[got != want][:5]
    assert oracle_lib.to_bf16(np.array([np.nan]))[0] & 0x7FFF == 0x7FC0


# ---------------------------------------------------------------- fp16 codec

def test_f16_decode_exhaustive(oracle_lib):
    bits = np.arange(1 << 16, dtype=np.uint16)
    got = oracle_lib.f16_to_double(bits)
    ref = bits.view(np.float16).astype(np.float64)          # numpy's binary16
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))
    assert got[0x0001] == 2.0 ** -24 and got[0x0400] == 2.0 ** -14 and got[0x7BFF] == 65504.0


_F16_TABLE = None


def _nearest_even_f16(v: float) -> int:
    """Brute-force RNE among all binary16 values, with exact fractions."""
    global _F16_TABLE
    if _F16_TABLE is None:      # every finite non-negative pattern, from its definition
        _F16_TABLE = [Fraction(m, 1 << 24) if (b >> 10) == 0 else
                      Fraction(1024 + m) * Fraction(2) ** ((b >> 10) - 25)
                      for b in range(0x7C00) for m in [b & 0x3FF]]
    vals = _F16_TABLE
    if math.isnan(v):
        return 0x7E00 | (0x8000 if math.copysign(1.0, v) < 0 else 0)
    sign = 0x8000 if math.copysign(1.0, v) < 0 else 0
    if not math.isfinite(v) or abs(v) >= 65520.0:
        return sign | 0x7C00
    a = Fraction(abs(v))
    if a >= vals[-1]:
        return sign | (len(vals) - 1)
    lo, hi = 0, len(vals) - 1
    while hi - lo > 1:                      # vals[lo] <= a < vals[hi]
        mid = (lo + hi) // 2
        if vals[mid] <= a:
            lo = mid
        else:
            hi = mid
    dlo, dhi = a - vals[lo], vals[hi] - a
    pick = lo if dlo < dhi else hi if dhi < dlo else (lo if lo % 2 == 0 else hi)
    return sign | pick


def test_f16_round_bruteforce(oracle_lib):
    rng = np.random.default_rng(12)
    vals = list(rng.standard_normal(60) * np.exp2(rng.integers(-26, 16, 60)))
    for p in list(rng.integers(0, 0x7BFE, 40)) + [0, 1, 0x3FF, 0x400, 0x7BFE]:
        a = float(np.uint16(p).view(np.float16))
        b = float(np.uint16(p + 1).view(np.float16))
        mid = (a + b) / 2.0                 # exact in double
        vals += [mid, np.nextafter(mid, 0.0), np.nextafter(mid, np.inf), -mid]
    vals += [0.0, -0.0, np.inf, -np.inf, 65504.0, 65519.99, 65520.0, 2.0 ** -25,
             3 * 2.0 ** -25, 2.0 ** -26, 1.0, 1.0 / 3.0, 1e-300]
    vals = np.array(vals, dtype=np.float64)
    got = oracle_lib.to_f16(vals)
    want = np.array([_nearest_even_f16(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, want), vals[got != want][:5]
    # And numpy's own double -> binary16 conversion on a wide random sample.
    x = rng.standard_normal(20000) * np.exp2(rng.uniform(-28, 16.5, 20000))
    with np.errstate(over="ignore"):
        assert np.array_equal(oracle_lib.to_f16(x), x.astype(np.float16).view(np.uint16))


def test_f16_input_matches_torch_double(oracle_lib):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(24)
    xf = (rng.standard_normal((21, 515)) * 6).astype(np.float16)
    xf[3, 7] = -np.inf
    bits = xf.view(np.uint16).reshape(-1)
    y = oracle_lib.softmax_rows(bits, 21, 515, dtype=F16)
    ref = torch.softmax(torch.from_numpy(xf.astype(np.float64)), dim=-1).numpy()
    assert np.all(np.abs(y - ref) <= 1e-14 * ref + 1e-300)


# --------------------------------------------------- closed forms and invariants

def _rows(x):
    x = np.ascontiguousarray(x, dtype=np.float32)
    return x.reshape(-1), x.shape[0], x.shape[1]


def test_constant_row_is_exactly_one_over_n(oracle_lib):
    for n in (1, 7, 1000, 4096):
        buf, r, c = _rows(np.full((2, n), 0.5))
        y = oracle_lib.softmax_rows(buf, r, c)
        assert np.all(y == 1.0 / n)
    buf, r, c = _rows(np.full((1, 4096), -3.25))
    assert np.all(oracle_lib.softmax_rows(buf, r, c) == 2.0 ** -12)


def test_all_but_one_neg_inf_gives_exactly_one(oracle_lib):
    n = 1024
    x = np.full((n, n), -np.inf, dtype=np.float32)
    rng = np.random.default_rng(3)
    keep = rng.integers(0, n, n)
    x[np.arange(n), keep] = rng.standard_normal(n).astype(np.float32) * 8
    y = oracle_lib.softmax_rows(*_rows(x))
    want = np.zeros((n, n))
    want[np.arange(n), keep] = 1.0
    assert np.array_equal(y, want)
    assert not np.any(np.signbit(y))        # zeros are +0


def test_one_hot_spike_matches_logistic_form(oracle_lib):
    rng = np.random.default_rng(5)
    n = 4096
    x = rng.standard_normal((3, n)).astype(np.float32)
    s = rng.integers(0, n, 3)
    x[np.arange(3), s] = 50.0
    y = oracle_lib.softmax_rows(*_rows(x))
    for r in range(3):
        rest = [math.exp(float(x[r, j]) - 50.0) for j in range(n) if j != s[r]]
        ys = 1.0 / (1.0 + math.fsum(rest))
        assert abs(y[r, s[r]] - ys) <= 2e-16
        assert y[r, s[r]] > 1.0 - 1e-15
        j = (s[r] + 1) % n
        assert math.isclose(y[r, j], math.exp(float(x[r, j]) - 50.0) * ys, rel_tol=1e-14)


def test_shift_invariance_exact_shifts(oracle_lib):
    rng = np.random.default_rng(7)
    base = rng.integers(-40, 40, size=(16, 300)).astype(np.float32) / 4   # exact
    y0 = oracle_lib.softmax_rows(*_rows(base))
    for c in (-1000.0, -64.0, 64.0, 1000.0):
        y = oracle_lib.softmax_rows(*_rows(base + np.float32(c)))
        assert np.array_equal(y, y0), c     # x_j - max is exact, so bitwise equal


def test_rows_sum_to_one_and_are_in_range(oracle_lib):
    w = oracle.softmax_rows  # module-level helper also works
    rng = np.random.default_rng(9)
    x = (rng.standard_normal((64, 777)) * 6).astype(np.float32)
    y = w(*_rows(x))
    assert np.all(y >= 0) and np.all(y <= 1)
    assert np.max(np.abs(y.sum(axis=1) - 1.0)) <= 777 * 2.0 ** -52


def test_row_permutation_permutes_output(oracle_lib):
    rng = np.random.default_rng(13)
    x = rng.standard_normal((50, 129)).astype(np.float32)
    p = rng.permutation(50)
    y = oracle_lib.softmax_rows(*_rows(x))
    yp = oracle_lib.softmax_rows(*_rows(x[p]))
    assert np.array_equal(yp, y[p])


def test_two_element_closed_form(oracle_lib):
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    rng = np.random.default_rng(17)
    x = (rng.standard_normal((200, 2)) * 10).astype(np.float32)
    y = oracle_lib.softmax_rows(*_rows(x))
    for r in range(200):
        a, b = mpmath.mpf(float(x[r, 0])), mpmath.mpf(float(x[r, 1]))
        y0 = 1 / (1 + mpmath.exp(b - a))
        assert abs(y[r, 0] - float(y0)) <= 4e-16 * max(float(y0), 1e-300) + 1e-300
        assert abs(y[r, 1] - float(1 - y0)) <= 4e-16 * max(float(1 - y0), 1e-300) + 1e-300


def test_bruteforce_high_precision_tiny_rows(oracle_lib):
    """Unshifted exp(x_j) / sum exp(x_k) at 50 digits, on rows of 1..9 values."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    rng = np.random.default_rng(19)
    for n in range(1, 10):
        x = (rng.standard_normal((20, n)) * 5).astype(np.float32)
        if n > 2:
            x[::3, 0] = -np.inf                       # some masked entries
        y = oracle_lib.softmax_rows(*_rows(x))
        for r in range(20):
            ex = [mpmath.exp(mpmath.mpf(float(v))) if np.isfinite(v) else mpmath.mpf(0)
                  for v in x[r]]
            tot = mpmath.fsum(ex)
            for j in range(n):
                want = float(ex[j] / tot)
                assert abs(y[r, j] - want) <= (n + 2) * 2.0 ** -53 * want + 1e-300, (n, r, j)


def test_bf16_input_matches_torch_double(oracle_lib):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(23)
    xf = (rng.standard_normal((33, 1024)) * 8).astype(np.float32)
    xf[np.arange(33)[:, None] < np.arange(1024)[None, :] - 500] = -np.inf
    xb = torch.from_numpy(xf).to(torch.bfloat16)
    bits = xb.view(torch.int16).numpy().view(np.uint16)
    y = oracle_lib.softmax_rows(bits.reshape(-1), 33, 1024, dtype=BF16)
    ref = torch.softmax(xb.to(torch.float64), dim=-1).numpy()
    # Two double implementations differ by a few ulp (summation order).
    assert np.all(np.abs(y - ref) <= 1e-14 * ref + 1e-300)


def test_f32_matches_torch_double(oracle_lib):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(29)
    x = (rng.standard_normal((40, 333)) * 3).astype(np.float32)
    x[rng.random(x.shape) < 0.05] = -np.inf
    x[5, :] = 0.5
    y = oracle_lib.softmax_rows(*_rows(x))
    ref = torch.softmax(torch.from_numpy(x).double(), dim=-1).numpy()
    assert np.all(np.abs(y - ref) <= 1e-14 * ref + 1e-300)


def test_degenerate_rows_are_nan(oracle_lib):
    torch = pytest.importorskip("torch")
    x = np.zeros((4, 8), dtype=np.float32)
    x[0, :] = -np.inf                      # all masked
    x[1, 3] = np.nan                       # one NaN
    x[2, 5] = np.inf                       # one +inf
    x[3, :] = np.arange(8)                 # ordinary row
    y = oracle_lib.softmax_rows(*_rows(x))
    assert np.all(np.isnan(y[:3]))
    assert np.all(np.isfinite(y[3]))
    ref = torch.softmax(torch.from_numpy(x).double(), dim=-1).numpy()
    assert np.array_equal(np.isnan(ref), np.isnan(y))


def test_padded_input_stride_never_reads_padding(oracle_lib):
    rng = np.random.default_rng(31)
    dense = rng.standard_normal((9, 127)).astype(np.float32)
    for pad in (np.nan, np.inf, 1e30):
        buf = np.full((9, 128), pad, dtype=np.float32)
        buf[:, :127] = dense
        flat = buf.reshape(-1)[: 8 * 128 + 127]       # exact extent: no last pad
        y = oracle_lib.softmax_rows(flat, 9, 127, in_row_stride=128)
        assert np.array_equal(y, oracle_lib.softmax_rows(dense.reshape(-1), 9, 127))


def test_bad_arguments_rejected(oracle_lib):
    with pytest.raises(ValueError):
        oracle_lib.softmax_rows(np.zeros(10, np.float32), 2, 6)     # buffer too small
    with pytest.raises(TypeError):
        oracle_lib.softmax_rows(np.zeros(10, np.float64), 1, 10)
    assert oracle_lib.softmax_rows(np.zeros(0, np.float32), 0, 5).shape == (0, 5)


# ----------------------------------------------------------- online recurrence

@pytest.mark.parametrize("tile", [1, 3, 4, 64, 1000])
def test_online_recurrence_equals_definition(oracle_lib, tile):
    rng = np.random.default_rng(37)
    x = (rng.standard_normal((24, 700)) * 6).astype(np.float32)
    x[:8][np.arange(8)[:, None] * 90 < np.arange(700)[None, :]] = -np.inf   # causal-like tails
    x[8:16, :200] = -np.inf                                                  # leading -inf tiles
    x[16, :] = 0.5
    plain = oracle_lib.softmax_rows(*_rows(x))
    online = oracle_lib.softmax_rows(*_rows(x), tile=tile)
    # Same result up to rounding order: each rescale adds a few ulp.
    assert np.all(np.abs(online - plain) <= 1e-14 * plain + 1e-300)
    assert np.array_equal(online == 0, plain == 0)


def test_online_recurrence_degenerate_rows(oracle_lib):
    x = np.full((3, 12), -np.inf, dtype=np.float32)
    x[1, 2] = np.nan                       # NaN inside a leading all -inf tile
    x[2, 9] = 1.0                          # survivor in the last tile
    y = oracle_lib.softmax_rows(*_rows(x), tile=4)
    assert np.all(np.isnan(y[0])) and np.all(np.isnan(y[1]))
    assert y[2, 9] == 1.0 and np.count_nonzero(y[2]) == 1


# ----------------------------------------------------- the pages' worked example

def _read_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, *v = line.split()
                out[k] = [float(t) for t in v]
    return out


def test_level2_tiled_row_sum_worked_example(oracle_lib):
    g = _read_golden("level2_row_sum.txt")
    block = int(g["block"][0])
    rng = np.random.default_rng(41)
    row = np.concatenate([g["row_prefix"], rng.integers(0, 10, 6)]).astype(np.float64)
    assert row.size == 12                      # the page's row length
    _, acc0 = oracle_lib.tiled_row_sum(row, block, snapshot_tiles=1)
    assert list(acc0) == g["after_tile0"]
    _, acc1 = oracle_lib.tiled_row_sum(row, block, snapshot_tiles=2)
    assert acc1[0] == g["after_tile1_lane0"][0] and acc1[1] == g["after_tile1_lane1"][0]
    total, acc3 = oracle_lib.tiled_row_sum(row, block, snapshot_tiles=99)
    assert total == math.fsum(row) and math.fsum(acc3) == total
    # A ragged row: masked lanes add nothing.
    total, _ = oracle_lib.tiled_row_sum(row[:10], block, snapshot_tiles=99)
    assert total == math.fsum(row[:10])


# ------------------------------------------------ scaled, causally masked rows
# "Triton GPU programming deep dive", section 3.1 (scores scaled before the
# softmax) and section 3.3 (scores whose key index exceeds the query index are
# -inf).  Row r is query (r mod period); column c takes part iff
# c <= (r mod period) + offset.

def test_causal_constant_rows_closed_form(oracle_lib):
    """Equal inputs: row r is exactly 1/(visible columns) on its visible part, 0 after it."""
    n_rows, n_cols = 11, 8
    x = np.full((n_rows, n_cols), 0.75, dtype=np.float32)
    for period, offset in ((0, 0), (4, 0), (3, 2), (5, -1)):
        y = oracle_lib.softmax_rows(*_rows(x), scale=1.5, causal=True,
                                    causal_period=period, causal_offset=offset)
        per = period if period > 0 else n_rows
        for r in range(n_rows):
            vis = min(max(r % per + offset + 1, 0), n_cols)
            if vis == 0:
                assert np.all(np.isnan(y[r])), (period, offset, r)
                continue
            assert np.all(y[r, :vis] == 1.0 / vis), (period, offset, r)
            assert np.all(y[r, vis:] == 0.0) and not np.any(np.signbit(y[r, vis:]))


def _torch_causal(torch, xd, scale, period, offset):
    """torch CPU double: scale, then -inf outside torch.tril(diagonal=offset) of each block."""
    n_rows, n_cols = xd.shape
    per = period if period > 0 else n_rows
    q = torch.arange(n_rows) % per
    keep = torch.tril(torch.ones(per, n_cols, dtype=torch.bool), diagonal=offset)[q]
    z = (xd * scale).masked_fill(~keep, float("-inf"))
    return torch.softmax(z, dim=-1).numpy()


def test_causal_scaled_matches_torch_tril_mask(oracle_lib):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(37)
    n_rows, n_cols = 23, 70
    x = (rng.standard_normal((n_rows, n_cols)) * 4).astype(np.float32)
    xb = torch.from_numpy(x).to(torch.bfloat16)
    bits = xb.view(torch.int16).numpy().view(np.uint16).reshape(-1)
    for scale, period, offset in ((0.125, 0, 0), (1 / 3, 7, 0), (2.5, 9, 40), (0.7, 0, -4),
                                  (1.0, 6, 100)):
        s32 = float(np.float32(scale))
        for dtype, buf, xd in ((F32, x.reshape(-1), torch.from_numpy(x).double()),
                               (BF16, bits, xb.double())):
            y = oracle_lib.softmax_rows(buf, n_rows, n_cols, dtype=dtype, scale=scale,
                                        causal=True, causal_period=period, causal_offset=offset)
            ref = _torch_causal(torch, xd, s32, period, offset)
            assert np.array_equal(np.isnan(y), np.isnan(ref)), (scale, period, offset, dtype)
            ok = ~np.isnan(ref)
            assert np.all(np.abs(y[ok] - ref[ok]) <= 1e-14 * ref[ok] + 1e-300), (scale, dtype)


def test_scale_two_element_closed_form(oracle_lib):
    """softmax(s * [a, b]) = [1/(1+exp(s(b-a))), ...] at 40 digits, s as a float32."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    rng = np.random.default_rng(41)
    x = (rng.standard_normal((64, 2)) * 6).astype(np.float32)
    for scale in (0.125, 0.0883883476, 3.0):
        s = mpmath.mpf(float(np.float32(scale)))
        y = oracle_lib.softmax_rows(*_rows(x), scale=scale)
        for r in range(64):
            a, b = mpmath.mpf(float(x[r, 0])), mpmath.mpf(float(x[r, 1]))
            y0 = float(1 / (1 + mpmath.exp(s * (b - a))))
            assert abs(y[r, 0] - y0) <= 4e-16 * y0 + 1e-300, (scale, r)


def test_power_of_two_scale_equals_rescaled_input(oracle_lib):
    rng = np.random.default_rng(43)
    x = (rng.standard_normal((12, 50)) * 3).astype(np.float32)
    for s in (0.25, 2.0, 8.0):
        y = oracle_lib.softmax_rows(*_rows(x), scale=s)
        assert np.array_equal(y, oracle_lib.softmax_rows(*_rows((x * s).astype(np.float32))))


def test_masked_columns_are_never_read(oracle_lib):
    rng = np.random.default_rng(47)
    n_rows, n_cols = 10, 33
    x = rng.standard_normal((n_rows, n_cols)).astype(np.float32)
    keep = np.arange(n_cols)[None, :] <= (np.arange(n_rows)[:, None] % 4) + 3
    y0 = oracle_lib.softmax_rows(*_rows(np.where(keep, x, 0).astype(np.float32)),
                                 causal=True, causal_period=4, causal_offset=3)
    for junk in (np.nan, np.inf, -np.inf, 3e38):
        xj = np.where(keep, x, junk).astype(np.float32)
        y = oracle_lib.softmax_rows(*_rows(xj), causal=True, causal_period=4, causal_offset=3)
        assert np.array_equal(y, y0), junk
    assert np.all(np.isfinite(y0))


@pytest.mark.parametrize("tile", [1, 3, 16])
def test_online_recurrence_causal_equals_definition(oracle_lib, tile):
    rng = np.random.default_rng(53)
    n_rows, n_cols = 17, 45
    x = (rng.standard_normal((n_rows, n_cols)) * 5).astype(np.float32)
    kw = dict(scale=0.3, causal=True, causal_period=6, causal_offset=-2)
    y = oracle_lib.softmax_rows(*_rows(x), **kw)
    yt = oracle_lib.softmax_rows(*_rows(x), tile=tile, **kw)
    assert np.array_equal(np.isnan(y), np.isnan(yt))
    assert np.isnan(y[0]).all() and np.isnan(y[6]).all()       # rows with no visible column
    ok = ~np.isnan(y)
    assert np.all(np.abs(yt[ok] - y[ok]) <= 1e-14 * y[ok] + 1e-300)


# ------------------------------------------------------------ softmax backward
# dx_i = y_i (dy_i - sum_j y_j dy_j): the chain rule through the row softmax.

def test_backward_matches_torch_softmax_backward(oracle_lib):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(61)
    for n_rows, n_cols in ((7, 1), (13, 37), (5, 1000)):
        x = torch.from_numpy(rng.standard_normal((n_rows, n_cols)) * 3)
        y = torch.softmax(x, dim=-1).float()
        dy = torch.from_numpy(rng.standard_normal((n_rows, n_cols))).float()
        got = oracle_lib.softmax_backward_rows(y.numpy().reshape(-1), dy.numpy().reshape(-1),
                                               n_rows, n_cols)
        # torch's own backward of softmax, from the output and the incoming
        # gradient, in double (the same exact y and dy values).
        ref = torch._softmax_backward_data(dy.double(), y.double(), -1, torch.float64).numpy()
        assert np.allclose(got, ref, rtol=1e-12, atol=1e-15)


def test_backward_finite_differences(oracle_lib):
    """The gradient of sum_j dy_j softmax(x)_j by central differences at 40 digits."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    rng = np.random.default_rng(62)
    for n in (2, 3, 6):
        x = [mpmath.mpf(float(v)) for v in rng.standard_normal(n) * 2]
        dy = rng.standard_normal(n).astype(np.float32)

        def loss(xs):
            e = [mpmath.exp(v) for v in xs]
            t = mpmath.fsum(e)
            return mpmath.fsum(float(dy[j]) * e[j] / t for j in range(n))

        e = [mpmath.exp(v) for v in x]
        t = mpmath.fsum(e)
        y = np.array([float(v / t) for v in e], dtype=np.float32)
        got = oracle_lib.softmax_backward_rows(y, dy, 1, n)[0]
        h = mpmath.mpf(10) ** -15
        for i in range(n):
            xp = list(x); xp[i] += h
            xm = list(x); xm[i] -= h
            fd = float((loss(xp) - loss(xm)) / (2 * h))
            assert abs(got[i] - fd) <= 1e-6 * (1 + abs(fd)), (n, i, got[i], fd)


def test_backward_exact_dyadic_rows(oracle_lib):
    """Dyadic y summing to 1 and small-integer dy: every value exact in double."""
    y = np.array([[0.5, 0.25, 0.125, 0.125], [1.0, 0.0, 0.0, 0.0], [0.25] * 4], np.float32)
    dy = np.array([[3, -1, 2, 0], [5, 7, -2, 1], [9, 9, 9, 9]], np.float32)
    got = oracle_lib.softmax_backward_rows(y.reshape(-1), dy.reshape(-1), 3, 4)
    for r in range(3):
        dot = sum(Fraction(float(y[r, j])) * Fraction(float(dy[r, j])) for j in range(4))
        for j in range(4):
            assert got[r, j] == float(Fraction(float(y[r, j])) * (Fraction(float(dy[r, j])) - dot))
        assert sum(Fraction(v) for v in got[r]) == 0
    assert np.all(got[2] == 0.0)                          # constant dy: zero gradient


def test_backward_strides_and_16bit(oracle_lib):
    rng = np.random.default_rng(63)
    y = rng.random((6, 50)).astype(np.float32)
    dy = rng.standard_normal((6, 50)).astype(np.float32)
    dense = oracle_lib.softmax_backward_rows(y.reshape(-1), dy.reshape(-1), 6, 50)
    yp = np.full((6, 64), np.nan, np.float32); yp[:, :50] = y
    gp = np.full((6, 57), np.nan, np.float32); gp[:, :50] = dy
    strided = oracle_lib.softmax_backward_rows(yp.reshape(-1)[:5 * 64 + 50],
                                               gp.reshape(-1)[:5 * 57 + 50], 6, 50, 64, 57)
    assert np.array_equal(dense, strided)
    for dtype, enc, dec in ((BF16, oracle_lib.to_bf16, oracle_lib.bf16_to_double),
                            (F16, oracle_lib.to_f16, oracle_lib.f16_to_double)):
        yb, gb = enc(y.astype(np.float64)), enc(dy.astype(np.float64))
        got = oracle_lib.softmax_backward_rows(yb.reshape(-1), gb.reshape(-1), 6, 50, dtype=dtype)
        yd, gd = dec(yb).astype(np.float32), dec(gb).astype(np.float32)    # exact in binary32
        ref = oracle_lib.softmax_backward_rows(yd.reshape(-1), gd.reshape(-1), 6, 50)
        assert np.array_equal(got, ref)


# ------------------------------------------------------ strided (column-wise)

def test_strided_column_softmax_matches_transpose(oracle_lib):
    """Column-wise softmax of a row-major matrix equals the row softmax of its
    transpose (numpy's transpose, copied dense)."""
    rng = np.random.default_rng(71)
    m = (rng.standard_normal((45, 17)) * 4).astype(np.float32)
    m[3, 5] = -np.inf
    cols = oracle_lib.softmax_strided(m.reshape(-1), 17, 45, 1, 17)
    rows_of_t = oracle_lib.softmax_rows(np.ascontiguousarray(m.T).reshape(-1), 17, 45)
    assert np.array_equal(cols, rows_of_t)
    # The unit column stride is the row-wise softmax.
    assert np.array_equal(oracle_lib.softmax_strided(m.reshape(-1), 45, 17, 17, 1),
                          oracle_lib.softmax_rows(m.reshape(-1), 45, 17))


def test_strided_matches_torch_dim0_and_16bit(oracle_lib):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(72)
    m = (rng.standard_normal((300, 40)) * 2).astype(np.float32)
    got = oracle_lib.softmax_strided(m.reshape(-1), 40, 300, 1, 40)
    ref = torch.softmax(torch.from_numpy(m).double(), dim=0).numpy().T
    assert np.all(np.abs(got - ref) <= 1e-14 * ref + 1e-300)
    for dtype, enc in ((BF16, oracle_lib.to_bf16), (F16, oracle_lib.to_f16)):
        b = enc(m.astype(np.float64))
        got = oracle_lib.softmax_strided(b.reshape(-1), 40, 300, 1, 40, dtype=dtype)
        ref = oracle_lib.softmax_rows(np.ascontiguousarray(b.T).reshape(-1), 40, 300, dtype=dtype)
        assert np.array_equal(got, ref)


def test_strided_general_gather(oracle_lib):
    """Row stride 3, column stride 7 over a buffer: each row gathered by index."""
    rng = np.random.default_rng(73)
    buf = rng.standard_normal(3 * 9 + 7 * 10 + 1).astype(np.float32)
    got = oracle_lib.softmax_strided(buf, 10, 11, 3, 7)
    for r in range(10):
        row = np.array([buf[r * 3 + c * 7] for c in range(11)], dtype=np.float32)
        assert np.array_equal(got[r], oracle_lib.softmax_rows(row, 1, 11)[0])
