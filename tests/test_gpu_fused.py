"""Parity of the scaled, causally masked softmax (softmax_rows_ex) with the oracle.

The options restate "Triton GPU programming deep dive", section 3.1 (scores
scaled before the softmax) and section 3.3 (a key index past the query index
is -inf): column c of row r takes part iff c <= (r mod period) + offset, and
the masked inputs are never read.  Every path is forced in turn on shapes with
ragged tails; the full-size causal workload checks that the mask computed from
indices gives what the mask written into the input gives (the same zeros, the
other outputs within one bf16 ulp: the options kernels sum in pairs).
"""
import numpy as np
import pytest

import oracle
import row_wise_softmax_gb300 as rws
import workloads as wl
from tests import parity

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

PATHS = [rws.PATH_WARP, rws.PATH_CTA, rws.PATH_CLUSTER, rws.PATH_TWOPASS]

# (scale, period, offset): plain causal; several blocks with a bottom-right
# shift; a negative shift (rows with nothing visible are NaN); scale alone.
OPTION_SETS = [
    (0.125, 0, 0),
    (0.08838834764831845, 16, None),        # offset = n_cols - 16
    (2.0, 5, -2),
    (0.3, None, 0),                          # causal off
]


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rws.build()
    rws.lib()
    yield
    assert rws.device_status(clear=True) == rws.OK


def options(n_cols, scale, period, offset):
    causal = period is not None
    return dict(scale=scale, causal=causal, causal_period=period or 0,
                causal_offset=(n_cols - 16 if offset is None else offset) if causal else 0)


def run_ex(w: wl.Workload, path=rws.PATH_AUTO, x=None, **opt):
    x = parity.device_input(w) if x is None else x
    y = parity.empty_output(w, fill=float("nan"))
    st = rws.softmax_rows_ex_ptr(x.data_ptr(), y.data_ptr(), w.n_rows, w.n_cols, w.in_row_stride,
                                 w.out_row_stride, w.dtype, path=path, **opt)
    assert st == rws.OK, rws.status_string(st)
    torch.cuda.synchronize()
    return parity.host_output(y, w)


def expected_ex(w: wl.Workload, **opt):
    return oracle.softmax_rows(w.data, w.n_rows, w.n_cols, w.in_row_stride, w.dtype, **opt)


def visible(n_rows, n_cols, causal, causal_period, causal_offset, **_):
    if not causal:
        return np.ones((n_rows, n_cols), dtype=bool)
    per = causal_period if causal_period > 0 else n_rows
    last = np.arange(n_rows) % per + causal_offset
    return np.arange(n_cols)[None, :] <= last[:, None]


SHAPES = {
    rws.PATH_WARP: [(37, 1), (37, 33), (29, 255), (41, 1024)],
    rws.PATH_CTA: [(23, 1025), (19, 4097), (9, 20001)],
    rws.PATH_CLUSTER: [(5, 4097), (4, 40000)],
    rws.PATH_TWOPASS: [(5, 4097), (3, 70001)],
}


@pytest.mark.parametrize("dtype", [wl.F32, wl.BF16, wl.F16])
@pytest.mark.parametrize("path", PATHS, ids=lambda p: rws.PATH_NAMES[p])
def test_scaled_causal_forced_paths(dtype, path):
    for i, (n_rows, n_cols) in enumerate(SHAPES[path]):
        w = wl.random_rows(n_rows, n_cols, dtype=dtype, seed=2000 + i, scale=6.0)
        for scale, period, offset in OPTION_SETS:
            opt = options(n_cols, scale, period, offset)
            got = run_ex(w, path, **opt)
            what = "%s %dx%d %s" % (rws.PATH_NAMES[path], n_rows, n_cols, opt)
            parity.compare(got, expected_ex(w, **opt), dtype, what)


@pytest.mark.parametrize("path", PATHS, ids=lambda p: rws.PATH_NAMES[p])
def test_masked_inputs_are_never_read(path):
    n_rows, n_cols = (40, 700) if path == rws.PATH_WARP else (6, 9000)
    opt = dict(scale=0.5, causal=True, causal_period=7, causal_offset=n_cols // 2)
    keep = visible(n_rows, n_cols, **opt)
    for dtype in (wl.F32, wl.BF16):
        w = wl.random_rows(n_rows, n_cols, dtype=dtype, seed=31, scale=3.0)
        clean = run_ex(w, path, **opt)
        junk = w.data.reshape(n_rows, n_cols).copy()
        junk[~keep] = np.nan if dtype == wl.F32 else 0x7FC0          # NaN (bf16: quiet NaN bits)
        wj = wl.Workload("junk", n_rows, n_cols, n_cols, n_cols, dtype,
                         np.ascontiguousarray(junk.reshape(-1)), 31)
        dirty = run_ex(wj, path, **opt)
        assert np.array_equal(clean.view(np.uint8), dirty.view(np.uint8)), rws.PATH_NAMES[path]
        parity.compare(clean, expected_ex(w, **opt), dtype, rws.PATH_NAMES[path])


def test_full_size_causal_mask_from_indices_matches_written_mask():
    """The causal workload (1024 keys, 32 blocks of 1024 queries) with its
    -inf written into the input, against the same scores with the mask from indices."""
    w = wl.make("causal_bf16")
    opt = dict(scale=1.0, causal=True, causal_period=w.n_cols, causal_offset=0)
    x = parity.device_input(w)
    written = parity.empty_output(w)
    st = rws.softmax_rows_ptr(x.data_ptr(), written.data_ptr(), w.n_rows, w.n_cols,
                              w.in_row_stride, w.out_row_stride, w.dtype)
    assert st == rws.OK
    # Replace the written -inf by NaN: the fused call must not read them.
    xn = x.clone()
    keep = torch.from_numpy(visible(w.n_rows, w.n_cols, **opt)).cuda()
    xn.view(w.n_rows, w.n_cols).masked_fill_(~keep, float("nan"))
    before = rws.launch_count()
    fused = run_ex(w, x=xn, **opt)
    assert rws.launch_count() - before == 1
    torch.cuda.synchronize()
    plain = parity.host_output(written, w)
    zero = ~visible(w.n_rows, w.n_cols, **opt)
    assert np.all(fused[zero] == 0) and np.all(plain[zero] == 0)
    d = np.abs(parity.bf16_ordered(fused) - parity.bf16_ordered(plain))
    assert d.max() <= 1, d.max()
    rows = np.random.default_rng(7).choice(w.n_rows, 64, replace=False)
    parity.compare(fused[rows], parity.expected(w, rows), w.dtype, "causal_bf16 fused (rows)")


def test_scale_folds_into_exponent_like_exact_product():
    """scale = 2^-3 on fp32 inputs: same result as softmax of the exactly scaled input."""
    w = wl.random_rows(300, 3000, seed=9, scale=20.0)
    ws = wl.Workload("scaled", w.n_rows, w.n_cols, w.n_cols, w.n_cols, wl.F32,
                     (w.data * np.float32(0.125)).astype(np.float32), 9)
    a = run_ex(w, scale=0.125)
    b = run_ex(ws)
    parity.compare(a, parity.expected(ws), wl.F32, "scale 1/8")
    assert np.max(np.abs(a.astype(np.float64) - b)) <= 2 * parity.F32_ABS_TOL


def test_torch_binding_scale_and_causal():
    g = torch.Generator().manual_seed(3)
    x = (torch.randn(64, 96, generator=g) * 4).cuda()
    y = rws.softmax_rows(x, scale=0.25, causal=True, causal_period=32, causal_offset=10)
    q = torch.arange(64) % 32
    keep = torch.tril(torch.ones(32, 96, dtype=torch.bool), diagonal=10)[q].cuda()
    ref = torch.softmax((x.double() * 0.25).masked_fill(~keep, float("-inf")), dim=-1)
    assert torch.all(y[~keep] == 0)
    assert (y.double() - ref).abs().max().item() <= parity.F32_ABS_TOL
    with pytest.raises(rws.SoftmaxError):
        rws.softmax_rows(x, scale=-1.0)


def test_mask_from_indices_on_a_multi_wave_tile_grid():
    """65536 x 1024 bf16 (four waves of the staged tile kernel): the causal mask
    from indices with a period of 1000 rows (tiles cross period boundaries) and
    an offset that leaves the first rows of each period with no kept column."""
    w = wl.random_rows(65536, 1024, dtype=wl.BF16, seed=21, scale=6.0)
    opt = dict(scale=0.125, causal=True, causal_period=1000, causal_offset=-3)
    got = run_ex(w, **opt)
    zero = ~visible(w.n_rows, w.n_cols, **opt)
    empty = zero.all(axis=1)                                            # rows keeping nothing
    assert empty.sum() == 3 * 66
    parity.compare(got, expected_ex(w, **opt), w.dtype, "mask from indices, four waves")
