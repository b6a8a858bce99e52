"""Parity of the CUDA path with the oracle, through the C ABI.

Full-size workloads (all five, every element) in the launch configuration the
benchmark times (automatic path), and a sweep of small shapes — ragged tails,
several tiles, every path forced — at sizes the oracle finishes in seconds.
"""
import numpy as np
import pytest

import row_wise_softmax_gb300 as rws
import workloads as wl
from tests import parity

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rws.build()
    rws.lib()
    yield
    assert rws.device_status(clear=True) == rws.OK


def run(w: wl.Workload, path=rws.PATH_AUTO, out=None, stream=0):
    x = parity.device_input(w)
    y = parity.empty_output(w) if out is None else out
    st = rws.softmax_rows_ptr(x.data_ptr(), y.data_ptr(), w.n_rows, w.n_cols, w.in_row_stride,
                              w.out_row_stride, w.dtype, stream, path)
    assert st == rws.OK, rws.status_string(st)
    torch.cuda.synchronize()
    return parity.host_output(y, w)


EXPECTED_PATH = {
    "small_f32": rws.PATH_WARP,
    "masked_f32": rws.PATH_CTA,
    "causal_bf16": rws.PATH_WARP,
    "short_f32": rws.PATH_WARP,
    "long_f32": rws.PATH_TWOPASS,
}


@pytest.mark.parametrize("name", wl.NAMES)
def test_full_size_workload(name):
    w = wl.make(name)
    p = rws.plan(w.n_rows, w.n_cols, in_row_stride=w.in_row_stride,
                 out_row_stride=w.out_row_stride, dtype=w.dtype)
    assert p.path == EXPECTED_PATH[name], str(p)
    before = rws.launch_count()
    got = run(w)
    assert rws.launch_count() - before == 1            # one kernel per call
    stats = parity.compare(got, parity.expected(w), w.dtype, name)
    print(name, str(p), stats)


def test_closed_forms_on_gpu():
    # masked_f32's constant row: exactly 2^-12; causal_bf16 row 0: exactly [1, 0, ...].
    w = wl.masked_f32(64)
    got = run(w)
    assert np.all(got[w.const_row] == np.float32(2.0 ** -12))
    wc = wl.causal_bf16(4)
    gb = run(wc)
    assert gb[0, 0] == 0x3F80 and np.all(gb[0, 1:] == 0)
    # long_f32: the +50 spike takes all the mass.
    wlng = wl.long_f32(4)
    gl = run(wlng)
    assert np.all(gl[np.arange(4), wlng.spike_cols] == 1.0)


SWEEP_COLS = [1, 2, 3, 4, 5, 7, 8, 9, 31, 32, 33, 63, 64, 65, 100, 127, 128, 129, 255, 256, 257,
              511, 513, 1000, 1023, 1024, 1025, 2047, 2049, 4095, 4096, 4097, 8191, 16385, 40000]
PATHS = [rws.PATH_WARP, rws.PATH_CTA, rws.PATH_CLUSTER, rws.PATH_TWOPASS]
CTA_CAPACITY_COLS = 32768        # a CTA holds at most 32 elements x 1024 threads


def test_forced_cta_beyond_capacity_is_unsupported():
    with pytest.raises(rws.SoftmaxError) as e:
        rws.plan(2, CTA_CAPACITY_COLS + 4, path=rws.PATH_CTA)
    assert e.value.status == rws.ERR_UNSUPPORTED
    assert rws.plan(2, CTA_CAPACITY_COLS, path=rws.PATH_CTA).path == rws.PATH_CTA


@pytest.mark.parametrize("dtype", [wl.F32, wl.BF16, wl.F16])
@pytest.mark.parametrize("path", PATHS, ids=lambda p: rws.PATH_NAMES[p])
def test_shape_sweep_forced_paths(dtype, path):
    checked = 0
    for i, n_cols in enumerate(SWEEP_COLS):
        if path == rws.PATH_WARP and n_cols > 1024:
            continue
        if path == rws.PATH_CTA and n_cols > CTA_CAPACITY_COLS:
            continue
        for n_rows in (1, 3, 7):
            w = wl.random_rows(n_rows, n_cols, dtype=dtype, seed=1000 + i, scale=4.0)
            got = run(w, path)
            parity.compare(got, parity.expected(w), dtype, "%s %dx%d" % (
                rws.PATH_NAMES[path], n_rows, n_cols))
            checked += 1
    assert checked > 20


@pytest.mark.parametrize("path", PATHS, ids=lambda p: rws.PATH_NAMES[p])
def test_many_rows_per_cta_or_cluster(path):
    # More rows than resident CTAs, so persistent loops take several rows each.
    n_cols = 700 if path == rws.PATH_WARP else 3000
    w = wl.random_rows(5000, n_cols, seed=77, scale=3.0)
    parity.compare(run(w, path), parity.expected(w), wl.F32, rws.PATH_NAMES[path])


def test_twopass_long_row_automatic():
    # Rows beyond 16 slices of 32 KB stream twice.
    w = wl.random_rows(3, 1_600_000, seed=5, scale=2.0)
    p = rws.plan(w.n_rows, w.n_cols)
    assert p.path == rws.PATH_TWOPASS
    parity.compare(run(w), parity.expected(w), wl.F32, "twopass auto")


@pytest.mark.parametrize("dtype", [wl.BF16, wl.F16])
def test_16bit_long_rows_cluster_and_twopass(dtype):
    w = wl.random_rows(6, 30_000, dtype=dtype, seed=8, scale=6.0)       # 60 KB rows
    p = rws.plan(w.n_rows, w.n_cols, dtype=dtype)
    assert p.path == rws.PATH_TWOPASS and p.bulk_copy == 1 and p.cluster == 1
    parity.compare(run(w), parity.expected(w), dtype, "16-bit two-pass, one CTA")
    assert rws.plan(w.n_rows, w.n_cols, dtype=dtype, path=rws.PATH_CLUSTER).cluster == 2
    parity.compare(run(w, rws.PATH_CLUSTER), parity.expected(w), dtype, "16-bit cluster")
    w = wl.random_rows(6, 250_000, dtype=dtype, seed=8, scale=6.0)      # 500 KB rows
    p = rws.plan(w.n_rows, w.n_cols, dtype=dtype)
    assert p.path == rws.PATH_TWOPASS and p.bulk_copy == 1
    parity.compare(run(w), parity.expected(w), dtype, "16-bit two-pass")


def test_full_size_f16_causal():
    """fp16 I/O at the causal workload's size (32768 x 1024, -inf written in)."""
    w = wl.causal_f16()
    p = rws.plan(w.n_rows, w.n_cols, dtype=w.dtype)
    assert p.path == rws.PATH_WARP and p.bulk_copy == 1
    got = run(w)
    stats = parity.compare(got, parity.expected(w), w.dtype, "causal_f16")
    assert np.all(got[0, 1:] == 0) and got[0, 0] == 0x3C00                # exactly [1, 0, ...]
    print("causal_f16", stats)


def test_reduced_workloads_every_path():
    for name, rows in (("small_f32", 32), ("masked_f32", 24), ("causal_bf16", 1100),
                       ("short_f32", 900), ("long_f32", 3)):
        w = wl.make(name, rows)
        want = parity.expected(w)
        for path in PATHS:
            if path == rws.PATH_WARP and w.n_cols > 1024:
                continue
            if path == rws.PATH_CTA and w.n_cols > CTA_CAPACITY_COLS:
                continue
            parity.compare(run(w, path), want, w.dtype, "%s/%s" % (name, rws.PATH_NAMES[path]))


def test_deterministic_run_to_run():
    w = wl.masked_f32(300)
    a, b = run(w), run(w)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    w5 = wl.long_f32(3)
    assert np.array_equal(run(w5).view(np.uint32), run(w5).view(np.uint32))


def _planned(w, plan):
    x = parity.device_input(w)
    y = parity.empty_output(w)
    st = rws.softmax_rows_planned_ptr(x.data_ptr(), y.data_ptr(), w.n_rows, w.n_cols,
                                      w.in_row_stride, w.out_row_stride, w.dtype, plan)
    torch.cuda.synchronize()
    return st, parity.host_output(y, w)


def test_planned_launch_shapes():
    w = wl.masked_f32(300)
    want = parity.expected(w)
    base = rws.plan(w.n_rows, w.n_cols)
    for threads, chunks in ((128, 8), (256, 4), (512, 2), (1024, 1), (1024, 8)):
        for stages in (1, 2, 3, 8):
            q = rws.Plan.from_buffer_copy(base)
            q.threads, q.chunks, q.stages = threads, chunks, stages
            q.smem_bytes = stages * q.slice_cols * 4
            st, got = _planned(w, q)
            assert st == rws.OK, str(q)
            parity.compare(got, want, wl.F32, str(q))
    q = rws.Plan.from_buffer_copy(base)
    q.grid = 7                                    # explicit, non-whole-wave grid still correct
    st, got = _planned(w, q)
    assert st == rws.OK
    parity.compare(got, want, wl.F32, "grid 7")
    w5 = wl.long_f32(5)
    b5 = rws.plan(w5.n_rows, w5.n_cols)
    for cs in (8, 16):
        q = rws.Plan.from_buffer_copy(b5)
        q.path, q.bulk_copy, q.vec, q.out_vec = rws.PATH_CLUSTER, 1, 4, 4
        q.cluster = cs
        q.slice_cols = w5.n_cols // cs
        q.threads = 1024 if cs == 8 else 512
        q.chunks = 8
        q.stages = 1
        q.smem_bytes = q.slice_cols * 4
        st, got = _planned(w5, q)
        assert st == rws.OK, str(q)
        parity.compare(got, parity.expected(w5), wl.F32, str(q))


def test_planned_rejects_unsafe_plans():
    w = wl.masked_f32(8)
    base = rws.plan(w.n_rows, w.n_cols)
    before = rws.launch_count()
    bad = []
    q = rws.Plan.from_buffer_copy(base); q.slice_cols = 2048; bad.append(q)        # row not covered
    q = rws.Plan.from_buffer_copy(base); q.threads = 128; q.chunks = 2; bad.append(q)  # slice > regs
    q = rws.Plan.from_buffer_copy(base); q.stages = 9; q.smem_bytes = 9 * 16384; bad.append(q)
    q = rws.Plan.from_buffer_copy(base); q.smem_bytes = 1024; bad.append(q)        # smem mismatch
    q = rws.Plan.from_buffer_copy(base); q.threads = 96; bad.append(q)
    q = rws.Plan.from_buffer_copy(base); q.path = rws.PATH_WARP; bad.append(q)     # 4096 > 1024
    q = rws.Plan.from_buffer_copy(base); q.dtype = rws.BF16; bad.append(q)
    q = rws.Plan.from_buffer_copy(base); q.cluster = 2; bad.append(q)              # CTA with cluster
    for q in bad:
        st, _ = _planned(w, q)
        assert st == rws.ERR_INVALID_ARG, str(q)
    assert rws.launch_count() == before


def test_plan_describe_matches_plan():
    """softmax_plan_describe is softmax_plan on contiguous aligned rows,
    formatted: the same text as the plan of real device buffers."""
    for name in wl.NAMES:
        w = wl.make(name, n_rows=4)
        n_rows = wl.FULL_ROWS[name]
        want = str(rws.plan(n_rows, w.n_cols, dtype=w.dtype))
        assert rws.plan_describe(n_rows, w.n_cols, w.dtype) == want, name
    before = rws.launch_count()
    with pytest.raises(rws.SoftmaxError):
        rws.plan_describe(4, 4, 9)
    assert rws.launch_count() == before


# Shapes whose automatic grid is several waves of resident CTAs: the CTA path
# (fp32 ten waves capped at 1.5 rows per CTA; 16-bit two waves) and the
# staged tile kernel (four waves from eight tiles per resident CTA).  Every
# row is compared with the oracle.
MULTI_WAVE = [
    (16384, 2048, wl.F32, rws.PATH_CTA),
    (3000, 4100, wl.F32, rws.PATH_CTA),        # fewer rows than 1.5 per CTA of ten waves
    (16384, 4096, wl.BF16, rws.PATH_CTA),
    (65536, 1024, wl.BF16, rws.PATH_WARP),     # 16384 tiles of 4 rows
    (262144, 256, wl.F16, rws.PATH_WARP),      # 16384 tiles of 16 rows
]


@pytest.mark.parametrize("n_rows,n_cols,dtype,path", MULTI_WAVE,
                         ids=["cta_f32_ten_waves", "cta_f32_few_rows", "cta_bf16_two_waves",
                              "tile_bf16_four_waves", "tile_f16_four_waves"])
def test_multi_wave_grids(n_rows, n_cols, dtype, path):
    w = wl.random_rows(n_rows, n_cols, dtype=dtype, seed=n_cols, scale=4.0)
    p = rws.plan(w.n_rows, w.n_cols, dtype=dtype)
    assert p.path == path and p.grid == 0 and p.bulk_copy == 1, str(p)
    before = rws.launch_count()
    got = run(w)
    assert rws.launch_count() - before == 1
    parity.compare(got, parity.expected(w), dtype, "%dx%d %s" % (n_rows, n_cols, str(p)))


# Short rows shared by fewer than 32 lanes, several rows to a warp: every
# group size, ragged row counts (a partly filled last group), degenerate rows,
# and the options build (scale and causal mask from indices).
SUB_WARP = [(1, wl.F32), (3, wl.F32), (8, wl.F32), (16, wl.F32), (60, wl.F32), (64, wl.F32),
            (8, wl.BF16), (24, wl.BF16), (64, wl.BF16), (128, wl.BF16), (16, wl.F16), (96, wl.F16)]


@pytest.mark.parametrize("n_cols,dtype", SUB_WARP, ids=lambda v: str(v))
def test_sub_warp_rows(n_cols, dtype):
    n_rows = 4099
    w = wl.random_rows(n_rows, n_cols, dtype=dtype, seed=n_cols + 40, scale=5.0)
    p = rws.plan(w.n_rows, w.n_cols, dtype=dtype)
    assert p.path == rws.PATH_WARP and p.bulk_copy == 0 and p.lanes_per_row < 32, str(p)
    got = run(w)
    parity.compare(got, parity.expected(w), dtype, "sub-warp %s" % str(p))
    # Degenerate rows: all -inf (NaN row), a NaN, a lone finite value.
    data = w.data.copy()
    neg = 0xFF80 if dtype == wl.BF16 else (0xFC00 if dtype == wl.F16 else None)
    nan = 0x7FC0 if dtype == wl.BF16 else (0x7E00 if dtype == wl.F16 else None)
    rows = data.reshape(n_rows, n_cols)
    if dtype == wl.F32:
        rows[5, :] = -np.inf
        rows[6, 0] = np.nan
        rows[7, :] = -np.inf
        rows[7, n_cols // 2] = 1.0
    else:
        rows[5, :] = neg
        rows[6, 0] = nan
        rows[7, :] = neg
        rows[7, n_cols // 2] = 0x3F80 if dtype == wl.BF16 else 0x3C00
    wd = wl.Workload("degenerate", n_rows, n_cols, n_cols, n_cols, dtype, data, 0)
    got = run(wd)
    parity.compare(got, parity.expected(wd), dtype, "sub-warp degenerate")
    # The options build: scale 1/4 and a causal mask from indices.
    import oracle
    opt = dict(scale=0.25, causal=True, causal_period=97, causal_offset=n_cols // 3)
    x = parity.device_input(w)
    y = parity.empty_output(w)
    st = rws.softmax_rows_ex_ptr(x.data_ptr(), y.data_ptr(), w.n_rows, w.n_cols, w.in_row_stride,
                                 w.out_row_stride, w.dtype, **opt)
    assert st == rws.OK, rws.status_string(st)
    torch.cuda.synchronize()
    want = oracle.softmax_rows(w.data, w.n_rows, w.n_cols, w.in_row_stride, w.dtype, **opt)
    parity.compare(parity.host_output(y, w), want, dtype, "sub-warp options")
