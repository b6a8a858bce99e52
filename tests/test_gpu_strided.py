"""Parity of softmax_strided (softmax over strided rows) with the oracle.

Column-wise softmax of row-major R x C matrices (row strides 1, column strides
C): the columns kernel, on one CTA or a cluster of them, aligned and not, for
f32, bf16 and fp16; columns too long for the staged tile and general strides
(the gather kernel); in place; the torch binding.  Tolerances are the
row-wise ones (tests/parity.py).
"""
import numpy as np
import pytest

import oracle
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


def matrix(r, c, dtype, seed, scale=4.0):
    """A dense R x C buffer of the dtype (uint16 bits for 16-bit), N(0, scale^2)."""
    w = wl.random_rows(r, c, dtype=dtype, seed=seed, scale=scale)
    return w.data


def run_strided(buf, dtype, n_rows, n_cols, irs, ics, ors, ocs, out_elems, out=None):
    x = torch.from_numpy(buf if dtype == wl.F32 else buf.view(np.int16)).cuda()
    if dtype != wl.F32:
        x = x.view(parity.torch_dtype(dtype))
    y = torch.full((out_elems,), float("nan"), dtype=x.dtype, device="cuda") if out is None else out
    st = rws.softmax_strided_ptr(x.data_ptr(), y.data_ptr(), n_rows, n_cols, irs, ics, ors, ocs,
                                 dtype)
    assert st == rws.OK, rws.status_string(st)
    torch.cuda.synchronize()
    flat = y.cpu()
    flat = flat.numpy() if dtype == wl.F32 else flat.view(torch.int16).numpy().view(np.uint16)
    idx = np.arange(n_rows)[:, None] * ors + np.arange(n_cols)[None, :] * ocs
    return flat[idx]


# (R, C): R is the softmax length; 4096 -> a cluster of 8, 9000 -> 8 CTAs of
# 1125 rows (f32 tile 144 KB), 20000 -> too long for the tile: gather kernel.
COLUMN_SHAPES = [(1, 40), (1000, 33), (4096, 256), (300, 1000), (5000, 129), (9000, 70),
                 (20000, 48)]


@pytest.mark.parametrize("dtype", [wl.F32, wl.BF16, wl.F16])
def test_column_softmax(dtype):
    for i, (R, C) in enumerate(COLUMN_SHAPES):
        if dtype != wl.F32 and R == 9000:
            R = 12000                      # 16-bit: 8 CTAs of 1500 rows
        buf = matrix(R, C, dtype, seed=500 + i)
        got = run_strided(buf, dtype, C, R, 1, C, 1, C, R * C)
        want = oracle.softmax_strided(buf, C, R, 1, C, dtype)
        parity.compare(got, want, dtype, "columns %dx%d" % (R, C))


# Staged columns kernel (16-byte aligned memory-row pitch): boxes of 128
# memory rows, tiles of 128 bytes of softmax rows.  R (the softmax length)
# covers one partial box, exact boxes, a box plus one, several CTAs of a
# cluster with ragged slices; C covers partial tiles and many tiles.
STAGED_SHAPES = [(1, 32), (127, 36), (128, 64), (129, 96), (1000, 100), (4097, 64),
                 (20000, 48), (300, 4096)]


@pytest.mark.parametrize("dtype", [wl.F32, wl.BF16, wl.F16])
def test_column_softmax_staged(dtype):
    esz = 4 if dtype == wl.F32 else 2
    for i, (R, C) in enumerate(STAGED_SHAPES):
        if (C * esz) % 16:
            C += (16 - C * esz % 16) // esz
        buf = matrix(R, C, dtype, seed=700 + i)
        got = run_strided(buf, dtype, C, R, 1, C, 1, C, R * C)
        want = oracle.softmax_strided(buf, C, R, 1, C, dtype)
        parity.compare(got, want, dtype, "staged columns %dx%d" % (R, C))
    # A padded input pitch (only C of every ld elements are softmax rows) and
    # an output pitch that is odd: element stores instead of pairs.
    R, C, ld = 3000, 40, 48
    buf = matrix(R, ld, dtype, seed=801)
    ocs = C + 1
    got = run_strided(buf, dtype, C, R, 1, ld, 1, ocs, (R - 1) * ocs + C)
    want = oracle.softmax_strided(buf, C, R, 1, ld, dtype)
    parity.compare(got, want, dtype, "staged columns padded in, odd out")


def test_column_softmax_staged_in_place_bf16():
    R, C = 5000, 64
    buf = matrix(R, C, wl.BF16, seed=802)
    x = torch.from_numpy(buf.view(np.int16)).cuda().view(torch.bfloat16)
    st = rws.softmax_strided_ptr(x.data_ptr(), x.data_ptr(), C, R, 1, C, 1, C, wl.BF16)
    assert st == rws.OK
    torch.cuda.synchronize()
    flat = x.cpu().view(torch.int16).numpy().view(np.uint16)
    got = np.ascontiguousarray(flat.reshape(R, C).T)
    parity.compare(got, oracle.softmax_strided(buf, C, R, 1, C, wl.BF16), wl.BF16, "in place")


@pytest.mark.parametrize("dtype", [wl.F32, wl.BF16])
def test_general_strides_gather(dtype):
    # Row stride 3, column stride 7 (rows interleaved); output dense rows.
    n_rows, n_cols = 50, 300
    buf = matrix(1, 3 * (n_rows - 1) + 7 * (n_cols - 1) + 1, dtype, seed=9)
    got = run_strided(buf, dtype, n_rows, n_cols, 3, 7, n_cols, 1, n_rows * n_cols)
    parity.compare(got, oracle.softmax_strided(buf, n_rows, n_cols, 3, 7, dtype), dtype, "gather")
    # Column-wise input, output written column-wise into a padded buffer.
    R, C = 700, 40
    buf = matrix(R, C, dtype, seed=10)
    got = run_strided(buf, dtype, C, R, 1, C, 1, C + 8, (R - 1) * (C + 8) + C)
    parity.compare(got, oracle.softmax_strided(buf, C, R, 1, C, dtype), dtype, "padded out")


def test_in_place_columns_and_errors():
    R, C = 3000, 64
    buf = matrix(R, C, wl.F32, seed=11)
    x = torch.from_numpy(buf).cuda()
    st = rws.softmax_strided_ptr(x.data_ptr(), x.data_ptr(), C, R, 1, C, 1, C, wl.F32)
    assert st == rws.OK
    torch.cuda.synchronize()
    got = x.cpu().numpy().reshape(R, C).T
    parity.compare(np.ascontiguousarray(got), oracle.softmax_strided(buf, C, R, 1, C, wl.F32),
                   wl.F32, "in place")
    before = rws.launch_count()
    y = torch.empty(R * C, device="cuda")
    bad = [
        (x.data_ptr(), y.data_ptr(), C, R, 1, C, 0, 0, wl.F32),            # outputs collide
        (x.data_ptr(), x.data_ptr() + 4, C, R, 1, C, 1, C, wl.F32),        # partial overlap
        (x.data_ptr(), y.data_ptr(), C, R, -1, C, 1, C, wl.F32),           # negative stride
        (x.data_ptr(), y.data_ptr(), C, R, 1, C, 1, C, 7),                 # dtype
    ]
    for args in bad:
        assert rws.softmax_strided_ptr(*args) == rws.ERR_INVALID_ARG, args
    assert rws.launch_count() == before


def test_torch_binding_dim0():
    x = (torch.randn(2048, 96, device="cuda") * 3)
    y = rws.softmax(x, dim=0)
    torch.cuda.synchronize()
    ref = torch.softmax(x.double(), dim=0)
    assert float((y.double() - ref).abs().max()) <= parity.F32_ABS_TOL
    y1 = rws.softmax(x, dim=1)
    assert float((y1.double() - torch.softmax(x.double(), dim=1)).abs().max()) <= parity.F32_ABS_TOL
    xt = x.t()                                  # a transposed view: dim 1 is strided
    assert float((rws.softmax(xt, dim=1).double() - torch.softmax(xt.double(), 1)).abs().max()) \
        <= parity.F32_ABS_TOL
