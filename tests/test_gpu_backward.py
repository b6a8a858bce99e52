"""Parity of softmax_backward_rows with the oracle's double-precision backward.

dx_i = y_i (dy_i - sum_j y_j dy_j) per row.  The inputs are the oracle's own
forward outputs (rounded to the dtype) and seeded N(0,1) gradients, at shapes
that take the warp kernel (<= 1024 columns) and the CTA kernel (one pass in
registers up to 8192 columns, two passes beyond), aligned and not.

Tolerance, from the fp32 arithmetic: the dot product d = sum_j y_j dy_j is a
sum of n products in fp32 (per-thread chains of at most 32, then a tree), so
its error is below about 50 * 2^-24 * S with S = sum_j |y_j dy_j|; the
subtraction and the product add two roundings.  Hence
    |dx_i - dx*_i| <= 4e-6 * y_i * (|dy_i| + S)        (fp32 outputs)
plus, for 16-bit outputs, the output rounding: one unit in the last place of
dx*_i in that format (the subnormal spacing below the normal range).
"""
import numpy as np
import pytest

import oracle
import row_wise_softmax_gb300 as rws
import workloads as wl
from tests import parity

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

REL = 4e-6
# Spacing relative to the value's binade, and the subnormal spacing below it.
ULP16 = {wl.BF16: (2.0 ** -7, 2.0 ** -133), wl.F16: (2.0 ** -10, 2.0 ** -24)}


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rws.build()
    rws.lib()


def encode(values: np.ndarray, dtype: int) -> np.ndarray:
    if dtype == wl.F32:
        return values.astype(np.float32)
    return oracle.to_bf16(values) if dtype == wl.BF16 else oracle.to_f16(values)


def decode(buf: np.ndarray, dtype: int) -> np.ndarray:
    return buf.astype(np.float64) if dtype == wl.F32 else parity.decode16(buf, dtype)


def make_inputs(n_rows, n_cols, dtype, seed, ld_y=None, ld_g=None):
    """y: the oracle's softmax of N(0, 3^2) rows, rounded to dtype; dy: N(0,1)."""
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((n_rows, n_cols)) * 3).astype(np.float32)
    y = encode(oracle.softmax_rows(x.reshape(-1), n_rows, n_cols), dtype)
    g = encode(rng.standard_normal((n_rows, n_cols)), dtype)
    out = []
    for a, ld in ((y, ld_y or n_cols), (g, ld_g or n_cols)):
        buf = np.zeros((n_rows, ld), dtype=a.dtype)
        buf[:, :n_cols] = a
        out.append(buf.reshape(-1)[: (n_rows - 1) * ld + n_cols] if n_rows else buf.reshape(-1))
    return out


def to_device(buf: np.ndarray, dtype: int):
    t = torch.from_numpy(buf.view(np.int16) if dtype != wl.F32 else buf).cuda()
    return t if dtype == wl.F32 else t.view(parity.torch_dtype(dtype))


def check(got, y, g, n_rows, n_cols, ld_y, ld_g, dtype, what):
    want = oracle.softmax_backward_rows(y, g, n_rows, n_cols, ld_y, ld_g, dtype=dtype)
    yd = np.stack([decode(y[r * ld_y: r * ld_y + n_cols], dtype) for r in range(n_rows)])
    gd = np.stack([decode(g[r * ld_g: r * ld_g + n_cols], dtype) for r in range(n_rows)])
    s = np.abs(yd * gd).sum(axis=1, keepdims=True)
    bound = REL * yd * (np.abs(gd) + s) + 1e-30
    gv = decode(got, dtype)
    if dtype != wl.F32:
        rel, sub = ULP16[dtype]
        bound = bound + np.maximum(rel * np.exp2(np.floor(np.log2(np.abs(want) + 1e-300))), sub)
    err = np.abs(gv - want)
    assert np.all(err <= bound), "%s: worst excess %.3g at %s" % (
        what, float((err - bound).max()), np.unravel_index(np.argmax(err - bound), err.shape))
    return float(err.max())


SHAPES = [(37, 1), (37, 33), (29, 255), (41, 1024), (23, 1025), (9, 5000), (5, 8192), (4, 8193),
          (3, 40000)]


@pytest.mark.parametrize("dtype", [wl.F32, wl.BF16, wl.F16])
def test_backward_shapes(dtype):
    for i, (n_rows, n_cols) in enumerate(SHAPES):
        y, g = make_inputs(n_rows, n_cols, dtype, seed=300 + i)
        ty, tg = to_device(y, dtype), to_device(g, dtype)
        dx = torch.full((n_rows * n_cols,), float("nan"), dtype=ty.dtype, device="cuda")
        st = rws.softmax_backward_rows_ptr(ty.data_ptr(), tg.data_ptr(), dx.data_ptr(), n_rows,
                                           n_cols, n_cols, n_cols, n_cols, dtype)
        assert st == rws.OK, rws.status_string(st)
        torch.cuda.synchronize()
        got = dx.cpu()
        got = got.numpy() if dtype == wl.F32 else got.view(torch.int16).numpy().view(np.uint16)
        check(got.reshape(n_rows, n_cols), y, g, n_rows, n_cols, n_cols, n_cols, dtype,
              "%dx%d" % (n_rows, n_cols))


@pytest.mark.parametrize("dtype", [wl.F32, wl.BF16])
def test_backward_strided_unaligned_and_in_place(dtype):
    for n_rows, n_cols, ld_y, ld_g in ((7, 300, 301, 303), (5, 3000, 3001, 3000), (3, 9001, 9009, 9003)):
        y, g = make_inputs(n_rows, n_cols, dtype, seed=n_cols, ld_y=ld_y, ld_g=ld_g)
        ty, tg = to_device(y, dtype), to_device(g, dtype)
        # dx written in place over dy (same stride): each element read first.
        st = rws.softmax_backward_rows_ptr(ty.data_ptr(), tg.data_ptr(), tg.data_ptr(), n_rows,
                                           n_cols, ld_y, ld_g, ld_g, dtype)
        assert st == rws.OK, rws.status_string(st)
        torch.cuda.synchronize()
        flat = tg.cpu()
        flat = flat.numpy() if dtype == wl.F32 else flat.view(torch.int16).numpy().view(np.uint16)
        got = np.stack([flat[r * ld_g: r * ld_g + n_cols] for r in range(n_rows)])
        check(got, y, g, n_rows, n_cols, ld_y, ld_g, dtype, "strided %d" % n_cols)


def test_backward_full_size_and_binding():
    """4096 x 4096 fp32 (the CTA kernel, one pass) against the oracle on sampled rows,
    and the torch binding against torch's own backward."""
    n_rows, n_cols = 4096, 4096
    y, g = make_inputs(n_rows, n_cols, wl.F32, seed=77)
    ty = torch.from_numpy(y).cuda().view(n_rows, n_cols)
    tg = torch.from_numpy(g).cuda().view(n_rows, n_cols)
    before = rws.launch_count()
    dx = rws.softmax_backward(ty, tg)
    torch.cuda.synchronize()
    assert rws.launch_count() - before == 1
    rows = np.random.default_rng(5).choice(n_rows, 48, replace=False)
    yr = np.ascontiguousarray(y.reshape(n_rows, n_cols)[rows]).reshape(-1)
    gr = np.ascontiguousarray(g.reshape(n_rows, n_cols)[rows]).reshape(-1)
    check(dx.cpu().numpy()[rows], yr, gr, len(rows), n_cols, n_cols, n_cols, wl.F32, "4096^2")
    ref = torch._softmax_backward_data(tg.double(), ty.double(), -1, torch.float64)
    assert float((dx.double() - ref).abs().max()) <= 1e-6
    before = rws.launch_count()
    st = rws.softmax_backward_rows_ptr(ty.data_ptr(), tg.data_ptr(), ty.data_ptr() + 4, n_rows,
                                       n_cols, n_cols, n_cols, n_cols, wl.F32)
    assert st == rws.ERR_INVALID_ARG                        # dx partially overlaps y
    assert rws.launch_count() == before
