"""Edge cases on the GPU: strides and guard zones, in place, unaligned
pointers, degenerate rows, empty inputs, streams, the host-buffer entry
point, the bounded-wait self-test, and calls that must launch nothing."""
import numpy as np
import pytest

import row_wise_softmax_gb300 as rws
import workloads as wl
from tests import parity

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

PATHS = [rws.PATH_WARP, rws.PATH_CTA, rws.PATH_CLUSTER, rws.PATH_TWOPASS]
GUARD = 1024            # elements of sentinel before and after every output


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rws.build()
    rws.lib()


def sentinel_run(w: wl.Workload, path):
    """Run into an output surrounded by guard zones, gaps filled with a sentinel."""
    x = parity.device_input(w)
    dt = parity.torch_dtype(w.dtype)
    full = torch.full((GUARD + w.out_elems + GUARD,), 7.0, dtype=dt, device="cuda")
    before = full.clone()
    y = full[GUARD:GUARD + w.out_elems]
    st = rws.softmax_rows_ptr(x.data_ptr(), y.data_ptr(), w.n_rows, w.n_cols, w.in_row_stride,
                              w.out_row_stride, w.dtype, 0, path)
    assert st == rws.OK, rws.status_string(st)
    torch.cuda.synchronize()
    written = torch.zeros_like(full, dtype=torch.bool)
    idx = (torch.arange(w.n_rows, device="cuda")[:, None] * w.out_row_stride
           + torch.arange(w.n_cols, device="cuda")[None, :]).reshape(-1) + GUARD
    written[idx] = True
    iv = torch.int32 if w.dtype == wl.F32 else torch.int16
    untouched = full.view(iv) == before.view(iv)
    assert bool(untouched[~written].all()), "wrote outside the output rows"
    return parity.host_output(y, w)


@pytest.mark.parametrize("dtype", [wl.F32, wl.BF16, wl.F16])
@pytest.mark.parametrize("path", PATHS, ids=lambda p: rws.PATH_NAMES[p])
def test_strided_rows_and_guard_zones(dtype, path):
    for n_cols, ld_in, ld_out in ((100, 128, 130), (1000, 1003, 1000), (600, 600, 777),
                                  (5000, 5008, 5016)):
        if path == rws.PATH_WARP and n_cols > 1024:
            continue
        w = wl.random_rows(9, n_cols, dtype=dtype, seed=n_cols, in_row_stride=ld_in, scale=3.0)
        w.out_row_stride = ld_out
        got = sentinel_run(w, path)
        parity.compare(got, parity.expected(w), dtype, "%s %d/%d/%d" % (
            rws.PATH_NAMES[path], n_cols, ld_in, ld_out))


@pytest.mark.parametrize("path", PATHS, ids=lambda p: rws.PATH_NAMES[p])
def test_in_place(path):
    for dtype in (wl.F32, wl.BF16, wl.F16):
        n_cols = 900 if path == rws.PATH_WARP else 20000
        w = wl.random_rows(11, n_cols, dtype=dtype, seed=3, scale=5.0)
        x = parity.device_input(w)
        st = rws.softmax_rows_ptr(x.data_ptr(), x.data_ptr(), w.n_rows, w.n_cols, w.n_cols,
                                  w.n_cols, dtype, 0, path)
        assert st == rws.OK
        torch.cuda.synchronize()
        parity.compare(parity.host_output(x, w), parity.expected(w), dtype, "in place")


@pytest.mark.parametrize("path", PATHS, ids=lambda p: rws.PATH_NAMES[p])
def test_unaligned_pointers_take_scalar_access(path):
    for dtype in (wl.F32, wl.BF16, wl.F16):
        n_cols = 333 if path == rws.PATH_WARP else 9001
        w = wl.random_rows(5, n_cols, dtype=dtype, seed=9, scale=2.0)
        x_big = parity.device_input(wl.random_rows(1, w.data.size + 1, dtype=dtype, seed=1))
        x = x_big[1:]                                    # 4 or 2 bytes off 16
        x.copy_(parity.device_input(w))
        y_big = torch.empty(w.out_elems + 3, dtype=x.dtype, device="cuda")
        y = y_big[3:]
        p = rws.plan(w.n_rows, w.n_cols, dtype=dtype, path=path, in_ptr=x.data_ptr(),
                     out_ptr=y.data_ptr())
        assert p.bulk_copy == 0 and p.out_vec == 1
        st = rws.softmax_rows_ptr(x.data_ptr(), y.data_ptr(), w.n_rows, w.n_cols, w.n_cols,
                                  w.n_cols, dtype, 0, path)
        assert st == rws.OK
        torch.cuda.synchronize()
        parity.compare(parity.host_output(y, w), parity.expected(w), dtype, "unaligned")


@pytest.mark.parametrize("path", PATHS, ids=lambda p: rws.PATH_NAMES[p])
def test_degenerate_rows(path):
    n_cols = 200 if path == rws.PATH_WARP else 12000
    for dtype in (wl.F32, wl.BF16, wl.F16):
        base = np.random.default_rng(4).standard_normal((6, n_cols)).astype(np.float32)
        base[0, :] = -np.inf                       # all masked: NaN row
        base[1, n_cols // 2] = np.nan              # NaN: NaN row
        base[2, 3] = np.inf                        # +inf: NaN row
        base[3, :] = -np.inf
        base[3, n_cols - 1] = 2.0                  # lone survivor at the tail: exactly 1
        base[4, : n_cols - 5] = -np.inf            # survivors only in the ragged tail
        base[5, :] = 0.25                          # constant
        w = wl.Workload("degenerate", 6, n_cols, n_cols, n_cols, wl.F32, base.reshape(-1), 0)
        if dtype == wl.BF16:
            w = wl.Workload("degenerate", 6, n_cols, n_cols, n_cols, wl.BF16,
                            wl._f32_to_bf16_bits(base.reshape(-1)), 0)
        elif dtype == wl.F16:
            w = wl.Workload("degenerate", 6, n_cols, n_cols, n_cols, wl.F16,
                            wl._f32_to_f16_bits(base.reshape(-1)), 0)
        got = sentinel_run(w, path)
        parity.compare(got, parity.expected(w), dtype, "degenerate")
        one = {wl.F32: 1.0, wl.BF16: 0x3F80, wl.F16: 0x3C00}[dtype]
        assert got[3, n_cols - 1] == one


def test_empty_inputs_are_noops():
    before = rws.launch_count()
    assert rws.softmax_rows_ptr(0, 0, 0, 100, 100, 100, wl.F32) == rws.OK
    assert rws.softmax_rows_ptr(0, 0, 100, 0, 0, 0, wl.F32) == rws.OK
    assert rws.launch_count() == before


def test_invalid_calls_launch_nothing():
    x = torch.zeros(64, device="cuda")
    before = rws.launch_count()
    assert rws.softmax_rows_ptr(x.data_ptr(), x.data_ptr() + 16, 2, 8, 8, 8, wl.F32) == \
        rws.ERR_INVALID_ARG                        # partial overlap
    assert rws.softmax_rows_ptr(x.data_ptr(), x.data_ptr(), 2, 40, 8, 8, wl.F32) == \
        rws.ERR_INVALID_ARG                        # short stride
    assert rws.softmax_rows_ptr(x.data_ptr(), x.data_ptr(), 1, 2000, 2000, 2000, wl.F32,
                                0, rws.PATH_WARP) == rws.ERR_UNSUPPORTED
    assert rws.launch_count() == before


def test_torch_binding_and_streams():
    x = torch.randn(300, 2500, device="cuda") * 3
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y = rws.softmax_rows(x)
    s.synchronize()
    ref = torch.softmax(x.double(), dim=-1)
    assert float((y.double() - ref).abs().max()) <= parity.F32_ABS_TOL
    xb = x.to(torch.bfloat16)
    yb = rws.softmax_rows(xb, stream=s)
    s.synchronize()
    assert yb.dtype == torch.bfloat16 and yb.shape == xb.shape
    xh = x.half()
    yh = rws.softmax_rows(xh)
    torch.cuda.synchronize()
    assert yh.dtype == torch.float16
    assert float((yh.double() - torch.softmax(xh.double(), dim=-1)).abs().max()) <= 1e-3
    with pytest.raises(TypeError):
        rws.softmax_rows(x.double())
    with pytest.raises(ValueError):
        rws.softmax_rows(x.t())                     # column stride != 1
    v = torch.randn(5000, device="cuda")
    assert abs(float(rws.softmax_rows(v).double().sum()) - 1.0) < 1e-5


def test_host_buffer_entry_point():
    w = wl.short_f32(4096)                          # strided host input, dense host output
    h_in = torch.from_numpy(w.data).pin_memory()
    h_out = torch.full((w.out_elems,), -1.0).pin_memory()
    d_in = torch.empty(w.n_rows * w.n_cols, device="cuda")
    d_out = torch.empty_like(d_in)
    s = torch.cuda.Stream()
    st = rws.lib().softmax_rows_host(h_in.data_ptr(), h_out.data_ptr(), w.n_rows, w.n_cols,
                                     w.in_row_stride, w.out_row_stride, w.dtype,
                                     d_in.data_ptr(), d_out.data_ptr(), s.cuda_stream)
    assert st == rws.OK
    s.synchronize()
    got = h_out.numpy().reshape(w.n_rows, w.n_cols)
    parity.compare(got, parity.expected(w), wl.F32, "host entry point")
    # Python wrapper, bf16, in place on the device.
    wb = wl.causal_bf16(512)
    hb = torch.from_numpy(wb.data.view(np.int16)).view(torch.bfloat16).reshape(512, 1024).pin_memory()
    ob = torch.empty_like(hb).pin_memory()
    d = torch.empty(512 * 1024, dtype=torch.bfloat16, device="cuda")
    rws.softmax_rows_host(hb, ob, d, d, stream=s)
    s.synchronize()
    got = ob.view(torch.int16).numpy().view(np.uint16)
    parity.compare(got, parity.expected(wb), wl.BF16, "host entry point bf16")


def test_bounded_wait_self_test_reports_timeout():
    assert rws.device_status(clear=True) == rws.OK
    assert rws.selftest_wait_timeout() == rws.OK
    assert rws.device_status(clear=False) == rws.ERR_DEVICE_TIMEOUT
    assert rws.device_status(clear=True) == rws.ERR_DEVICE_TIMEOUT
    assert rws.device_status(clear=True) == rws.OK
    # The context is still usable.
    w = wl.masked_f32(16)
    x = parity.device_input(w)
    y = parity.empty_output(w)
    assert rws.softmax_rows_ptr(x.data_ptr(), y.data_ptr(), 16, 4096, 4096, 4096, wl.F32) == rws.OK
    torch.cuda.synchronize()
    parity.compare(parity.host_output(y, w), parity.expected(w), wl.F32, "after self-test")


def test_host_direct_mode_pinned_buffers():
    """Direct mode: no device buffers; the kernel reads and writes pinned host rows."""
    for w in (wl.masked_f32(300), wl.short_f32(5000), wl.causal_bf16(700),
              wl.random_rows(3, 100_000, seed=4, scale=3.0)):
        if w.dtype == wl.F32:
            h_in = torch.from_numpy(w.data).pin_memory()
            h_out = torch.full((w.out_elems,), -1.0).pin_memory()
        else:
            h_in = torch.from_numpy(w.data.view(np.int16)).view(torch.bfloat16).pin_memory()
            h_out = torch.zeros(w.out_elems, dtype=torch.bfloat16).pin_memory()
        s = torch.cuda.Stream()
        before = rws.launch_count()
        st = rws.lib().softmax_rows_host(h_in.data_ptr(), h_out.data_ptr(), w.n_rows, w.n_cols,
                                         w.in_row_stride, w.out_row_stride, w.dtype,
                                         None, None, s.cuda_stream)
        assert st == rws.OK, rws.status_string(st)
        s.synchronize()
        assert rws.launch_count() - before == 1
        flat = h_out.view(torch.int16).numpy().view(np.uint16) if w.dtype == wl.BF16 else h_out.numpy()
        idx = np.arange(w.n_rows)[:, None] * w.out_row_stride + np.arange(w.n_cols)[None, :]
        parity.compare(flat[idx], parity.expected(w), w.dtype, "direct " + w.name)


def test_host_direct_mode_rejects_pageable_and_half_staged():
    x = torch.randn(16, 64)                        # pageable: not device-accessible
    y = torch.empty_like(x)
    before = rws.launch_count()
    st = rws.lib().softmax_rows_host(x.data_ptr(), y.data_ptr(), 16, 64, 64, 64, wl.F32,
                                     None, None, None)
    assert st == rws.ERR_INVALID_ARG
    d = torch.empty(16 * 64, device="cuda")
    st = rws.lib().softmax_rows_host(x.data_ptr(), y.data_ptr(), 16, 64, 64, 64, wl.F32,
                                     d.data_ptr(), None, None)
    assert st == rws.ERR_INVALID_ARG
    assert rws.launch_count() == before
    xp, yp = x.pin_memory(), torch.empty_like(x).pin_memory()
    rws.softmax_rows_host(xp, yp)                  # Python wrapper, direct mode
    torch.cuda.synchronize()
    ref = torch.softmax(xp.double(), dim=-1)
    assert float((yp.double() - ref).abs().max()) <= parity.F32_ABS_TOL
