"""The library's launches inside CUDA graphs.

Every kernel is launched with programmatic dependent launch on the caller's
stream; under stream capture those launches become graph nodes (with their
programmatic edges).  A graph of many softmax calls replays to the same bits
as the calls made one by one, for the row path, the options path, the
backward, the attention forward and the column-wise softmax.
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


def test_graph_of_softmax_calls_replays_exactly():
    ws = [wl.small_f32(128), wl.masked_f32(512), wl.causal_bf16(2048), wl.short_f32(3000),
          wl.long_f32(2)]
    xs = [parity.device_input(w) for w in ws]
    eager = []
    for w, x in zip(ws, xs):
        y = parity.empty_output(w)
        assert rws.softmax_rows_ptr(x.data_ptr(), y.data_ptr(), w.n_rows, w.n_cols,
                                    w.in_row_stride, w.out_row_stride, w.dtype) == rws.OK
        eager.append(y)
    warm = parity.empty_output(ws[2])                          # options build, first call eager
    assert rws.softmax_rows_ex_ptr(xs[2].data_ptr(), warm.data_ptr(), ws[2].n_rows, ws[2].n_cols,
                                   ws[2].in_row_stride, ws[2].out_row_stride, ws[2].dtype,
                                   causal=True, causal_period=ws[2].n_cols) == rws.OK
    torch.cuda.synchronize()
    outs = [torch.zeros_like(y) for y in eager]
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    before = rws.launch_count()
    with torch.cuda.graph(g, stream=s):
        h = torch.cuda.current_stream().cuda_stream
        for rep in range(3):                                   # repeated calls, same buffers
            for w, x, y in zip(ws, xs, outs):
                st = rws.softmax_rows_ptr(x.data_ptr(), y.data_ptr(), w.n_rows, w.n_cols,
                                          w.in_row_stride, w.out_row_stride, w.dtype, h)
                assert st == rws.OK
            st = rws.softmax_rows_ex_ptr(xs[2].data_ptr(), outs[2].data_ptr(), ws[2].n_rows,
                                         ws[2].n_cols, ws[2].in_row_stride,
                                         ws[2].out_row_stride, ws[2].dtype, scale=1.0,
                                         causal=True, causal_period=ws[2].n_cols, stream=h)
            assert st == rws.OK
    assert rws.launch_count() - before == 3 * (len(ws) + 1)     # captured, not run
    for _ in range(4):
        g.replay()
    torch.cuda.synchronize()
    for i, (a, b) in enumerate(zip(eager, outs)):
        if i == 2:                                             # the options build sums in pairs
            d = parity.bf16_ordered(parity.host_output(a, ws[i])) - \
                parity.bf16_ordered(parity.host_output(b, ws[i]))
            assert np.abs(d).max() <= 1
        else:
            assert torch.equal(a.view(torch.int16) if a.dtype != torch.float32 else a,
                               b.view(torch.int16) if b.dtype != torch.float32 else b), i


def test_graph_of_attention_and_backward():
    qb, kb, vb = wl.attention_inputs(2, 300, 300, 128, wl.BF16, 3)
    tq, tk, tv = (torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
                  for a in (qb, kb, vb))
    o_eager = torch.empty_like(tq)
    assert rws.attention_forward_ptr(tq.data_ptr(), tk.data_ptr(), tv.data_ptr(),
                                     o_eager.data_ptr(), 0, 2, 300, 300, 128, wl.BF16,
                                     None, True, 0) == rws.OK
    y, gy = wl.backward_pair(64, 3000)
    ty, tg = torch.from_numpy(y).cuda(), torch.from_numpy(gy).cuda()
    dx_eager = torch.empty_like(ty)
    assert rws.softmax_backward_rows_ptr(ty.data_ptr(), tg.data_ptr(), dx_eager.data_ptr(), 64,
                                         3000, 3000, 3000, 3000, wl.F32) == rws.OK
    torch.cuda.synchronize()
    o, dx = torch.zeros_like(o_eager), torch.zeros_like(dx_eager)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=torch.cuda.Stream()):
        h = torch.cuda.current_stream().cuda_stream
        assert rws.attention_forward_ptr(tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), o.data_ptr(),
                                         0, 2, 300, 300, 128, wl.BF16, None, True, 0,
                                         stream=h) == rws.OK
        assert rws.softmax_backward_rows_ptr(ty.data_ptr(), tg.data_ptr(), dx.data_ptr(), 64,
                                             3000, 3000, 3000, 3000, wl.F32, h) == rws.OK
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), o_eager.view(torch.int16))
    assert torch.equal(dx, dx_eager)


def test_graph_of_column_softmax():
    """softmax_strided down the columns (the tensor-copy kernel, whose tensor
    map is a kernel parameter captured with the launch) and the staged-tile
    kernel (an unaligned memory-row pitch) replay to the eager bits."""
    cases = []
    for R, C, dtype in ((3000, 96, wl.F32), (5000, 64, wl.BF16), (700, 33, wl.F32)):
        w = wl.random_rows(R, C, dtype=dtype, seed=R + C, scale=3.0)
        x = torch.from_numpy(w.data if dtype == wl.F32 else w.data.view(np.int16)).cuda()
        if dtype != wl.F32:
            x = x.view(parity.torch_dtype(dtype))
        cases.append((R, C, dtype, x))
    eager = []
    for R, C, dtype, x in cases:
        y = torch.empty_like(x)
        assert rws.softmax_strided_ptr(x.data_ptr(), y.data_ptr(), C, R, 1, C, 1, C, dtype) == rws.OK
        eager.append(y)
    torch.cuda.synchronize()
    outs = [torch.zeros_like(y) for y in eager]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=torch.cuda.Stream()):
        h = torch.cuda.current_stream().cuda_stream
        for (R, C, dtype, x), y in zip(cases, outs):
            assert rws.softmax_strided_ptr(x.data_ptr(), y.data_ptr(), C, R, 1, C, 1, C, dtype,
                                           h) == rws.OK
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, outs):
        iv = torch.int32 if a.dtype == torch.float32 else torch.int16
        assert torch.equal(a.view(iv), b.view(iv))
