"""The largest sizes the ABI accepts: one row of 2^31 - 1 columns (the n_cols
limit), and more than 2^31 rows.  The outputs are checked against closed
forms of the softmax (no oracle pass over billions of elements): a row of
zeros with one spike of height a has y_spike = e^a / (e^a + n - 1) and every
other y = 1 / (e^a + n - 1); one column gives exactly 1.  Each test holds at
most about 17 GB on the device.
"""
import math

import numpy as np
import pytest

import oracle
import row_wise_softmax_gb300 as rws
import workloads as wl
from tests import parity

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

N_MAX = 0x7FFFFFFF


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rws.build()
    rws.lib()
    yield
    torch.cuda.empty_cache()
    assert rws.device_status(clear=True) == rws.OK


def spike_row(n, dtype, pos, a):
    x = torch.zeros(n, dtype=parity.torch_dtype(dtype), device="cuda")
    x[pos] = a
    return x


@pytest.mark.parametrize("dtype", [wl.F32, wl.BF16])
def test_one_row_of_max_columns(dtype):
    n, a = N_MAX, 10.0
    pos = n - 3                                         # near the end: 64-bit offsets
    x = spike_row(n, dtype, pos, a)
    y = torch.empty_like(x)
    p = rws.plan(1, n, dtype=dtype, in_ptr=x.data_ptr(), out_ptr=y.data_ptr())
    assert p.path == rws.PATH_TWOPASS
    before = rws.launch_count()
    st = rws.softmax_rows_ptr(x.data_ptr(), y.data_ptr(), 1, n, n, n, dtype)
    assert st == rws.OK, rws.status_string(st)
    torch.cuda.synchronize()
    assert rws.launch_count() - before == 1
    z = math.exp(a) + (n - 1)
    want = np.array([math.exp(a) / z, 1.0 / z])
    idx = torch.tensor([pos, 0, 1, n // 2, n - 1], device="cuda")
    got = y[idx].float().cpu().numpy().astype(np.float64)
    if dtype == wl.F32:
        # The row sum adds 2^31 fp32 terms: 2^28 columns per CTA of a cluster
        # of 8, 2^20 per thread of 256, summed 16 at a time into the running
        # l (2^16 sequential additions), then 8 + 3 reduction steps.  The
        # recursive-summation bound (additions x 2^-24) is 2^-8 relative.
        tol = 2.0 ** -8
        assert abs(got[0] - want[0]) <= tol * want[0]
        assert np.all(np.abs(got[1:] - want[1]) <= tol * want[1])
        total = float(y.sum(dtype=torch.float64))
        assert abs(total - 1.0) <= tol
    else:
        # 32 columns a batch: 2^15 additions, within 2^-9 relative, less than
        # half a bf16 ulp, so the rounded results differ by one ulp at most.
        wb = oracle.to_bf16(want)
        gb = y[idx].view(torch.int16).cpu().numpy().view(np.uint16)
        assert abs(int(parity.bf16_ordered(gb[:1])[0]) - int(parity.bf16_ordered(wb[:1])[0])) <= 1
        assert np.all(np.abs(parity.bf16_ordered(gb[1:]) - parity.bf16_ordered(wb[1:2])) <= 1)
    # Every non-spike element equals the others (one value, read back sampled).
    del x
    samples = y[torch.randint(0, n, (4096,), device="cuda")]
    samples = samples[samples != y[pos]]
    assert bool((samples == y[0]).all())
    del y
    torch.cuda.empty_cache()


def test_more_than_2_31_rows_of_one_column():
    n_rows = (1 << 31) + 5
    x = torch.randn(n_rows, device="cuda")
    y = torch.zeros_like(x)
    st = rws.softmax_rows_ptr(x.data_ptr(), y.data_ptr(), n_rows, 1, 1, 1, wl.F32)
    assert st == rws.OK, rws.status_string(st)
    torch.cuda.synchronize()
    assert bool((y == 1.0).all())                       # the softmax of one value is 1
    del x, y
    torch.cuda.empty_cache()


def test_beyond_the_column_limit_is_rejected():
    assert rws.softmax_rows_ptr(1 << 20, 1 << 40, 1, N_MAX + 1, N_MAX + 1, N_MAX + 1,
                                wl.F32) == rws.ERR_INVALID_ARG
