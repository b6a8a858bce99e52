"""Parity of softmax_attention_forward with the oracle's attention in double.

Q, K, V are seeded N(0,1) 16-bit tensors; the oracle takes their exact
values.  Tolerance, from the arithmetic of the kernel: the scores, softmax and
accumulators are fp32 (errors near 2^-20 relative), the probabilities are
rounded to the operand type before P V (relative error e = 2^-8 for bf16,
2^-11 for fp16, at most half that), and the output is rounded once more:
    |O - O*| <= e * (P* |V|) + e * |O*| + 1e-6,
where P* |V| is the oracle's attention with |V| in place of V.  The
logsumexp is fp32: |lse - lse*| <= 1e-5 * (1 + |lse*|).
"""
import numpy as np
import pytest

import row_wise_softmax_gb300 as rws
import workloads as wl
from oracle import attention as oatt
from tests import parity

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

EPS = {wl.BF16: 2.0 ** -8, wl.F16: 2.0 ** -11}


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rws.build()
    rws.lib()


def run(bh, n_q, n_k, d, dtype, seed, scale=None, causal=False, offset=0, qscale=1.0, impl=0):
    qb, kb, vb = wl.attention_inputs(bh, n_q, n_k, d, dtype, seed, qscale)
    dt = parity.torch_dtype(dtype)
    tq, tk, tv = (torch.from_numpy(a.view(np.int16)).cuda().view(dt) for a in (qb, kb, vb))
    to = torch.full_like(tq, float("nan"))
    lse = torch.full((bh, n_q), 123.0, device="cuda")
    before = rws.launch_count()
    st = rws.attention_forward_ptr(tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), to.data_ptr(),
                                   lse.data_ptr(), bh, n_q, n_k, d, dtype, scale, causal, offset,
                                   impl=impl)
    assert st == rws.OK, rws.status_string(st)
    torch.cuda.synchronize()
    assert rws.launch_count() - before == 1
    dec = (lambda a: parity.decode16(a, dtype))
    return (dec(to.cpu().view(torch.int16).numpy().view(np.uint16)), lse.cpu().numpy(),
            dec(qb), dec(kb), dec(vb))


def check(o, lse, q, k, v, dtype, scale=None, causal=False, offset=0, what=""):
    want = oatt.attention(q, k, v, scale, causal, offset)
    mag = oatt.attention(q, k, np.abs(v), scale, causal, offset)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(o), nan), what
    e = EPS[dtype]
    bound = e * mag + e * np.abs(want) + 1e-6
    err = np.abs(o - want)
    assert np.all(err[~nan] <= bound[~nan]), "%s: worst excess %.3g" % (
        what, float(np.max(np.where(nan, -1, err - bound))))
    lw = oatt.logsumexp(q, k, scale, causal, offset)
    fin = np.isfinite(lw)
    assert np.all(np.isneginf(lse[~fin])), what
    assert np.all(np.abs(lse[fin] - lw[fin]) <= 1e-5 * (1 + np.abs(lw[fin]))), what
    return float(err[~nan].max()) if (~nan).any() else 0.0


CASES = [  # bh, n_q, n_k, d, causal, offset
    (3, 128, 128, 64, False, 0),
    (2, 100, 77, 128, False, 0),
    (2, 130, 130, 64, True, 0),
    (2, 96, 200, 128, True, 104),           # bottom-right aligned: n_k - n_q
    (1, 70, 70, 64, True, -5),              # first queries see nothing: NaN
    (4, 33, 1, 64, False, 0),               # one key
    (1, 1, 300, 128, False, 0),
    (2, 515, 517, 128, True, 2),            # several 256-query CTAs, ragged tails
    (1, 300, 1000, 64, False, 0),
    (2, 50, 0, 64, False, 0),               # no key at all: NaN rows, lse -inf
    (7, 600, 600, 64, True, 0),             # many heads, several query tiles each
    (7, 600, 600, 128, True, 0),
]


IMPLS = [rws.ATT_MMA, rws.ATT_TCGEN05, rws.ATT_TCGEN05_PINGPONG]
IMPL_IDS = ["mma_sync", "tcgen05", "tcgen05_pingpong"]


@pytest.mark.parametrize("impl", IMPLS, ids=IMPL_IDS)
@pytest.mark.parametrize("dtype", [wl.BF16, wl.F16])
def test_attention_cases(dtype, impl):
    for i, (bh, n_q, n_k, d, causal, offset) in enumerate(CASES):
        o, lse, q, k, v = run(bh, n_q, n_k, d, dtype, 40 + i, causal=causal, offset=offset,
                              impl=impl)
        check(o, lse, q, k, v, dtype, None, causal, offset, "case %d" % i)


def test_attention_kernels_agree():
    """The tcgen05 kernels and the mma.sync kernel on the same inputs agree within the
    P-rounding error bound (both are checked against the oracle elsewhere;
    their fp32 sums run in different orders): |a - b| <= 2^-7 (1 + |a|) for
    N(0, 1) values."""
    for causal in (False, True):
        a = run(4, 300, 300, 128, wl.BF16, 71, causal=causal, impl=rws.ATT_MMA)[0]
        for other in (rws.ATT_TCGEN05, rws.ATT_TCGEN05_PINGPONG):
            b = run(4, 300, 300, 128, wl.BF16, 71, causal=causal, impl=other)[0]
            assert np.array_equal(np.isnan(a), np.isnan(b))
            ok = ~np.isnan(a)
            excess = np.abs(a[ok] - b[ok]) - 2.0 ** -7 * (1.0 + np.abs(a[ok]))
            assert np.all(excess <= 0), float(excess.max())
            assert np.mean(a[ok] == b[ok]) > 0.5        # mostly the same bf16 values


@pytest.mark.parametrize("impl", IMPLS, ids=IMPL_IDS)
def test_attention_scale_and_large_scores(impl):
    """An explicit scale, and scores spread over +-100 (queries scaled by 8)."""
    o, lse, q, k, v = run(2, 64, 256, 64, wl.BF16, 9, scale=0.3, qscale=8.0, impl=impl)
    check(o, lse, q, k, v, wl.BF16, 0.3, False, 0, "scaled")


@pytest.mark.parametrize("impl", IMPLS, ids=IMPL_IDS)
def test_attention_full_size_sampled(impl):
    """8 heads x 2048 x 2048, d = 128, causal: sampled query rows of 2 heads."""
    bh, n, d = 8, 2048, 128
    o, lse, q, k, v = run(bh, n, n, d, wl.BF16, 11, causal=True, impl=impl)
    rows = np.random.default_rng(2).choice(n, 64, replace=False)
    for b in (0, 5):
        # Causal rows: each sampled query i sees keys 0..i; compare one at a time.
        for i in rows[:16]:
            oi, li = o[b:b + 1, i:i + 1], lse[b:b + 1, i:i + 1]
            check(oi, li, q[b:b + 1, i:i + 1], k[b:b + 1, :i + 1], v[b:b + 1, :i + 1],
                  wl.BF16, None, False, 0, "head %d query %d" % (b, i))


def test_attention_binding_and_errors():
    q = torch.randn(2, 3, 200, 64, device="cuda", dtype=torch.bfloat16)
    k = torch.randn(2, 3, 150, 64, device="cuda", dtype=torch.bfloat16)
    v = torch.randn(2, 3, 150, 64, device="cuda", dtype=torch.bfloat16)
    o, lse = rws.attention(q, k, v, return_lse=True)
    torch.cuda.synchronize()
    ref = torch.nn.functional.scaled_dot_product_attention(q.double(), k.double(), v.double())
    assert o.shape == q.shape and lse.shape == q.shape[:-1]
    assert float((o.double() - ref).abs().max()) <= 0.02
    before = rws.launch_count()
    assert rws.attention_forward_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), 0,
                                     6, 200, 150, 96, wl.BF16) == rws.ERR_UNSUPPORTED
    assert rws.attention_forward_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), k.data_ptr(), 0,
                                     6, 200, 150, 64, wl.BF16) == rws.ERR_INVALID_ARG
    assert rws.attention_forward_ptr(q.data_ptr() + 2, k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                     0, 6, 200, 150, 64, wl.BF16) == rws.ERR_INVALID_ARG
    assert rws.launch_count() == before
    assert rws.device_status(clear=True) == rws.OK
