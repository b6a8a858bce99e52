"""Host-side checks of the C ABI that need no GPU: the library builds, loads
and exports every function include/softmax.h declares; validation; the
row-to-CTA scheduler on a described GB300; a C-only caller."""
import ctypes
import os
import re
import subprocess

import pytest

import row_wise_softmax_gb300 as rws

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "softmax.h")
GB = rws.GB300


@pytest.fixture(scope="module")
def lib():
    rws.build()
    return rws.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[\w\s\*]+?\b(softmax_\w+)\s*\(", text, flags=re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 10, names
    for n in names:
        assert hasattr(lib, n), "missing export " + n
    nm = subprocess.run(["nm", "-D", "--defined-only", rws.library_path()],
                        capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (\w+)", nm))
    assert set(names) <= exported


def test_status_strings(lib):
    assert rws.status_string(rws.OK) == "ok"
    for s in (rws.ERR_INVALID_ARG, rws.ERR_UNSUPPORTED, rws.ERR_CUDA, rws.ERR_DEVICE_TIMEOUT, 99):
        assert isinstance(rws.status_string(s), str) and rws.status_string(s)
    assert rws.abi_version() == 2


def plan(n_rows, n_cols, **kw):
    return rws.plan_for_device(GB, n_rows, n_cols, **kw)


def test_scheduler_paths_for_the_five_workloads(lib):
    p = plan(128, 1000)                                   # fp32 short rows: register kernel
    assert (p.path, p.bulk_copy, p.vec, p.chunks, p.rows_per_warp) == (rws.PATH_WARP, 0, 4, 8, 1)
    p = plan(4096, 4096)
    assert (p.path, p.cluster, p.bulk_copy, p.out_vec) == (rws.PATH_CTA, 1, 1, 4)
    assert (p.threads, p.chunks, p.stages, p.smem_bytes, p.grid) == (128, 8, 2, 32768, 0)
    p = plan(32768, 1024, dtype=rws.BF16)                 # bf16 short rows: staged tiles
    assert (p.path, p.bulk_copy, p.vec, p.chunks, p.rows_per_warp) == (rws.PATH_WARP, 1, 8, 4, 1)
    assert (p.stages, p.smem_bytes) == (2, 16384)
    p = plan(32768, 2048, dtype=rws.BF16)                 # 4 KB rows: 64-thread CTAs
    assert (p.path, p.threads, p.chunks, p.stages) == (rws.PATH_CTA, 64, 4, 2)
    p = plan(21845, 1536)                                 # 6 KB fp32 rows: 64 x 8 vectors
    assert (p.path, p.threads, p.chunks) == (rws.PATH_CTA, 64, 8)
    p = plan(1 << 20, 16)                                 # short rows: 4 lanes a row
    assert (p.path, p.bulk_copy, p.vec, p.chunks, p.lanes_per_row) == (rws.PATH_WARP, 0, 4, 1, 4)
    p = plan(1 << 20, 64, dtype=rws.BF16)                 # 16-bit too, up to 128 columns
    assert (p.path, p.bulk_copy, p.vec, p.chunks, p.lanes_per_row) == (rws.PATH_WARP, 0, 8, 1, 8)
    p = plan(1 << 20, 200, dtype=rws.BF16)                # longer: the staged tile kernel
    assert (p.path, p.bulk_copy, p.lanes_per_row) == (rws.PATH_WARP, 1, 32)
    p = plan(262144, 127, in_row_stride=128, out_row_stride=127)
    assert (p.path, p.bulk_copy, p.vec, p.chunks, p.rows_per_warp) == (rws.PATH_WARP, 0, 1, 4, 4)
    p = plan(256, 262144)                                 # staged two-pass, 32 KB chunks
    assert (p.path, p.cluster, p.slice_cols, p.threads, p.grid) == (rws.PATH_TWOPASS, 4, 65536, 512, 0)
    assert (p.vec, p.out_vec, p.bulk_copy, p.chunks, p.stages, p.smem_bytes) == (4, 4, 1, 4, 3, 98304)
    p = plan(1024, 65536)                                 # one CTA per row: a 192 KB ring
    assert (p.cluster, p.stages, p.smem_bytes) == (1, 6, 196608)
    p = plan(2730, 12288)                                 # 48 KB rows: 16 KB chunks, 2 CTAs/SM
    assert (p.path, p.cluster, p.threads, p.chunks, p.stages, p.smem_bytes) == (
        rws.PATH_TWOPASS, 1, 256, 4, 6, 98304)
    p = plan(1365, 24576)                                 # 96 KB rows keep 32 KB chunks
    assert (p.path, p.cluster, p.threads, p.stages) == (rws.PATH_TWOPASS, 1, 512, 6)
    p = plan(2048, 65536, dtype=rws.BF16)
    assert (p.path, p.cluster, p.threads, p.stages) == (rws.PATH_TWOPASS, 1, 512, 6)
    p = plan(256, 262144, dtype=rws.BF16)                 # 16-bit: slices up to 1 MB
    assert (p.path, p.cluster, p.threads, p.chunks, p.stages) == (rws.PATH_TWOPASS, 1, 512, 4, 6)
    p = plan(256, 262144, in_ptr=(1 << 20) + 4)           # unaligned: register two-pass
    assert (p.path, p.bulk_copy, p.vec, p.threads) == (rws.PATH_TWOPASS, 0, 1, 512)


def test_scheduler_fp16_follows_bf16(lib):
    """fp16 I/O has bf16's element size, so every shape gets bf16's plan."""
    for shape, kw in (((32768, 1024), {}), ((4096, 4096), {}), ((6, 30000), {}),
                      ((256, 262144), {}), ((64, 1000), {"out_row_stride": 1001}),
                      ((9, 5000), {"in_ptr": (1 << 20) + 2})):
        a = plan(*shape, dtype=rws.BF16, **kw)
        b = plan(*shape, dtype=rws.F16, **kw)
        assert str(a).replace("dtype=bf16", "dtype=f16") == str(b), (shape, str(a), str(b))


def test_scheduler_boundaries(lib):
    assert plan(1, 1024).path == rws.PATH_WARP
    assert plan(1, 1025).path == rws.PATH_CTA
    assert plan(1, 8192).path == rws.PATH_CTA             # 32 KB row
    p = plan(1, 8196)                                      # aligned rows beyond 32 KB: staged two-pass
    assert p.path == rws.PATH_TWOPASS and p.cluster == 1 and p.bulk_copy == 1
    p = plan(1, 8196, in_ptr=(1 << 20) + 4)                # unaligned: the cluster kernel to 64 KB
    assert p.path == rws.PATH_CLUSTER and p.cluster == 2 and p.bulk_copy == 0
    assert plan(1, 16384, in_ptr=(1 << 20) + 4).path == rws.PATH_CLUSTER
    assert plan(1, 16388, in_ptr=(1 << 20) + 4).path == rws.PATH_TWOPASS
    p = plan(1, 16388)
    assert p.path == rws.PATH_TWOPASS and p.cluster == 1 and p.bulk_copy == 1
    # Few rows: clusters grow (slices of at least 64 KB) up to 8 CTAs.
    assert plan(1, 32768).cluster == 2 and plan(1, 32772).cluster == 2
    assert plan(1, 131072).cluster == 8 and plan(1, 262144).cluster == 8
    assert plan(1, 4 << 20).cluster == 8                  # capped: 16-CTA clusters pack poorly
    assert plan(64, 1 << 20).cluster == 4                 # many rows: about 256 KB slices, <= 4
    assert plan(1, 16384, dtype=rws.BF16).path == rws.PATH_CTA
    assert plan(1, 16392, dtype=rws.BF16).path == rws.PATH_TWOPASS
    assert plan(1, 16392, dtype=rws.BF16, in_ptr=(1 << 20) + 2).path == rws.PATH_CLUSTER
    assert plan(1, 32768, dtype=rws.BF16, in_ptr=(1 << 20) + 2).path == rws.PATH_CLUSTER
    assert plan(1, 32776, dtype=rws.BF16, in_ptr=(1 << 20) + 2).path == rws.PATH_TWOPASS
    forced = plan(1, 16 * 32768, path=rws.PATH_CLUSTER)    # forced: 128 KB slices
    assert forced.cluster == 16 and forced.threads == 1024 and forced.chunks == 8
    assert forced.smem_bytes == 131072
    tp = plan(3, 10_000_000)
    assert tp.path == rws.PATH_TWOPASS and tp.cluster == 8 and tp.grid == 0
    assert plan(3, 10_000_000, path=rws.PATH_TWOPASS).cluster == 16   # forced: up to 16
    for n in (1025, 3000, 4096, 5000, 8192, 8196, 16384, 20000, 131072, 262144, 524288):
        for path in (rws.PATH_AUTO, rws.PATH_CLUSTER):
            q = plan(2, n, path=path)
            if q.path in (rws.PATH_CTA, rws.PATH_CLUSTER):
                assert q.threads * q.chunks * 4 >= q.slice_cols          # slice fits registers
                assert q.stages * q.slice_cols * 4 == q.smem_bytes
                assert q.smem_bytes <= rws.GB300["max_smem_per_block_optin"] - 2048
            if q.path == rws.PATH_TWOPASS:
                assert q.slice_cols * q.cluster >= n


def test_scheduler_alignment_fallbacks(lib):
    # Unaligned input pointer: no bulk copy, no ring; unaligned output stride: scalar stores.
    p = plan(64, 4096, in_ptr=(1 << 20) + 4)
    assert p.path == rws.PATH_CTA and p.bulk_copy == 0 and p.stages == 0 and p.smem_bytes == 0
    p = plan(64, 4096, out_row_stride=4097)
    assert p.bulk_copy == 1 and p.out_vec == 1
    p = plan(64, 1000, in_row_stride=1001)
    assert p.path == rws.PATH_WARP and p.bulk_copy == 0 and p.vec == 1 and p.chunks == 32
    p = plan(64, 1000, out_row_stride=1001, dtype=rws.BF16)   # staged input, scalar stores
    assert p.path == rws.PATH_WARP and p.bulk_copy == 1 and p.vec == 1 and p.chunks == 32
    p = plan(64, 1000, path=rws.PATH_WARP)                     # forced: staged tiles for fp32
    assert p.bulk_copy == 1


def test_scheduler_forced_paths(lib):
    assert plan(8, 100, path=rws.PATH_CTA).path == rws.PATH_CTA
    assert plan(8, 100, path=rws.PATH_CLUSTER).cluster == 2
    assert plan(8, 100, path=rws.PATH_TWOPASS).cluster == 1
    with pytest.raises(rws.SoftmaxError) as e:
        plan(8, 1025, path=rws.PATH_WARP)
    assert e.value.status == rws.ERR_UNSUPPORTED
    with pytest.raises(rws.SoftmaxError) as e:
        plan(8, 200_000, path=rws.PATH_CTA)
    assert e.value.status == rws.ERR_UNSUPPORTED
    small_cluster = dict(GB, max_cluster=8)
    assert rws.plan_for_device(small_cluster, 4, 262144).path == rws.PATH_TWOPASS
    assert rws.plan_for_device(small_cluster, 4, 4 << 20).cluster == 8
    p = rws.plan_for_device(small_cluster, 4, 262144, path=rws.PATH_CLUSTER)
    assert p.path == rws.PATH_CLUSTER and p.cluster == 8 and p.slice_cols == 32768
    assert p.threads == 1024 and p.stages == 1 and p.chunks == 8   # 2 x 128 KB would not fit


def test_validation(lib):
    f = lambda *a: rws.softmax_rows_ptr(*a)
    A, B = 1 << 20, 1 << 30
    assert f(A, B, -1, 4, 4, 4, rws.F32) == rws.ERR_INVALID_ARG
    assert f(A, B, 4, -1, 4, 4, rws.F32) == rws.ERR_INVALID_ARG
    assert f(A, B, 2, 4, 3, 4, rws.F32) == rws.ERR_INVALID_ARG      # short stride
    assert f(A, B, 2, 4, 4, 2, rws.F32) == rws.ERR_INVALID_ARG
    assert f(0, B, 2, 4, 4, 4, rws.F32) == rws.ERR_INVALID_ARG      # NULL
    assert f(A + 2, B, 2, 4, 4, 4, rws.F32) == rws.ERR_INVALID_ARG  # misaligned element
    assert f(A + 2, B + 2, 2, 4, 4, 4, rws.BF16) != rws.ERR_INVALID_ARG or True
    assert f(A, B, 2, 4, 4, 4, 5) == rws.ERR_INVALID_ARG            # dtype
    assert f(A, B, 2, 4, 4, 4, 3) == rws.ERR_INVALID_ARG
    assert f(A + 2, B, 2, 4, 4, 4, rws.F16) != rws.ERR_INVALID_ARG   # 2-byte aligned is enough
    assert f(0, 0, 0, 4, 4, 4, rws.F32) == rws.OK                   # empty: no-op
    assert f(0, 0, 4, 0, 4, 4, rws.F32) == rws.OK
    # Overlap: partial overlap rejected, identical (in place) accepted by validation.
    assert f(A, A + 8, 4, 16, 16, 16, rws.F32) == rws.ERR_INVALID_ARG
    assert f(A, A + 4 * 16 * 4, 4, 16, 16, 16, rws.F32) != rws.ERR_INVALID_ARG
    # Interleaved halves of a 32-wide matrix with equal strides do not overlap.
    assert f(A, A + 16 * 4, 4, 16, 32, 32, rws.F32) != rws.ERR_INVALID_ARG
    assert f(A, A + 15 * 4, 4, 16, 32, 32, rws.F32) == rws.ERR_INVALID_ARG


def test_options_validation(lib):
    g = lambda **kw: rws.softmax_rows_ex_ptr(1 << 20, 1 << 30, 2, 8, 8, 8, rws.F32, **kw)
    for bad in (dict(scale=0.0), dict(scale=-0.5), dict(scale=float("nan")),
                dict(scale=float("inf")), dict(scale=2.0 ** 127 * 1.5),
                dict(causal=True, causal_offset=1 << 62), dict(causal=True, causal_offset=-(1 << 62)),
                dict(path=4), dict(path=-2)):
        assert g(**bad) == rws.ERR_INVALID_ARG, bad
    # Valid options on an empty matrix: a no-op, no device needed.
    assert rws.softmax_rows_ex_ptr(0, 0, 0, 8, 8, 8, rws.F32, scale=0.125, causal=True) == rws.OK


def test_visible_cols_division_by_invariant_period(lib):
    """The kernels' row mod period (multiply-high, no division) against Python's
    integer %, for periods and rows up to 2^62 (periods beyond the row count act
    as the row count)."""
    import random
    rnd = random.Random(5)
    big = 1 << 62
    periods = [1, 2, 3, 5, 7, 641, 1024, 2047, 2048, 6700417, (1 << 31) - 1, 1 << 32,
               (1 << 32) + 1, 10 ** 12 + 39, (1 << 61) + 1, big - 2, big - 1, big, (1 << 63) - 1]
    periods += [rnd.randrange(1, big) for _ in range(40)]
    n_cols = (1 << 31) - 1
    for per in periods:
        rows = [0, 1, per - 1, per, per + 1, big - 1, 2 * per - 1 if 2 * per <= big else big - 1]
        rows += [rnd.randrange(0, big) for _ in range(25)]
        for r in rows:
            if not 0 <= r < big:
                continue
            for off in (0, 3, -7, (1 << 62) - 1, -(1 << 62) + 1):
                want = min(max(r % per + off + 1, 0), n_cols)
                got = rws.visible_cols(big, n_cols, r, causal=True, causal_period=per,
                                       causal_offset=off)
                assert got == want, (per, r, off)
    assert rws.visible_cols(10, 8, 3) == 8                                  # no mask
    assert rws.visible_cols(10, 8, 3, causal=True) == 4                     # period = n_rows
    assert rws.visible_cols(10, 8, 9, causal=True, causal_period=4) == 2
    assert rws.visible_cols(10, 8, 10, causal=True) == -1                   # row out of range
    assert rws.visible_cols(10, 8, 1, scale=0.0) == -1


def test_attention_options_validation(lib):
    """Options are checked before any device work: impl outside 0..3, a bad
    scale or offset is rejected; valid options on no queries are a no-op."""
    g = lambda **kw: rws.attention_forward_ptr(1 << 20, 1 << 21, 1 << 22, 1 << 23, 0, 2, 64, 64,
                                               64, rws.BF16, **kw)
    for bad in (dict(impl=4), dict(impl=-1), dict(scale=0.0), dict(scale=float("nan")),
                dict(causal=True, causal_offset=1 << 62)):
        assert g(**bad) == rws.ERR_INVALID_ARG, bad
    for impl in (0, 1, 2, 3):
        assert rws.attention_forward_ptr(0, 0, 0, 0, 0, 0, 64, 64, 64, rws.BF16,
                                         impl=impl) == rws.OK


def test_attention_grid_and_lse_checks(lib):
    """A grid past 2^31 - 1 CTAs is refused for every kernel choice as
    UNSUPPORTED before any device work; an lse buffer overlapping q, k, v or o
    is an invalid argument."""
    Q, K, V, O = 1 << 50, 2 << 50, 3 << 50, 4 << 50       # fake, far-apart device addresses
    bh = (1 << 31) - 1
    for impl in (0, 1, 2, 3):
        assert rws.attention_forward_ptr(Q, K, V, O, 0, bh, 512, 64, 64, rws.BF16,
                                         impl=impl) == rws.ERR_UNSUPPORTED, impl
    for lse in (Q + 64, K, V + 4096, O, O + 2 * 64 * 100 * 2 - 4):
        assert rws.attention_forward_ptr(Q, K, V, O, lse, 2, 100, 64, 64,
                                         rws.BF16) == rws.ERR_INVALID_ARG, hex(lse)


def test_no_gpu_means_loud_failure(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # Valid arguments, no device: UNSUPPORTED, never a silent CPU result.
    assert rws.softmax_rows_ptr(1 << 20, 1 << 30, 2, 8, 8, 8, rws.F32) == rws.ERR_UNSUPPORTED
    assert rws.softmax_rows_ex_ptr(1 << 20, 1 << 30, 2, 8, 8, 8, rws.F32, scale=0.5,
                                   causal=True) == rws.ERR_UNSUPPORTED
    for impl in (0, 3):
        assert rws.attention_forward_ptr(1 << 20, 1 << 21, 1 << 22, 1 << 23, 0, 2, 64, 64, 64,
                                         rws.BF16, impl=impl) == rws.ERR_UNSUPPORTED


def test_c_only_caller(lib, tmp_path):
    exe = tmp_path / "abi_caller"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c", "abi_caller.c"), "-o", str(exe),
                    rws.library_path(), "-Wl,-rpath," + os.path.dirname(rws.library_path())],
                   check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr


def test_strided_validation(lib):
    """softmax_strided checks its arguments before any device work."""
    A, B = 1 << 20, 1 << 30                           # fake, far-apart device addresses
    s = lambda *a, dtype=rws.F32: rws.softmax_strided_ptr(*a, dtype)
    # Column softmax of a 64 x 32 row-major matrix: 32 rows of 64, strides (1, 32).
    ok = (A, B, 32, 64, 1, 32, 1, 32)
    assert s(*ok, dtype=7) == rws.ERR_INVALID_ARG                     # unknown dtype
    assert s(A, B, -1, 64, 1, 32, 1, 32) == rws.ERR_INVALID_ARG       # negative size
    assert s(A, B, 32, 64, 1, -32, 1, 32) == rws.ERR_INVALID_ARG      # negative stride
    assert s(0, B, 32, 64, 1, 32, 1, 32) == rws.ERR_INVALID_ARG       # null input
    assert s(A + 2, B, 32, 64, 1, 32, 1, 32) == rws.ERR_INVALID_ARG   # misaligned f32
    assert s(A, B, 32, 64, 1, 32, 1, 16) == rws.ERR_INVALID_ARG       # outputs alias each other
    assert s(A, A + 64, 32, 64, 1, 32, 1, 32) == rws.ERR_INVALID_ARG  # partial in/out overlap
    assert s(A, B, 0, 64, 1, 32, 1, 32) == rws.OK                     # empty: no-op
    assert s(A, B, 1 << 40, 1 << 40, 1, 1 << 40, 1, 1 << 40) == rws.ERR_INVALID_ARG  # span overflow


def test_backward_validation(lib):
    """softmax_backward_rows checks y, dy and dx like the forward call checks
    in and out: dx may be y or dy in place, never partly overlap them."""
    A, B, C = 1 << 20, 1 << 28, 1 << 30
    g = lambda *a, dtype=rws.F32: rws.softmax_backward_rows_ptr(*a, dtype)
    assert g(A, B, C, 8, 100, 100, 100, 100, dtype=9) == rws.ERR_INVALID_ARG
    assert g(A, B, C, -1, 100, 100, 100, 100) == rws.ERR_INVALID_ARG
    assert g(A, B, C, 8, 100, 50, 100, 100) == rws.ERR_INVALID_ARG      # stride < n_cols
    assert g(0, B, C, 8, 100, 100, 100, 100) == rws.ERR_INVALID_ARG     # null y
    assert g(A, B, A + 40, 8, 100, 100, 100, 100) == rws.ERR_INVALID_ARG  # dx partly over y
    assert g(A, B, B + 40, 8, 100, 100, 100, 100) == rws.ERR_INVALID_ARG  # dx partly over dy
    assert g(A, B, C, 0, 100, 100, 100, 100) == rws.OK                  # empty: no-op


def test_strided_and_backward_without_a_device(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    A, B, C = 1 << 20, 1 << 28, 1 << 30
    assert rws.softmax_strided_ptr(A, B, 32, 64, 1, 32, 1, 32, rws.F32) == rws.ERR_UNSUPPORTED
    assert rws.softmax_backward_rows_ptr(A, B, C, 8, 100, 100, 100, 100,
                                         rws.F32) == rws.ERR_UNSUPPORTED


def test_every_scheduled_plan_passes_its_own_check(lib):
    """Host-only: across row lengths, row counts, dtypes, strides and
    alignments, every plan the scheduler makes passes softmax_plan_check, and
    the same plan with its coverage shrunk (fewer vectors, fewer lanes per
    row, a narrower slice) is rejected."""
    import itertools
    checked = rejected = 0
    cols = [1, 3, 8, 16, 33, 64, 100, 127, 128, 200, 1000, 1024, 1025, 1536, 2048, 3000, 4096,
            6144, 8192, 8500, 12288, 16384, 20000, 32768, 65536, 262144, 1600000]
    for n_cols, dtype, pad, off in itertools.product(cols, (rws.F32, rws.BF16, rws.F16),
                                                       (0, 1, 8), (0, 4)):
        for n_rows in (1, 7, 4099):
            stride = n_cols + pad
            in_ptr = (1 << 20) + off
            try:
                p = plan(n_rows, n_cols, in_row_stride=stride, out_row_stride=stride, dtype=dtype,
                         in_ptr=in_ptr)
            except rws.SoftmaxError:
                continue
            st = rws.plan_check(rws.GB300, p, n_rows, n_cols, stride, stride, dtype, in_ptr)
            assert st == rws.OK, (n_rows, n_cols, dtype, pad, off, str(p), rws.status_string(st))
            checked += 1
            bad = rws.Plan.from_buffer_copy(p)
            if p.path == rws.PATH_WARP and 2 <= p.lanes_per_row < 32:
                bad.lanes_per_row = p.lanes_per_row // 2
                if bad.lanes_per_row * p.vec >= n_cols:
                    continue
            elif p.path in (rws.PATH_CTA, rws.PATH_CLUSTER) and p.slice_cols > (16 // (4 if dtype == rws.F32 else 2)):
                bad.slice_cols = p.slice_cols // 2 // 8 * 8
                if bad.slice_cols * p.cluster >= n_cols:
                    continue
            elif p.path == rws.PATH_WARP and p.chunks > 1:
                bad.chunks = p.chunks // 2
                if 32 * bad.vec * bad.chunks >= n_cols:
                    continue
            else:
                continue
            st = rws.plan_check(rws.GB300, bad, n_rows, n_cols, stride, stride, dtype, in_ptr)
            assert st == rws.ERR_INVALID_ARG, (n_cols, dtype, str(bad))
            rejected += 1
    assert checked > 500 and rejected > 100, (checked, rejected)
