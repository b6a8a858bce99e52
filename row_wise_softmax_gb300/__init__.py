"""Python binding of libsoftmax (row-wise softmax for GB300, sm_103a).

Argument marshalling only: every step of the softmax runs in the library's
CUDA kernels.  The names mirror the C ABI in include/softmax.h:

    softmax_rows(x, out=None, stream=None, path=None)  torch tensors (CUDA)
    softmax_rows_ptr(...)                               raw pointers, C ABI call
    softmax_rows_host(h_in, h_out, d_in, d_out, ...)    host buffers, staged
    plan(...), plan_for_device(desc, ...)               scheduler decision
    device_status(clear), launch_count(), abi_version()

The shared library must have been built (``build()``); loading fails loudly
otherwise — there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "F32", "BF16", "F16", "PATH_AUTO", "PATH_WARP", "PATH_CTA", "PATH_CLUSTER", "PATH_TWOPASS",
    "OK", "ERR_INVALID_ARG", "ERR_UNSUPPORTED", "ERR_CUDA", "ERR_DEVICE_TIMEOUT",
    "SoftmaxError", "DeviceDesc", "Plan", "build", "lib", "library_path",
    "softmax_rows", "softmax_rows_ptr", "softmax_rows_ex_ptr", "softmax_rows_planned_ptr",
    "visible_cols", "softmax_backward", "softmax_backward_rows_ptr", "softmax",
    "softmax_strided_ptr", "attention", "attention_forward_ptr", "AttentionOptions",
    "ATT_AUTO", "ATT_MMA", "ATT_TCGEN05", "ATT_TCGEN05_PINGPONG",
    "Options", "softmax_rows_host", "plan", "plan_for_device",
    "status_string", "device_status", "launch_count", "selftest_wait_timeout", "abi_version", "GB300",
]

F32, BF16, F16 = 0, 1, 2
PATH_AUTO, PATH_WARP, PATH_CTA, PATH_CLUSTER, PATH_TWOPASS = -1, 0, 1, 2, 3
PATH_NAMES = {PATH_WARP: "warp", PATH_CTA: "cta", PATH_CLUSTER: "cluster", PATH_TWOPASS: "twopass"}
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_DEVICE_TIMEOUT = 0, 1, 2, 3, 4

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libsoftmax.so")
_lib = None


class SoftmaxError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = status_string(status) if _lib is not None else "status %d" % status
        super().__init__("%s%s (status %d)" % (what + ": " if what else "", msg, status))


class DeviceDesc(ctypes.Structure):
    _fields_ = [("sm_count", ctypes.c_int), ("max_threads_per_sm", ctypes.c_int),
                ("max_smem_per_sm", ctypes.c_int), ("max_smem_per_block_optin", ctypes.c_int),
                ("regs_per_sm", ctypes.c_int), ("cc_major", ctypes.c_int),
                ("cc_minor", ctypes.c_int), ("max_cluster", ctypes.c_int)]


class Options(ctypes.Structure):
    _fields_ = [("scale", ctypes.c_float), ("causal", ctypes.c_int32),
                ("causal_period", ctypes.c_int64), ("causal_offset", ctypes.c_int64)]


class AttentionOptions(ctypes.Structure):
    _fields_ = [("scale", ctypes.c_float), ("causal", ctypes.c_int32),
                ("causal_offset", ctypes.c_int64), ("impl", ctypes.c_int32)]


ATT_AUTO, ATT_MMA, ATT_TCGEN05, ATT_TCGEN05_PINGPONG = 0, 1, 2, 3


class Plan(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("dtype", ctypes.c_int), ("vec", ctypes.c_int),
                ("out_vec", ctypes.c_int), ("bulk_copy", ctypes.c_int),
                ("threads", ctypes.c_int), ("cluster", ctypes.c_int),
                ("rows_per_warp", ctypes.c_int), ("chunks", ctypes.c_int),
                ("slice_cols", ctypes.c_int64), ("stages", ctypes.c_int),
                ("smem_bytes", ctypes.c_int),
                ("grid", ctypes.c_int64), ("lanes_per_row", ctypes.c_int)]

    def __str__(self) -> str:
        buf = ctypes.create_string_buffer(256)
        lib().softmax_plan_format(ctypes.byref(self), buf, 256)
        return buf.value.decode()

    @property
    def path_name(self) -> str:
        return PATH_NAMES.get(self.path, "?")


# A GB300 as the scheduler sees it (for host-only planning and tests).
GB300 = dict(sm_count=152, max_threads_per_sm=2048, max_smem_per_sm=233472,
             max_smem_per_block_optin=232448, regs_per_sm=65536, cc_major=10, cc_minor=3,
             max_cluster=16)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libsoftmax.so for sm_103a in-tree (nvcc) and return its path."""
    from . import _build
    return _build.build(force=force, verbose=verbose)


def library_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded shared library.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                "libsoftmax.so is not built (expected at %s); run "
                "row_wise_softmax_gb300.build() — there is no fallback path" % _LIB_PATH)
        L = ctypes.CDLL(_LIB_PATH)
        i64, vp, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        L.softmax_rows.argtypes = [vp, vp, i64, i64, i64, i64, ci, vp]
        L.softmax_rows.restype = ci
        L.softmax_rows_path.argtypes = [vp, vp, i64, i64, i64, i64, ci, vp, ci]
        L.softmax_rows_path.restype = ci
        L.softmax_rows_ex.argtypes = [vp, vp, i64, i64, i64, i64, ci, ctypes.POINTER(Options), ci,
                                      vp]
        L.softmax_rows_ex.restype = ci
        L.softmax_attention_forward.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, ci,
                                                ctypes.POINTER(AttentionOptions), vp]
        L.softmax_attention_forward.restype = ci
        L.softmax_strided.argtypes = [vp, vp, i64, i64, i64, i64, i64, i64, ci, vp]
        L.softmax_strided.restype = ci
        L.softmax_backward_rows.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, ci, vp]
        L.softmax_backward_rows.restype = ci
        L.softmax_visible_cols.argtypes = [ctypes.POINTER(Options), i64, i64, i64]
        L.softmax_visible_cols.restype = i64
        L.softmax_rows_planned.argtypes = [vp, vp, i64, i64, i64, i64, ci, ctypes.POINTER(Plan), vp]
        L.softmax_rows_planned.restype = ci
        L.softmax_rows_host.argtypes = [vp, vp, i64, i64, i64, i64, ci, vp, vp, vp]
        L.softmax_rows_host.restype = ci
        L.softmax_status_string.argtypes = [ci]
        L.softmax_status_string.restype = ctypes.c_char_p
        L.softmax_plan.argtypes = [ctypes.POINTER(DeviceDesc), vp, vp, i64, i64, i64, i64, ci, ci,
                                   ctypes.POINTER(Plan)]
        L.softmax_plan.restype = ci
        L.softmax_plan_format.argtypes = [ctypes.POINTER(Plan), ctypes.c_char_p, ctypes.c_size_t]
        L.softmax_plan_format.restype = ci
        L.softmax_plan_describe.argtypes = [i64, i64, ci, ctypes.c_char_p, ctypes.c_size_t]
        L.softmax_plan_describe.restype = ci
        L.softmax_plan_check.argtypes = [ctypes.POINTER(DeviceDesc), vp, vp, i64, i64, i64, i64, ci,
                                         ctypes.POINTER(Plan)]
        L.softmax_plan_check.restype = ci
        L.softmax_device_status.argtypes = [ci]
        L.softmax_device_status.restype = ci
        L.softmax_selftest_wait_timeout.argtypes = [vp]
        L.softmax_selftest_wait_timeout.restype = ci
        L.softmax_launch_count.argtypes = []
        L.softmax_launch_count.restype = ctypes.c_uint64
        L.softmax_abi_version.argtypes = []
        L.softmax_abi_version.restype = ci
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().softmax_status_string(status).decode()


def abi_version() -> int:
    return lib().softmax_abi_version()


def selftest_wait_timeout(stream: int = 0) -> int:
    """Queue the bounded-wait self-test kernel (see include/softmax.h)."""
    return lib().softmax_selftest_wait_timeout(stream)


def launch_count() -> int:
    return int(lib().softmax_launch_count())


def device_status(clear: bool = True) -> int:
    """Synchronise the device; OK or ERR_DEVICE_TIMEOUT if a kernel gave up a wait."""
    return lib().softmax_device_status(1 if clear else 0)


def softmax_rows_ptr(in_ptr: int, out_ptr: int, n_rows: int, n_cols: int, in_row_stride: int,
                     out_row_stride: int, dtype: int, stream: int = 0, path: int = PATH_AUTO) -> int:
    """Direct C ABI call; returns the status code (no exception)."""
    if path == PATH_AUTO:
        return lib().softmax_rows(in_ptr, out_ptr, n_rows, n_cols, in_row_stride,
                                  out_row_stride, dtype, stream)
    return lib().softmax_rows_path(in_ptr, out_ptr, n_rows, n_cols, in_row_stride,
                                   out_row_stride, dtype, stream, path)


def softmax_rows_ex_ptr(in_ptr: int, out_ptr: int, n_rows: int, n_cols: int, in_row_stride: int,
                       out_row_stride: int, dtype: int, scale: float = 1.0, causal: bool = False,
                       causal_period: int = 0, causal_offset: int = 0, stream: int = 0,
                       path: int = -1) -> int:
    """C ABI call of the scaled / causally masked softmax; returns the status."""
    o = Options(scale, 1 if causal else 0, causal_period, causal_offset)
    return lib().softmax_rows_ex(in_ptr, out_ptr, n_rows, n_cols, in_row_stride, out_row_stride,
                                 dtype, ctypes.byref(o), path, stream)


def attention_forward_ptr(q: int, k: int, v: int, o: int, lse: int, batch_heads: int, n_q: int,
                          n_k: int, head_dim: int, dtype: int, scale: float | None = None,
                          causal: bool = False, causal_offset: int = 0, stream: int = 0,
                          impl: int = 0) -> int:
    """C ABI call of the attention forward; returns the status.  ``impl``:
    0 the library's choice, 1 the mma.sync kernel, 2 the single-tile tcgen05
    kernel, 3 the ping-pong tcgen05 kernel."""
    opt = None
    if scale is not None or causal or causal_offset or impl:
        sc = scale if scale is not None else 1.0 / (head_dim ** 0.5)
        opt = ctypes.byref(AttentionOptions(sc, 1 if causal else 0, causal_offset, impl))
    return lib().softmax_attention_forward(q, k, v, o, lse or None, batch_heads, n_q, n_k,
                                           head_dim, dtype, opt, stream)


def attention(q, k, v, scale: float | None = None, causal: bool = False, causal_offset: int = 0,
              return_lse: bool = False, stream=None, impl: int = 0):
    """softmax(scale q k^T, causal mask) v for CUDA tensors [..., n, head_dim]
    (bf16 or fp16, contiguous; leading dimensions are batch and heads)."""
    import torch
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous() or t.dim() < 2:
            raise ValueError("attention: q, k, v must be contiguous CUDA tensors [..., n, d]")
    if q.dtype != k.dtype or q.dtype != v.dtype or k.shape != v.shape or \
            q.shape[:-2] != k.shape[:-2] or q.shape[-1] != k.shape[-1]:
        raise ValueError("attention: shapes or dtypes do not match")
    d, n_q, n_k = q.shape[-1], q.shape[-2], k.shape[-2]
    bh = q.numel() // max(n_q * d, 1) if q.numel() else 0
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device) if return_lse else None
    with torch.cuda.device(q.device):
        st = attention_forward_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr() if lse is not None else 0, bh, n_q, n_k, d,
                                   _dtype_code(q), scale, causal, causal_offset,
                                   _stream_handle(stream, q.device), impl)
    if st != OK:
        raise SoftmaxError(st, "attention")
    return (o, lse) if return_lse else o


def softmax_strided_ptr(in_ptr: int, out_ptr: int, n_rows: int, n_cols: int, in_row_stride: int,
                       in_col_stride: int, out_row_stride: int, out_col_stride: int, dtype: int,
                       stream: int = 0) -> int:
    """C ABI call of the strided softmax; returns the status."""
    return lib().softmax_strided(in_ptr, out_ptr, n_rows, n_cols, in_row_stride, in_col_stride,
                                 out_row_stride, out_col_stride, dtype, stream)


def softmax(x, dim: int = -1, out=None, stream=None):
    """softmax(x) along ``dim`` of a 2-D CUDA tensor with any strides (dim 0:
    column-wise).  ``out`` defaults to a new tensor laid out like ``x``."""
    import torch
    if x.dim() != 2 or not x.is_cuda:
        raise ValueError("softmax: expects a 2-D CUDA tensor")
    d = dim % 2
    if out is None:
        out = torch.empty_like(x)
    if out.shape != x.shape or out.dtype != x.dtype or out.device != x.device:
        raise ValueError("softmax: out must match x in dtype, shape and device")
    # Softmax rows run along `dim`: row index over the other dimension.
    r, c = (1, 0) if d == 0 else (0, 1)
    with torch.cuda.device(x.device):
        st = softmax_strided_ptr(x.data_ptr(), out.data_ptr(), x.shape[r], x.shape[c],
                                 x.stride(r), x.stride(c), out.stride(r), out.stride(c),
                                 _dtype_code(x), _stream_handle(stream, x.device))
    if st != OK:
        raise SoftmaxError(st, "softmax")
    return out


def softmax_backward_rows_ptr(y_ptr: int, dy_ptr: int, dx_ptr: int, n_rows: int, n_cols: int,
                              y_row_stride: int, dy_row_stride: int, dx_row_stride: int,
                              dtype: int, stream: int = 0) -> int:
    """C ABI call of the softmax backward; returns the status."""
    return lib().softmax_backward_rows(y_ptr, dy_ptr, dx_ptr, n_rows, n_cols, y_row_stride,
                                       dy_row_stride, dx_row_stride, dtype, stream)


def softmax_backward(y, dy, out=None, stream=None):
    """dx = y * (dy - sum(y * dy)) along the last dimension of CUDA tensors
    (1-D or 2-D, same dtype and shape); ``out`` may be ``dy`` or ``y``."""
    import torch
    if y.shape != dy.shape or y.dtype != dy.dtype or y.device != dy.device:
        raise ValueError("softmax_backward: y and dy must match in shape, dtype and device")
    if y.dim() not in (1, 2) or not y.is_cuda:
        raise ValueError("softmax_backward: expects 1-D or 2-D CUDA tensors")
    y2, g2 = (y.unsqueeze(0), dy.unsqueeze(0)) if y.dim() == 1 else (y, dy)
    if y2.stride(-1) != 1 or g2.stride(-1) != 1:
        raise ValueError("softmax_backward: rows must be contiguous (column stride 1)")
    if out is None:
        out = torch.empty_like(y)
    o2 = out.unsqueeze(0) if out.dim() == 1 else out
    if out.shape != y.shape or out.dtype != y.dtype or o2.stride(-1) != 1:
        raise ValueError("softmax_backward: out must match y")
    dt = _dtype_code(y)
    with torch.cuda.device(y.device):
        st = softmax_backward_rows_ptr(y2.data_ptr(), g2.data_ptr(), o2.data_ptr(), y2.shape[0],
                                       y2.shape[1], y2.stride(0), g2.stride(0), o2.stride(0), dt,
                                       _stream_handle(stream, y.device))
    if st != OK:
        raise SoftmaxError(st, "softmax_backward")
    return out


def visible_cols(n_rows: int, n_cols: int, row: int, scale: float = 1.0, causal: bool = False,
                 causal_period: int = 0, causal_offset: int = 0) -> int:
    """Leading columns of ``row`` that take part in its softmax (host-side, the
    kernels' own arithmetic); -1 for invalid arguments."""
    o = Options(scale, 1 if causal else 0, causal_period, causal_offset)
    return lib().softmax_visible_cols(ctypes.byref(o), n_rows, n_cols, row)


def softmax_rows_planned_ptr(in_ptr: int, out_ptr: int, n_rows: int, n_cols: int,
                             in_row_stride: int, out_row_stride: int, dtype: int, plan: Plan,
                             stream: int = 0) -> int:
    """C ABI call with an explicit (checked) scheduler decision; returns the status."""
    return lib().softmax_rows_planned(in_ptr, out_ptr, n_rows, n_cols, in_row_stride,
                                      out_row_stride, dtype, ctypes.byref(plan), stream)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float16:
        return F16
    raise TypeError("softmax_rows: dtype must be float32, bfloat16 or float16, got %s" % t.dtype)


def _as_rows(t, name: str):
    if t.dim() == 1:
        return 1, t.shape[0], t.shape[0]
    if t.dim() != 2:
        raise ValueError("%s must be 1-D or 2-D (rows x cols)" % name)
    if t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError("%s must have unit column stride" % name)
    return t.shape[0], t.shape[1], t.stride(0) if t.shape[0] > 1 else t.shape[1]


def _stream_handle(stream, device) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def softmax_rows(x, out=None, stream=None, path: int = PATH_AUTO, scale: float = 1.0,
                 causal: bool = False, causal_period: int = 0, causal_offset: int = 0):
    """y = softmax(scale * x) along the last dimension of a CUDA tensor (1-D or 2-D).

    ``out`` (optional) receives the result and may be ``x`` itself.  With
    ``causal``, column c of row r takes part iff c <= (r mod causal_period) +
    causal_offset (period <= 0: n_rows); masked inputs are not read and give
    exactly 0.  Runs on ``stream`` (default: torch's current stream) without
    synchronising.
    """
    import torch
    if not x.is_cuda:
        raise ValueError("softmax_rows: x must be a CUDA tensor (use softmax_rows_host for host data)")
    dt = _dtype_code(x)
    if out is None:
        out = torch.empty_like(x, memory_format=torch.contiguous_format)
    if out.dtype != x.dtype or out.shape != x.shape or out.device != x.device:
        raise ValueError("softmax_rows: out must match x in dtype, shape and device")
    n_rows, n_cols, ld_in = _as_rows(x, "x")
    _, _, ld_out = _as_rows(out, "out")
    transform = scale != 1.0 or causal
    with torch.cuda.device(x.device):
        h = _stream_handle(stream, x.device)
        if transform:
            st = softmax_rows_ex_ptr(x.data_ptr(), out.data_ptr(), n_rows, n_cols, ld_in, ld_out,
                                     dt, scale, causal, causal_period, causal_offset, h, path)
        else:
            st = softmax_rows_ptr(x.data_ptr(), out.data_ptr(), n_rows, n_cols, ld_in, ld_out, dt,
                                  h, path)
    if st != OK:
        raise SoftmaxError(st, "softmax_rows")
    return out


def softmax_rows_host(h_in, h_out, d_in=None, d_out=None, stream=None, device=None):
    """Softmax of host (CPU) rows.

    h_in / h_out: CPU tensors, 1-D or 2-D with unit column stride.
    Staged mode (d_in, d_out given): CUDA tensors with at least rows*cols
    elements each (may be the same tensor); pinned h_in / h_out make the
    copies asynchronous.  Direct mode (no device tensors): h_in / h_out must
    be pinned; the kernel reads and writes them over the host link.  Queued
    on ``stream``; synchronise before reading h_out.
    """
    import torch
    if h_in.is_cuda or h_out.is_cuda:
        raise ValueError("softmax_rows_host: h_in and h_out must be host tensors")
    dt = _dtype_code(h_in)
    if h_out.dtype != h_in.dtype:
        raise ValueError("softmax_rows_host: all buffers must share one dtype")
    n_rows, n_cols, ld_in = _as_rows(h_in, "h_in")
    r2, c2, ld_out = _as_rows(h_out, "h_out")
    if (r2, c2) != (n_rows, n_cols):
        raise ValueError("softmax_rows_host: h_out shape differs from h_in")
    if (d_in is None) != (d_out is None):
        raise ValueError("softmax_rows_host: give both device buffers or neither")
    if d_in is not None:
        if d_in.dtype != h_in.dtype or d_out.dtype != h_in.dtype:
            raise ValueError("softmax_rows_host: all buffers must share one dtype")
        if d_in.numel() < n_rows * n_cols or d_out.numel() < n_rows * n_cols:
            raise ValueError("softmax_rows_host: device buffers too small")
        device = d_in.device
        dptr_in, dptr_out = d_in.data_ptr(), d_out.data_ptr()
    else:
        device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
        dptr_in = dptr_out = None
    with torch.cuda.device(device):
        st = lib().softmax_rows_host(h_in.data_ptr(), h_out.data_ptr(), n_rows, n_cols, ld_in,
                                     ld_out, dt, dptr_in, dptr_out,
                                     _stream_handle(stream, device))
    if st != OK:
        raise SoftmaxError(st, "softmax_rows_host")
    return h_out


def plan_for_device(desc: dict | DeviceDesc | None, n_rows: int, n_cols: int,
                    in_row_stride: int | None = None, out_row_stride: int | None = None,
                    dtype: int = F32, path: int = PATH_AUTO, in_ptr: int = 1 << 20,
                    out_ptr: int = 1 << 30) -> Plan:
    """Run the scheduler.  desc=None queries the current GPU; a dict or
    DeviceDesc plans on the host only (pointers are inspected for alignment)."""
    if in_row_stride is None:
        in_row_stride = n_cols
    if out_row_stride is None:
        out_row_stride = n_cols
    p = Plan()
    if desc is None:
        dp = None
    else:
        d = desc if isinstance(desc, DeviceDesc) else DeviceDesc(**desc)
        dp = ctypes.byref(d)
    st = lib().softmax_plan(dp, in_ptr, out_ptr, n_rows, n_cols, in_row_stride, out_row_stride,
                            dtype, path, ctypes.byref(p))
    if st != OK:
        raise SoftmaxError(st, "softmax_plan")
    return p


def plan_check(desc: dict | DeviceDesc | None, plan_: Plan, n_rows: int, n_cols: int,
               in_row_stride: int | None = None, out_row_stride: int | None = None,
               dtype: int = F32, in_ptr: int = 1 << 20, out_ptr: int = 1 << 30) -> int:
    """softmax_plan_check: the status softmax_rows_planned would give this plan
    before launching (desc=None: the current GPU; a dict or DeviceDesc: host only)."""
    if in_row_stride is None:
        in_row_stride = n_cols
    if out_row_stride is None:
        out_row_stride = n_cols
    dp = None
    if desc is not None:
        d = desc if isinstance(desc, DeviceDesc) else DeviceDesc(**desc)
        dp = ctypes.byref(d)
    return lib().softmax_plan_check(dp, in_ptr, out_ptr, n_rows, n_cols, in_row_stride,
                                    out_row_stride, dtype, ctypes.byref(plan_))


def plan(n_rows: int, n_cols: int, **kw) -> Plan:
    """Scheduler decision on the current GPU."""
    return plan_for_device(None, n_rows, n_cols, **kw)


def plan_describe(n_rows: int, n_cols: int, dtype: int = F32) -> str:
    """The scheduler's decision for contiguous, aligned rows on the current
    GPU, as the library's one-line text (softmax_plan_describe)."""
    buf = ctypes.create_string_buffer(256)
    st = lib().softmax_plan_describe(n_rows, n_cols, dtype, buf, 256)
    if st != OK:
        raise SoftmaxError(st, "softmax_plan_describe")
    return buf.value.decode()
