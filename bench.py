"""Row-wise softmax benchmark: GB/s and fraction of the GB300 HBM roofline.

One step = one softmax_rows call (the whole hot path: load, max, exp, sum,
normalise, store) over the headline workload, 4096 x 4096 fp32 with -inf
entries and a constant row.  Bytes are algorithmic: n_rows * n_cols *
(in + out element size), one read and one write of every element.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line (rank 0).  Timing: one pair of CUDA events on the
launching stream around the K steps, launched back to back.  L2 never holds a step's
inputs: the steps rotate over enough input/output buffer sets that together
they exceed three times the L2 size ("inputs larger than L2"), so each step
reads its input from HBM and pays, like any steady stream of calls, for the
write-back of the previous step's outputs.  Inputs are resident in HBM before
the timed region starts.  Under torchrun (N > 1) every rank runs its own copy
of the workload (rows shard with no exchange: weak scaling) and the time is
the maximum over ranks.

--impl reference times the CPU oracle (double precision, single-threaded) on
the same workload and prints the same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as wl  # noqa: E402

HEADLINE = "masked_f32"
METRIC = "softmax GB/s and % of GB300 HBM roofline (fp32/bf16) per row-length config"
UNIT = "GB/s"
L2_FACTOR = 3            # rotating buffer sets cover at least 3x the L2 size
PROFILE_DIR = os.path.join(ROOT, "profiles")
# The kernel a plan launches (path, and whether it stages rows with bulk
# copies) and its sources, hashed to tell whether committed ncu counters
# still describe the kernel being timed.
KERNELS = {
    ("warp", 0): ("warp_rows_kernel", ["warp_rows.cu"]),
    ("warp", 1): ("tile_rows_kernel", ["tile_rows.cu"]),
    ("cta", 0): ("row_slices_kernel", ["row_slices.cu"]),
    ("cta", 1): ("row_slices_kernel", ["row_slices.cu"]),
    ("cluster", 0): ("row_slices_kernel", ["row_slices.cu"]),
    ("cluster", 1): ("row_slices_kernel", ["row_slices.cu"]),
    ("twopass", 0): ("twopass_kernel", ["twopass.cu"]),
    ("twopass", 1): ("stream_rows_kernel", ["stream_rows.cu", "cluster_ring.cuh"]),
}
COMMON_SOURCES = ["common.cuh", "kernels.h"]
DTYPE_NAMES = {wl.F32: "f32", wl.BF16: "bf16", wl.F16: "f16"}
WORKLOAD_DATA = {
    "small_f32": "synthetic (seeded: N(0,1))",
    "masked_f32": "synthetic (seeded: N(0,3^2), 41 -inf columns per row, one constant row)",
    "causal_bf16": "synthetic (seeded: bf16(N(0,1)*8), causal: row r keeps columns <= r mod 1024)",
    "short_f32": "synthetic (seeded: U[-80,80], input stride 128 with a NaN padding column)",
    "long_f32": "synthetic (seeded: N(0,1), one +50 spike per row)",
    "causal_f16": "synthetic (seeded: fp16(N(0,1)*8), causal: row r keeps columns <= r mod 1024)",
}


# The five configurations' short tags, in the order the configurations are listed.
CONFIG_TAGS = {"small_f32": "C1", "masked_f32": "C2", "causal_bf16": "C3", "short_f32": "C4",
               "long_f32": "C5"}


def kernel_of(plan):
    return KERNELS[(plan.path_name, 1 if plan.bulk_copy else 0)]


def workload_label(w: wl.Workload, options: bool = False) -> str:
    """The workload as both arms name it in config.workload."""
    return "%s: %d x %d %s, row strides %d/%d%s" % (
        w.name, w.n_rows, w.n_cols, DTYPE_NAMES[w.dtype], w.in_row_stride, w.out_row_stride,
        ", mask from indices, scale %g" % FUSED_SCALE if options else "")


def sig(x: float, digits: int = 4) -> float:
    """x rounded to `digits` significant digits (keeps the JSON line short)."""
    return float("%.*g" % (digits, x))


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def shard_rows(n_rows: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous row block [lo, hi) of a row-split across ranks (no exchange)."""
    base, extra = divmod(n_rows, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def max_over_ranks(value: float, world: int, device: str = "cpu") -> float:
    """The largest value over all ranks (the job's time is its slowest rank's)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def source_hash(plan) -> str:
    h = hashlib.sha256()
    for f in kernel_of(plan)[1] + COMMON_SOURCES:
        with open(os.path.join(ROOT, "row_wise_softmax_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def committed_record(plan, workload: str):
    """The committed one-launch ncu record (DRAM bytes, duration) of the
    kernel this plan launches on this workload, if the kernel's sources still
    hash to the captured value: (record or None, its path or why not)."""
    fn = os.path.join(PROFILE_DIR, "%s.%s.json" % (kernel_of(plan)[0], workload))
    try:
        with open(fn) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None, "no committed ncu summary"
    if rec.get("source_sha") != source_hash(plan):
        return None, "kernel changed since the ncu capture"
    return rec, os.path.relpath(fn, ROOT)


def committed_traffic(plan, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if still valid."""
    rec, src = committed_record(plan, workload)
    return (rec.get("dram_bytes_per_launch") if rec else None), src


def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while a region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)       # let the first sample land before the region
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- GPU arm

def torch_dtype(dtype: int, torch):
    return {wl.F32: torch.float32, wl.BF16: torch.bfloat16, wl.F16: torch.float16}[dtype]


def to_device(w: wl.Workload, torch):
    if w.dtype == wl.F32:
        return torch.from_numpy(w.data).cuda()
    return torch.from_numpy(w.data.view(np.int16)).cuda().view(torch_dtype(w.dtype, torch))


def device_buffers(w: wl.Workload, torch, l2_bytes: int):
    """Input/output buffer sets, enough that their total exceeds L2_FACTOR x L2."""
    x = to_device(w, torch)
    dt = torch_dtype(w.dtype, torch)
    set_bytes = (x.numel() + max(w.out_elems, 1)) * x.element_size()
    n_sets = max(1, -(-L2_FACTOR * l2_bytes // set_bytes))
    sets = []
    for i in range(n_sets):
        xi = x if i == 0 else x.clone()
        sets.append((xi, torch.empty(max(w.out_elems, 1), dtype=dt, device="cuda")))
    return sets


def hold_stream(torch, steps: int):
    """Keep the stream busy (torch's sleep kernel) while the host enqueues the
    timed launches, so that the timed region starts with the whole batch
    queued: it then measures the device back to back, not the host's launch
    rate or the latency of the first launch after an idle GPU."""
    torch.cuda._sleep(int(min(20e-3, 30e-6 * steps + 100e-6) * 2.0e9))


def time_device(w: wl.Workload, sets, steps: int, warmup: int, torch, rws, stream,
                options=None):
    """softmax_rows (softmax_rows_ex with ``options``, a rws.Options) over
    rotating buffer sets, steps back to back (inputs resident in HBM, never in
    L2).  Returns (total ms of the timed steps from one pair of CUDA events on
    the launching stream, kernel launches)."""
    if options is None:
        calls = [(x.data_ptr(), y.data_ptr(), w.n_rows, w.n_cols, w.in_row_stride,
                  w.out_row_stride, w.dtype, stream.cuda_stream) for x, y in sets]
        call = rws.lib().softmax_rows
    else:
        import ctypes
        calls = [(x.data_ptr(), y.data_ptr(), w.n_rows, w.n_cols, w.in_row_stride,
                  w.out_row_stride, w.dtype, ctypes.byref(options), rws.PATH_AUTO,
                  stream.cuda_stream) for x, y in sets]
        call = rws.lib().softmax_rows_ex
    for i in range(warmup):
        st = call(*calls[i % len(calls)])
        if st != rws.OK:
            raise RuntimeError("softmax_rows: " + rws.status_string(st))
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = rws.launch_count()
    hold_stream(torch, steps)
    a.record(stream)
    for i in range(steps):
        call(*calls[(warmup + i) % len(calls)])
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b), rws.launch_count() - launches0


def time_each_step(w: wl.Workload, sets, steps: int, torch, rws, stream):
    """softmax_rows over the rotating sets with every step bracketed by its own
    pair of CUDA events (each launch's ramp and drain included, no overlap
    with its neighbours): the per-step times in ms."""
    calls = [(x.data_ptr(), y.data_ptr(), w.n_rows, w.n_cols, w.in_row_stride,
              w.out_row_stride, w.dtype, stream.cuda_stream) for x, y in sets]
    call = rws.lib().softmax_rows
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    torch.cuda.synchronize()
    hold_stream(torch, steps)
    for i, (a, b) in enumerate(ev):
        a.record(stream)
        call(*calls[i % len(calls)])
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def percentile(xs, q: float) -> float:
    """The q-quantile of xs by linear interpolation between order statistics."""
    ys = sorted(xs)
    pos = q * (len(ys) - 1)
    lo = int(pos)
    hi = min(lo + 1, len(ys) - 1)
    return ys[lo] + (ys[hi] - ys[lo]) * (pos - lo)


def copy_calibration(w: wl.Workload, sets, torch, stream, peak):
    """torch copy_ of the same number of bytes (read n, write n), timed like a
    step over the same rotating sets: the rate a plain copy of this size gets."""
    n = w.n_rows * w.n_cols
    pairs = [(x.reshape(-1)[:n], y.reshape(-1)[:n]) for x, y in sets if y.numel() >= n]
    if not pairs:
        return None
    for i in range(5):
        src, dst = pairs[i % len(pairs)]
        dst.copy_(src)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    hold_stream(torch, 30)
    a.record(stream)
    for i in range(30):
        src, dst = pairs[i % len(pairs)]
        dst.copy_(src)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / 30
    gbs = 2 * n * pairs[0][0].element_size() / (ms * 1e-3) / 1e9
    return {"GB/s": round(gbs, 1), "mean_ms": round(ms, 5), "frac_of_peak": round(gbs / peak, 4)}


FUSED_SCALE = 0.125          # 1/sqrt(64), a head dimension of 64


def fused_causal_setup(w: wl.Workload, rws):
    """Options of the causal workload with its mask computed from indices
    (query r mod n_cols sees keys 0..r mod n_cols) and a 1/sqrt(64) scale,
    and its algorithmic bytes: the masked inputs are never read, so the
    kept inputs plus every output."""
    period = w.n_cols
    opt = rws.Options(FUSED_SCALE, 1, period, 0)
    kept = sum(min(r % period + 1, w.n_cols) for r in range(w.n_rows))
    return opt, (kept + w.n_rows * w.n_cols) * w.elem_bytes


def fused_causal_entry(torch, rws, stream, l2_bytes, peak):
    """softmax_rows_ex on the causal bf16 workload with the mask from indices."""
    w = wl.make("causal_bf16")
    period = w.n_cols
    opt, algo = fused_causal_setup(w, rws)
    bc = device_buffers(w, torch, l2_bytes)
    tot, launches = time_device(w, bc, 50, 5, torch, rws, stream, options=opt)
    del bc
    med = tot / 50
    gbs = algo / (med * 1e-3) / 1e9
    return {"shape": [w.n_rows, w.n_cols], "dtype": "bf16",
            "options": {"scale": FUSED_SCALE, "causal": 1, "causal_period": period,
                        "causal_offset": 0},
            "algorithmic_bytes": algo, "mean_ms": round(med, 5), "GB/s": round(gbs, 1),
            "frac_of_measured_peak": round(gbs / peak, 4), "launches": launches,
            "rows_per_s": round(w.n_rows / (med * 1e-3), 1)}


def backward_entry(torch, rws, stream, l2_bytes, peak, n_rows=4096, n_cols=4096, dtype=wl.F32):
    """softmax_backward_rows over rotating (y, dy, dx) sets: three element
    transfers per element (read y, read dy, write dx)."""
    y, g = wl.backward_pair(n_rows, n_cols, dtype)
    dt = torch_dtype(dtype, torch)

    def dev(a):
        t = torch.from_numpy(a if dtype == wl.F32 else a.view(np.int16)).cuda()
        return t if dtype == wl.F32 else t.view(dt)

    ty, tg = dev(y), dev(g)
    esz = 4 if dtype == wl.F32 else 2
    algo = 3 * n_rows * n_cols * esz
    n_sets = max(1, -(-L2_FACTOR * l2_bytes // algo))
    sets = [(ty if i == 0 else ty.clone(), tg if i == 0 else tg.clone(), torch.empty_like(ty))
            for i in range(n_sets)]
    call = rws.lib().softmax_backward_rows
    args = [(a.data_ptr(), b.data_ptr(), c.data_ptr(), n_rows, n_cols, n_cols, n_cols, n_cols,
             dtype, stream.cuda_stream) for a, b, c in sets]
    for i in range(5):
        if call(*args[i % n_sets]) != rws.OK:
            raise RuntimeError("softmax_backward_rows failed")
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = rws.launch_count()
    hold_stream(torch, 50)
    a.record(stream)
    for i in range(50):
        call(*args[i % n_sets])
    b.record(stream)
    torch.cuda.synchronize()
    med = a.elapsed_time(b) / 50
    gbs = algo / (med * 1e-3) / 1e9
    return {"shape": [n_rows, n_cols], "dtype": DTYPE_NAMES[dtype],
            "op": "softmax_backward_rows: dx = y * (dy - sum(y * dy))",
            "algorithmic_bytes": algo, "mean_ms": round(med, 5), "GB/s": round(gbs, 1),
            "frac_of_measured_peak": round(gbs / peak, 4),
            "launches": rws.launch_count() - launches0, "rows_per_s": round(n_rows / (med * 1e-3), 1)}


def columns_entry(torch, rws, stream, l2_bytes, peak, R=4096, C=4096, dtype=wl.F32):
    """softmax_strided down the columns of a row-major R x C matrix (row
    strides 1, column strides C), over rotating input/output sets."""
    w = wl.random_rows(R, C, dtype=dtype, seed=12, scale=3.0)
    dt = torch_dtype(dtype, torch)
    x = torch.from_numpy(w.data if dtype == wl.F32 else w.data.view(np.int16)).cuda()
    x = x if dtype == wl.F32 else x.view(dt)
    esz = 4 if dtype == wl.F32 else 2
    algo = 2 * R * C * esz
    n_sets = max(1, -(-L2_FACTOR * l2_bytes // algo))
    sets = [(x if i == 0 else x.clone(), torch.empty_like(x)) for i in range(n_sets)]
    call = rws.lib().softmax_strided
    args = [(a.data_ptr(), b.data_ptr(), C, R, 1, C, 1, C, dtype, stream.cuda_stream)
            for a, b in sets]
    for i in range(5):
        if call(*args[i % n_sets]) != rws.OK:
            raise RuntimeError("softmax_strided failed")
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = rws.launch_count()
    hold_stream(torch, 50)
    a.record(stream)
    for i in range(50):
        call(*args[i % n_sets])
    b.record(stream)
    torch.cuda.synchronize()
    med = a.elapsed_time(b) / 50
    gbs = algo / (med * 1e-3) / 1e9
    return {"shape": [R, C], "dtype": DTYPE_NAMES[dtype],
            "op": "softmax_strided down the columns (rows of the softmax = columns)",
            "algorithmic_bytes": algo, "mean_ms": round(med, 5), "GB/s": round(gbs, 1),
            "frac_of_measured_peak": round(gbs / peak, 4),
            "launches": rws.launch_count() - launches0}


def tensor_peak():
    """Measured dense bf16 tensor rate (burst), TFLOP/s, and its kind."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, ValueError, KeyError):
        return 1900.0, "fallback"


def attention_entry(torch, rws, stream, bh=64, n=4096, d=128, causal=False, dtype=wl.BF16,
                    impl=0):
    """softmax_attention_forward on seeded N(0,1) inputs: the (m, l) recurrence
    inside attention; FLOPs 4 * bh * n * n * d (halved with the causal mask)."""
    qb, kb, vb = wl.attention_inputs(bh, n, n, d, dtype, seed=21)
    dt = torch_dtype(dtype, torch)
    tq, tk, tv = (torch.from_numpy(a.view(np.int16)).cuda().view(dt) for a in (qb, kb, vb))
    to = torch.empty_like(tq)
    call = rws.lib().softmax_attention_forward
    opt = rws.AttentionOptions(1.0 / (d ** 0.5), 1 if causal else 0, 0, impl)
    import ctypes
    args = (tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), to.data_ptr(), None, bh, n, n, d, dtype,
            ctypes.byref(opt), stream.cuda_stream)
    for _ in range(3):
        if call(*args) != rws.OK:
            raise RuntimeError("softmax_attention_forward failed")
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    steps = 10
    hold_stream(torch, steps)
    a.record(stream)
    for _ in range(steps):
        call(*args)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    flops = 4.0 * bh * n * n * d * (0.5 if causal else 1.0)
    tf = flops / (ms * 1e-3) / 1e12
    peak, kind = tensor_peak()
    return {"shape": {"batch_heads": bh, "n_q": n, "n_k": n, "head_dim": d},
            "dtype": DTYPE_NAMES[dtype], "causal": causal,
            "kernel": {1: "attention_mma_kernel (mma.sync m16n8k16)",
                       2: "attention_tc_kernel (tcgen05.mma, TMEM accumulators)"}.get(
                           impl, "attention_pp_kernel (tcgen05.mma, two query tiles ping-pong, "
                                 "TMA operands with 128-byte swizzle)"),
            "mean_ms": round(ms, 4),
            "TFLOP/s": round(tf, 1), "frac_of_%s_bf16_peak" % kind: round(tf / peak, 4)}


def graph_entry(torch, rws, stream, l2_bytes, peak, name="small_f32", calls=200):
    """A launch-bound workload replayed from a CUDA graph of `calls`
    softmax_rows calls over rotating input/output sets (launch overhead paid
    once per replay instead of once per call)."""
    w = wl.make(name)
    sets = device_buffers(w, torch, l2_bytes)
    call = rws.lib().softmax_rows
    for x, y in sets[:3]:                                  # first calls outside capture
        call(x.data_ptr(), y.data_ptr(), w.n_rows, w.n_cols, w.in_row_stride,
             w.out_row_stride, w.dtype, stream.cuda_stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=cap):
        h = torch.cuda.current_stream().cuda_stream
        for i in range(calls):
            x, y = sets[i % len(sets)]
            if call(x.data_ptr(), y.data_ptr(), w.n_rows, w.n_cols, w.in_row_stride,
                    w.out_row_stride, w.dtype, h) != rws.OK:
                raise RuntimeError("softmax_rows failed under capture")
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    reps = 10
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    hold_stream(torch, reps)
    a.record()
    for _ in range(reps):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    per_call = a.elapsed_time(b) / (reps * calls)
    gbs = w.algorithmic_bytes / (per_call * 1e-3) / 1e9
    return {"shape": [w.n_rows, w.n_cols], "calls_per_graph": calls,
            "mean_ms_per_call": round(per_call, 5), "GB/s": round(gbs, 1),
            "frac_of_measured_peak": round(gbs / peak, 4)}


def time_e2e(w: wl.Workload, steps: int, warmup: int, torch, rws, stream, staged: bool):
    """softmax_rows_host on pinned host buffers, timed over `steps` calls.

    direct (staged=False): the kernel reads the pinned host input and writes
    the pinned host output over the host link (no device buffers);
    staged: H2D copy into device buffers, kernel, D2H copy, on one stream."""
    dt = torch_dtype(w.dtype, torch)
    if w.dtype == wl.F32:
        h_in = torch.from_numpy(w.data).pin_memory()
    else:
        h_in = torch.from_numpy(w.data.view(np.int16)).view(dt).pin_memory()
    h_out = torch.empty(max(w.out_elems, 1), dtype=dt).pin_memory()
    if staged:
        d_in = torch.empty(w.n_rows * w.n_cols, dtype=dt, device="cuda")
        d_out = torch.empty_like(d_in)
        dp_in, dp_out = d_in.data_ptr(), d_out.data_ptr()
    else:
        dp_in = dp_out = None
    args = (h_in.data_ptr(), h_out.data_ptr(), w.n_rows, w.n_cols, w.in_row_stride,
            w.out_row_stride, w.dtype, dp_in, dp_out, stream.cuda_stream)
    call = rws.lib().softmax_rows_host
    for _ in range(warmup):
        st = call(*args)
        if st != rws.OK:
            raise RuntimeError("softmax_rows_host: " + rws.status_string(st))
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        call(*args)
    b.record(stream)
    b.synchronize()
    ms = a.elapsed_time(b) / steps
    esz = w.elem_bytes
    return ms, w.n_rows * w.n_cols * esz, w.n_rows * w.n_cols * esz


def cpu_oracle_time(w: wl.Workload, reps: int):
    import oracle
    oracle.load()
    ts = []
    for _ in range(reps):
        t0 = time.perf_counter()
        oracle.softmax_rows(w.data, w.n_rows, w.n_cols, w.in_row_stride, w.dtype)
        ts.append(time.perf_counter() - t0)
    return statistics.median(ts)


def cpu_model() -> str:
    """The host CPU's name from /proc/cpuinfo (x86 "model name"; on Arm the
    implementer and part numbers), else the platform's machine string."""
    import platform
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
    except OSError:
        return platform.machine()
    fields = {}
    for line in info.splitlines():
        k, _, v = line.partition(":")
        fields.setdefault(k.strip(), v.strip())
    if "model name" in fields:
        return fields["model name"]
    if "CPU part" in fields:
        return "%s, CPU implementer %s, part %s" % (platform.machine(),
                                                    fields.get("CPU implementer", "?"),
                                                    fields["CPU part"])
    return platform.machine()


def torch_cpu_time(w: wl.Workload, reps: int):
    """Median time of torch.softmax over the workload's rows on the host, fp32,
    with every intra-op thread torch has (the library's own CPU kernel, a
    context figure beside the single-threaded oracle).  None for 16-bit
    workloads (torch's CPU bf16 softmax is not the fp32 figure asked for)."""
    import torch
    if w.dtype != wl.F32 or w.n_rows == 0:
        return None
    item = w.data.itemsize
    x = torch.from_numpy(np.lib.stride_tricks.as_strided(
        w.data, shape=(w.n_rows, w.n_cols), strides=(w.in_row_stride * item, item)).copy())
    torch.softmax(x, dim=-1)                             # warm-up
    ts = []
    for _ in range(reps):
        t0 = time.perf_counter()
        torch.softmax(x, dim=-1)
        ts.append(time.perf_counter() - t0)
    return statistics.median(ts)


def run_ours(args):
    import torch
    import row_wise_softmax_gb300 as rws

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    rws.build()
    rws.lib()
    stream = torch.cuda.current_stream()
    l2_bytes = int(torch.cuda.get_device_properties(local).L2_cache_size)
    peak, peak_kind = measured_peak()

    w = wl.make(args.workload)
    plan = rws.plan(w.n_rows, w.n_cols, in_row_stride=w.in_row_stride,
                    out_row_stride=w.out_row_stride, dtype=w.dtype)
    options, bytes_step = None, w.algorithmic_bytes
    workload_key = args.workload
    if args.mask_from_indices:
        options, bytes_step = fused_causal_setup(w, rws)
        workload_key = "causal_bf16_mask_from_indices"

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    bufs = device_buffers(w, torch, l2_bytes)
    barrier()
    with ClockSampler(local) as clk:
        t_wall0 = time.perf_counter()
        total_ms, launches = time_device(w, bufs, args.steps, args.warmup, torch, rws, stream,
                                         options)
        wall = time.perf_counter() - t_wall0
        # Keep the sampled window at least ~1.5 s: repeat the same step (not
        # counted) if the timed steps were shorter than that.
        extra = 0
        while (not args.no_clock_window and time.perf_counter() - t_wall0 < 1.5
               and extra < 400000):
            time_device(w, bufs, 2000, 0, torch, rws, stream, options)
            extra += 2000
    barrier()
    total_ms = max_over_ranks(total_ms, world, "cuda")
    ms_per_step = total_ms / args.steps
    value = world * bytes_step * args.steps / (total_ms * 1e-3) / 1e9
    # One softmax kernel per step: average launch duration = timed region / launches.
    achieved = bytes_step * launches / (total_ms * 1e-3) / 1e9
    traffic, traffic_src = committed_traffic(plan, workload_key)

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32",        # the arithmetic type (bf16 workloads compute in fp32 too)
        "data": WORKLOAD_DATA[args.workload],
        "config": {"workload": workload_label(w, options is not None),
                   "n_rows": w.n_rows, "n_cols": w.n_cols, "bytes_per_step": bytes_step,
                   "l2": "inputs larger than L2: %d rotating input/output sets (%.0f MB, "
                         ">= %dx the %.0f MB L2), steps back to back" % (
                             len(bufs), len(bufs) * (bytes_step / 1e6), L2_FACTOR, l2_bytes / 1e6),
                   "parallelism": "rows sharded per rank, no exchange" if world > 1 else "1 GPU",
                   "plan": str(plan)},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_kind": peak_kind, "traffic": traffic,
                     "kernel": kernel_of(plan)[0],
                     "traffic_source": traffic_src if traffic else traffic_src},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "copy_same_bytes": copy_calibration(w, bufs, torch, stream, peak),
        "wall_s_timed_region": round(wall, 3),
    }
    if traffic:
        result["roofline"]["traffic_over_algorithmic"] = round(traffic / bytes_step, 4)

    if rank == 0 and not args.no_e2e:
        n = max(3, min(args.steps, 20))
        ms, bi, bo = time_e2e(w, n, 2, torch, rws, stream, staged=False)
        result["e2e"] = {"value": round(bytes_step / (ms * 1e-3) / 1e9, 1), "unit": UNIT,
                         "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
                         "ms_per_step": round(ms, 4),
                         "api": "softmax_rows_host, direct mode: the kernel reads the pinned "
                                "host input and writes the pinned host output (no staging)"}
        ms, bi, bo = time_e2e(w, n, 2, torch, rws, stream, staged=True)
        result["e2e_staged"] = {"value": round(bytes_step / (ms * 1e-3) / 1e9, 1), "unit": UNIT,
                                "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
                                "ms_per_step": round(ms, 4),
                                "api": "softmax_rows_host, staged mode: H2D copy, kernel, D2H "
                                       "copy on one stream"}
    if rank == 0 and not args.no_cpu:
        reps = 3
        t = cpu_oracle_time(w, reps)
        result["cpu_baseline"] = {
            "value": round(bytes_step / t / 1e9, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": "the full %d x %d workload, median of %d runs of the double-precision "
                      "single-threaded oracle" % (w.n_rows, w.n_cols, reps),
            "seconds_per_step": round(t, 4)}
        try:
            import torch as _t
            tt = torch_cpu_time(w, 5)
            if tt is not None:
                result["cpu_baseline"]["torch_cpu_all_cores"] = {
                    "value": round(bytes_step / tt / 1e9, 3), "unit": UNIT,
                    "threads": _t.get_num_threads(), "cpu_count": os.cpu_count(),
                    "cpu": cpu_model(), "seconds_per_step": round(tt, 5),
                    "what": "torch.softmax(x, dim=-1), fp32, on the host, median of 5"}
        except Exception as e:                       # context figure only: never fatal
            result["cpu_baseline"]["torch_cpu_all_cores"] = {"unavailable": str(e)[:200]}
    if rank == 0 and not args.no_per_config:
        per = {}

        cpu_oracle = {}

        def workload_entry(name):
            wc = w if name == args.workload else wl.make(name)
            pc = rws.plan(wc.n_rows, wc.n_cols, in_row_stride=wc.in_row_stride,
                          out_row_stride=wc.out_row_stride, dtype=wc.dtype)
            bc = bufs if name == args.workload else device_buffers(wc, torch, l2_bytes)
            tot, _ = time_device(wc, bc, 50, 5, torch, rws, stream)
            each = time_each_step(wc, bc, 50, torch, rws, stream)
            cal = copy_calibration(wc, bc, torch, stream, peak)
            del bc
            mean = tot / 50
            gbs = wc.algorithmic_bytes / (mean * 1e-3) / 1e9
            entry = {"shape": [wc.n_rows, wc.n_cols], "dtype": DTYPE_NAMES[wc.dtype],
                     "workload": workload_label(wc),
                     "path": pc.path_name, "kernel": kernel_of(pc)[0], "plan": str(pc),
                     "mean_ms": round(mean, 5),
                     "median_ms_single": round(statistics.median(each), 5),
                     "p95_ms_single": round(percentile(each, 0.95), 5),
                     "copy_same_bytes_GB/s": cal["GB/s"] if cal else None,
                     "GB/s": round(gbs, 1), "frac_of_measured_peak": round(gbs / peak, 4),
                     "frac_of_8000": round(gbs / 8000.0, 4),
                     "rows_per_s": sig(wc.n_rows / (mean * 1e-3))}
            rec, src = committed_record(pc, name)
            if rec and rec.get("gpu_time_us"):
                ncu_gbs = wc.algorithmic_bytes / (rec["gpu_time_us"] * 1e-6) / 1e9
                entry["ncu_one_launch"] = {
                    "gpu_time_us": rec["gpu_time_us"], "GB/s": round(ncu_gbs, 1),
                    "frac_of_measured_peak": round(ncu_gbs / peak, 4),
                    "traffic_over_algorithmic": round(
                        rec["dram_bytes_per_launch"] / wc.algorithmic_bytes, 4),
                    "source": src}
            else:
                entry["ncu_one_launch"] = {"unavailable": src}
            if name in CONFIG_TAGS and not args.no_cpu:
                t = cpu_oracle_time(wc, 3)
                cpu_oracle[name] = t
                entry["cpu_oracle"] = {"seconds": round(t, 4), "cores": 1, "runs": 3,
                                       "GB/s": sig(wc.algorithmic_bytes / t / 1e9),
                                       "rows_per_s": sig(wc.n_rows / t)}
            return entry

        entries = [(name, lambda name=name: workload_entry(name))
                   for name in wl.NAMES + wl.EXTRA_NAMES]
        entries.append(("causal_bf16_mask_from_indices",
                        lambda: fused_causal_entry(torch, rws, stream, l2_bytes, peak)))
        entries.append(("backward_f32_4096x4096",
                        lambda: backward_entry(torch, rws, stream, l2_bytes, peak)))
        entries.append(("small_f32_cuda_graph",
                        lambda: graph_entry(torch, rws, stream, l2_bytes, peak)))
        entries.append(("attention_tcgen05_pingpong_bf16_64x4096x4096_d64_causal",
                        lambda: attention_entry(torch, rws, stream, d=64, causal=True, impl=3)))
        for impl, tag in ((3, "tcgen05_pingpong"), (2, "tcgen05"), (1, "mma_sync")):
            entries.append(("attention_%s_bf16_64x4096x4096_d128" % tag,
                            lambda impl=impl: attention_entry(torch, rws, stream, impl=impl)))
            entries.append(("attention_%s_bf16_64x4096x4096_d128_causal" % tag,
                            lambda impl=impl: attention_entry(torch, rws, stream, causal=True,
                                                              impl=impl)))
            entries.append(("attention_%s_bf16_64x4096x4096_d64" % tag,
                            lambda impl=impl: attention_entry(torch, rws, stream, d=64,
                                                              impl=impl)))
        entries.append(("columns_f32_4096x4096",
                        lambda: columns_entry(torch, rws, stream, l2_bytes, peak)))
        entries.append(("columns_bf16_8192x4096",
                        lambda: columns_entry(torch, rws, stream, l2_bytes, peak, 8192, 4096,
                                              wl.BF16)))
        entries.append(("backward_bf16_32768x1024",
                        lambda: backward_entry(torch, rws, stream, l2_bytes, peak, 32768, 1024,
                                               wl.BF16)))
        only = set(args.per_config_only.split(",")) if args.per_config_only else None
        if only is not None and not only <= {k for k, _ in entries}:
            raise SystemExit("--per-config-only: unknown entries %s" %
                             sorted(only - {k for k, _ in entries}))
        for key, fn in entries:
            if only is None or key in only:
                per[key] = fn()
        result["per_config"] = per
        # The five configurations again, compactly, as the line's last key
        # (a reader that keeps only the end of the line still sees them).
        result["configs"] = configs_block(per, peak)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)


def configs_block(per, peak):
    """C1..C5 in a few keys each: GB/s and rows/s of the back-to-back steps,
    their fraction of the measured copy peak and of 8000 GB/s, the median and
    95th percentile of singly timed steps, the committed one-launch ncu
    figures (fraction of the peak, DRAM traffic over algorithmic bytes) and
    the single-threaded CPU oracle's time."""
    out = {"peak_GB/s": peak, "cpu": "oracle, double, 1 thread, median of 3"}
    for name, tag in CONFIG_TAGS.items():
        e = per.get(name)
        if e is None:
            continue
        c = {"w": "%s %dx%d %s" % (name, e["shape"][0], e["shape"][1], e["dtype"]),
             "GB/s": e["GB/s"], "frac": e["frac_of_measured_peak"],
             "frac8000": e["frac_of_8000"], "rows/s": e["rows_per_s"],
             "med_ms": e["median_ms_single"], "p95_ms": e["p95_ms_single"]}
        n = e.get("ncu_one_launch", {})
        if "frac_of_measured_peak" in n:
            c["ncu_frac"] = n["frac_of_measured_peak"]
            c["traffic"] = n["traffic_over_algorithmic"]
        if "cpu_oracle" in e:
            c["cpu_s"] = e["cpu_oracle"]["seconds"]
            c["cpu_GB/s"] = e["cpu_oracle"]["GB/s"]
        out[tag] = c
    return out


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = wl.make(HEADLINE)
    import oracle
    oracle.build()
    oracle.load()
    for _ in range(args.warmup):
        cpu_oracle_time(w, 1)
    ts = [cpu_oracle_time(w, 1) for _ in range(args.steps)]
    total = sum(ts)
    value = w.algorithmic_bytes * args.steps / total / 1e9
    sample = ("the full %d x %d workload per step, double-precision single-threaded oracle"
              % (w.n_rows, w.n_cols))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_label(w)},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-per-config", action="store_true")
    ap.add_argument("--per-config-only", default="",
                    help="comma-separated per_config entries to time (default: all)")
    ap.add_argument("--no-clock-window", action="store_true",
                    help="do not extend the clock-sampling window past the timed steps")
    ap.add_argument("--workload", default=HEADLINE, choices=list(wl.NAMES + wl.EXTRA_NAMES),
                    help="workload timed as the step (default: the headline)")
    ap.add_argument("--mask-from-indices", action="store_true",
                    help="with --workload causal_bf16: time softmax_rows_ex with the causal "
                         "mask computed from indices and a 1/sqrt(64) scale (no end-to-end "
                         "or CPU legs)")
    args = ap.parse_args()
    if args.mask_from_indices:
        if args.workload != "causal_bf16":
            ap.error("--mask-from-indices applies to --workload causal_bf16")
        args.no_e2e = args.no_cpu = True
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
