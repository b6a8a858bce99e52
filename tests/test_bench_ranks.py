"""The benchmark's multi-rank host logic on CPU (gloo, world size 2): the row
split covers every row exactly once with no exchange, and the job time is the
maximum over ranks."""
import os
import socket

import pytest

import bench

torch = pytest.importorskip("torch")
mp = pytest.importorskip("torch.multiprocessing")


def test_shard_rows_covers_every_row_once():
    for n_rows in (0, 1, 7, 4096, 4097):
        for world in (1, 2, 3, 8):
            spans = [bench.shard_rows(n_rows, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == n_rows
            assert all(spans[i][1] == spans[i + 1][0] for i in range(world - 1))
            sizes = [hi - lo for lo, hi in spans]
            assert max(sizes) - min(sizes) <= 1


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(10.0 + 5.0 * rank, world)
        out[rank] = got
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    world = 2
    with mp.get_context("spawn").Manager() as mgr:   # no fork of a threaded process
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        assert dict(out) == {0: 15.0, 1: 15.0}
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_torch_cpu_context_figure():
    """The optional all-core torch.softmax timing runs on an fp32 workload and
    is skipped (None) for 16-bit ones; the CPU name is a non-empty string."""
    import workloads as wl
    t = bench.torch_cpu_time(wl.make("small_f32"), 2)
    assert t is not None and t > 0
    assert bench.torch_cpu_time(wl.make("short_f32"), 1) > 0        # in-stride 128, 127 columns
    assert bench.torch_cpu_time(wl.make("causal_bf16"), 1) is None
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()
