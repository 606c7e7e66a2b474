"""The multi-GPU path of the benchmark on CPU: two gloo ranks, each with its own layer; the
job's time is the slowest rank's and its throughput counts every rank's units."""
import os

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    try:
        layer = bench.layer_of_rank(rank)
        ms = [10.0 + 5.0 * rank, 20.0 - rank]            # rank 1 is slower on the first timing
        got = bench.max_over_ranks(ms, world, "cpu")
        thr = bench.job_throughput(432000, world, got[0])
        out[rank] = (layer, got, thr)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = 29500 + os.getpid() % 1000
    ps = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(120)
        assert p.exitcode == 0
    assert out[0][0] == 0 and out[1][0] == 1                     # distinct layers
    assert out[0][1] == out[1][1] == [15.0, 20.0]                # maxima agree on every rank
    assert out[0][2] == pytest.approx(2 * 432000 / 0.015)        # both ranks' units / slowest time


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks([3.0, 4.0], 1) == [3.0, 4.0]
    assert bench.job_throughput(100, 1, 1000.0) == 100.0
