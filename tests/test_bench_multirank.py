"""Host logic of bench.py's multi-GPU replicas, run as world_size-2 gloo
process groups on the CPU: the timed region is the slowest rank's, and the
job value counts every rank's tokens."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        m = bench.max_over_ranks(times[rank])
        out[rank] = (m, bench.job_tokens_per_s(8192, world, m))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_value_two_ranks():
    port = _free_port()
    times = [2.0, 3.5]
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(2, port, times, out), nprocs=2, join=True)
        res = dict(out)
    for r in (0, 1):
        m, v = res[r]
        assert m == 3.5
        assert v == pytest.approx(2 * 8192 / 3.5e-3)


def test_single_process_identity():
    assert bench.max_over_ranks(1.25) == 1.25
    assert bench.job_tokens_per_s(100, 1, 10.0) == pytest.approx(1e4)


@pytest.mark.parametrize("T", [1, 64, 128, 1000, 8192, 8200, 16384])
@pytest.mark.parametrize("parts", [(1, 1, 1, 1), (1, 3, 3, 1), (1, 8, 5, 2), (4, 7, 4, 1)])
def test_pipeline_plan_sizes(T, parts):
    # the end-to-end pipeline's chunks cover the batch once, in order, and
    # every chunk but the last starts and ends on a 128-token block boundary
    sizes = bench.plan_sizes(T, parts)
    assert sum(sizes) == T and all(n > 0 for n in sizes)
    assert all(n % 128 == 0 for n in sizes[:-1])
    assert len(sizes) <= len(parts)
    if T == 8192:
        assert sizes == [8192 * p // sum(parts) for p in parts]
