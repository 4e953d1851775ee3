"""The benchmark's multi-GPU reduction (replicas: max time over ranks, the
ranks' bytes summed) on a world of 2 CPU processes over gloo."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

from conftest import ROOT  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [2.0, 3.5][rank]
    mx = bench._max_over_ranks(ms, dist, torch.device("cpu"))
    value = bench.replica_value(8_041_103_360, world, mx)
    out[rank] = (mx, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world, port = 2, _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 3.5
    assert res[0][1] == res[1][1] == pytest.approx(2 * 8_041_103_360 / 3.5e-3 / 1e9)
