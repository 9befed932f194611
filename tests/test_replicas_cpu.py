"""The bench's multi-GPU mode runs independent replicas (sequences are
independent units; no step exchanges data).  Its only cross-rank logic is the
aggregation of the timed region: max over ranks, throughput summed over every
rank's sequences.  Checked here with two gloo ranks on CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms_local = [40.0, 50.0][rank]          # rank 1 is the slower replica
    ms, value = bench.aggregate_replicas(ms_local, world, B=3, steps=100, device="cpu")
    q.put((rank, ms, value))
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for _, ms, value in got:
        assert ms == 50.0
        assert value == pytest.approx(2 * 3 * 100 / 0.050)


def test_single_replica_is_local_time():
    import bench
    ms, value = bench.aggregate_replicas(20.0, 1, B=1, steps=10, device="cpu")
    assert ms == 20.0 and value == pytest.approx(500.0)
