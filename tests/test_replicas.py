"""Multi-process host logic of the benchmark's replica mode (N ranks, one
independent verify call stream each, no collective on the data path): two
gloo ranks on the CPU agree on the slowest rank's time and on the summed
throughput."""
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [10.0, 12.5][rank]
    value, ms_max = bench.replica_value(71_337_984, 100, ms, world)
    bench.barrier(world)
    out.put((rank, value, ms_max))
    dist.destroy_process_group()


def test_replica_value_two_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    want = 2 * 71_337_984 * 100 / (12.5e-3) / 1e9
    for rank, value, ms_max in res:
        assert ms_max == 12.5
        assert value == pytest.approx(want, rel=1e-12)


def test_replica_value_single_rank():
    import bench
    value, ms_max = bench.replica_value(1_000_000_000, 10, 5.0, 1)
    assert ms_max == 5.0
    assert value == pytest.approx(2000.0)
