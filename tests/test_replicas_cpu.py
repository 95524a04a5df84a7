"""The multi-GPU path is replicas only: every rank compresses its own layers,
and the only collectives are the barriers around the timed region and the
max-over-ranks of the step time.  This runs bench.py's aggregation on two
gloo ranks on the CPU (127.0.0.1)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = bench.replica_ms(1.0 + rank, world, "cpu")   # rank 1 is the slower one
    dist.barrier()
    out[rank] = (ms, bench.replica_value(1000, world, ms))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(2, _free_port(), out), nprocs=2, join=True,
                           start_method="spawn")
        res = dict(out)
    assert res[0][0] == res[1][0] == 2.0
    assert res[0][1] == pytest.approx(1000 * 2 / 2e-3)


def test_single_rank_is_local():
    import bench
    assert bench.replica_ms(3.5, 1, "cpu") == 3.5
    assert bench.replica_value(10, 1, 2.0) == pytest.approx(5000.0)
