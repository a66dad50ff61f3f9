"""Cross-rank aggregation of bench.py on two gloo ranks (CPU): the job time is the
slowest rank's, and throughput counts every rank's bytes (weak scaling)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local = (1.0 + rank, 0.4 + rank, 0.6)            # rank 1 is slower
    got = bench.reduce_step_times(*local, pg=dist, device="cpu")
    q.put((rank, got, bench.job_throughput_gbs(world, 10, 1 << 20, got[0])))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, gbs in res:
        assert got == (2.0, 1.4, 0.6)
        assert gbs == pytest.approx(2 * 10 * 4 * (1 << 20) / 2.0 / 1e9)


def test_single_process_is_identity():
    import bench
    assert bench.reduce_step_times(1.5, 1.0, 0.5) == (1.5, 1.0, 0.5)
