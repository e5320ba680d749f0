"""The N-GPU bench path on the CPU: N independent replicas, one per rank,
with the job time taken as the maximum over ranks (gloo, world size 2 and 4)
and the whole-job throughput summed over ranks.  The data path has no
collective: the workloads here are single sequences, which run as replicas."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t_max, value = bench.job_throughput(times[rank], 282 * 10, world)
    out.put((rank, t_max, value))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_job_throughput_takes_the_slowest_rank(world):
    times = [0.50 + 0.1 * r for r in range(world)]        # seconds per rank
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank, args=(r, world, port, times, q)) for r in range(world)]
    for p in ps:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in ps:
        p.join(timeout=120)
        assert p.exitcode == 0
    t_slow = max(times)
    for rank, t_max, value in res:
        assert t_max == pytest.approx(t_slow)
        assert value == pytest.approx(282 * 10 * world / t_slow)   # every rank reports the job total


def test_single_rank_needs_no_process_group():
    import bench
    t_max, value = bench.job_throughput(0.25, 282, 1)
    assert t_max == 0.25 and value == pytest.approx(282 / 0.25)
