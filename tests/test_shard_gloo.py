"""The adapter-drift workload sharded by sequence, on the CPU (gloo ranks):
its batch of 4 sequences are independent problems (own cache, selection and
boundary states), so each rank owns a contiguous shard and nothing crosses
between ranks on the data path ("CacheReforge", Bounded Recovery: the repair
is per sequence).  Checked here: every sequence lands on exactly one rank, the
ranks' row counts and row-layer units sum to the single-process totals, the
ranks' outputs assemble in sequence order into the single-process result, and
the job throughput takes the slowest rank's time and the summed units."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from selective_kv_cache_gb300 import workloads as wl
    from selective_kv_cache_gb300.harness import shard_sequences

    w = wl.WORKLOADS["qwen1p5b_drift"]
    lo, hi = shard_sequences(w.batch, world, rank)
    shards = bench.gather_shards(lo, hi, world)
    # the rank's own inputs: the full batch's selections, sliced to its shard
    pos = wl.make_positions(w)[lo:hi]
    rows = sum(len(p) for p in pos)
    r0, r1 = w.range_layers
    S = w.n_tokens - w.suffix_start
    units = rows * (w.model.n_layers - (r1 - r0)) + (hi - lo) * S * (r1 - r0)
    # a per-sequence output standing in for the refreshed rows: the sorted
    # positions, gathered in rank order
    mine = torch.from_numpy(np.concatenate([np.sort(p) for p in pos]).astype(np.int64))
    sizes = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
    dist.all_gather(sizes, torch.tensor([mine.numel()]))
    cap = int(max(n.item() for n in sizes))          # gloo gathers equal sizes: pad, then trim
    parts = [torch.zeros(cap, dtype=torch.int64) for _ in range(world)]
    dist.all_gather(parts, torch.cat([mine, torch.zeros(cap - mine.numel(), dtype=torch.int64)]))
    parts = [p[:int(n.item())] for p, n in zip(parts, sizes)]
    t_max, total, value = bench.sharded_throughput(0.5 + 0.25 * rank, units, world)
    out.put((rank, lo, hi, rows, units, shards, torch.cat(parts).numpy(), t_max, total, value))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_sequence_shards_cover_the_batch_once(world):
    from selective_kv_cache_gb300 import workloads as wl

    w = wl.WORKLOADS["qwen1p5b_drift"]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in ps:
        p.start()
    res = sorted([q.get(timeout=120) for _ in range(world)], key=lambda r: r[0])
    for p in ps:
        p.join(timeout=120)
        assert p.exitcode == 0
    owner = np.full(w.batch, -1)
    for rank, lo, hi, *_ in res:
        assert np.all(owner[lo:hi] == -1), "a sequence on two ranks"
        owner[lo:hi] = rank
    assert np.all(owner >= 0), "a sequence on no rank"
    assert list(owner) == sorted(owner), "shards are contiguous and in rank order"
    # single-process totals
    pos = wl.make_positions(w)
    r0, r1 = w.range_layers
    S = w.n_tokens - w.suffix_start
    rows1 = sum(len(p) for p in pos)
    units1 = rows1 * (w.model.n_layers - (r1 - r0)) + w.batch * S * (r1 - r0)
    assert sum(r[3] for r in res) == rows1
    assert sum(r[4] for r in res) == units1
    whole = np.concatenate([np.sort(p) for p in pos])
    for rank, lo, hi, rows, units, shards, assembled, t_max, total, value in res:
        assert shards == [(r[1], r[2]) for r in res]          # every rank sees every shard, in rank order
        np.testing.assert_array_equal(assembled, whole)     # outputs assemble in sequence order
        assert t_max == pytest.approx(0.5 + 0.25 * (world - 1))
        assert total == units1 and value == pytest.approx(units1 / t_max)


def test_shard_sequences_edges():
    from selective_kv_cache_gb300.harness import shard_sequences

    assert [shard_sequences(4, 1, 0)] == [(0, 4)]
    assert [shard_sequences(4, 4, r) for r in range(4)] == [(0, 1), (1, 2), (2, 3), (3, 4)]
    assert [shard_sequences(5, 2, r) for r in range(2)] == [(0, 3), (3, 5)]
    assert shard_sequences(2, 4, 3) == (2, 2)                 # more ranks than sequences: an empty shard
    with pytest.raises(ValueError):
        shard_sequences(4, 2, 2)
