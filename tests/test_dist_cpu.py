"""Multi-rank logic of the benchmark on the CPU (gloo, world size 2): rows
shard contiguously with no overlap and no gap, and the step time reported is
the maximum over ranks.  No GPU and no data-path collective are involved."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, total_rows, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    lo, hi = bench.shard_rows(total_rows, world, rank)
    t = 1.0 + rank * 0.5                      # per-rank "step time"
    worst = bench.max_over_ranks(t, dist)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, lo, hi, worst))


@pytest.mark.parametrize("total_rows", [65536 * 2, 131073, 3])
def test_shards_and_max_over_ranks(total_rows):
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, total_rows, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    ranges = [(lo, hi) for _, lo, hi, _ in res]
    assert ranges[0][0] == 0 and ranges[-1][1] == total_rows
    assert all(ranges[i][1] == ranges[i + 1][0] for i in range(world - 1))
    sizes = [hi - lo for lo, hi in ranges]
    assert max(sizes) - min(sizes) <= 1
    assert all(w == 1.5 for *_, w in res)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(2.5, None) == 2.5
    assert bench.shard_rows(10, 1, 0) == (0, 10)
