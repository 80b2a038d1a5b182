"""Multi-rank logic of the benchmark on the CPU (gloo, world size 2): rows
shard contiguously with no overlap and no gap, the step time reported is the
maximum over ranks, and the rows each rank draws and computes (its shard of
one seeded problem, the oracle on those rows) gathered together equal the
single-process result bit for bit.  No GPU, and no collective on the data
path (the gather here is the test's own check)."""
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


def _shard_worker(rank, world, port, q):
    import numpy as np
    import torch
    import torch.distributed as dist

    import nf_inputs
    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = nf_inputs.Workload("dist_small", 301, 72, 264, 1e-5, ("post_ln",), gamma=True, beta=True)
    inp = nf_inputs.workload_shard(w, world, rank, chunk_rows=64)
    lo, hi = inp["rows"]
    y = oracle.get().gemm_postnorm_ln(inp["X"], inp["W"], w.eps, inp["gamma"], inp["beta"])[0]
    sizes = [nf_inputs.shard_rows(world * w.M, world, r) for r in range(world)]
    buf = [torch.zeros((b - a, w.N), dtype=torch.float64) for a, b in sizes]
    dist.all_gather(buf, torch.from_numpy(np.ascontiguousarray(y)))
    dist.barrier()
    dist.destroy_process_group()
    if rank == 0:
        q.put(torch.cat(buf).numpy())


def test_shards_of_one_problem_gather_to_the_whole():
    import numpy as np

    import nf_inputs
    import oracle
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = q.get(timeout=300)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    w = nf_inputs.Workload("dist_small", world * 301, 72, 264, 1e-5, ("post_ln",), gamma=True, beta=True)
    whole = nf_inputs.workload_inputs(w)
    want = oracle.get().gemm_postnorm_ln(whole["X"], whole["W"], w.eps, whole["gamma"], whole["beta"])[0]
    assert got.shape == want.shape
    assert np.array_equal(got, want)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(2.5, None) == 2.5
    assert bench.shard_rows(10, 1, 0) == (0, 10)
