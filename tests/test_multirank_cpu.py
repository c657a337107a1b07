"""The benchmark's multi-rank host logic on CPU (gloo, world size 2).

Tokens are independent, so ranks exchange no data; the only cross-rank steps
are the barrier around the timed region and the max over ranks of the
elapsed time.  These run here as two gloo processes."""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    m = bench.max_over_ranks(10.0 + 5.0 * rank, w)
    out[rank] = m
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_max_over_ranks_and_barrier_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
    assert all(p.exitcode == 0 for p in procs)
    assert out[0] == out[1] == 15.0


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    import bench
    args = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    assert bench.run_reference(args, rank=1, world=2) == 0
