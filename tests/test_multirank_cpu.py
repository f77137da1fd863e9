"""The benchmark's multi-rank plumbing on CPU with gloo, world size 2: every rank runs an
independent replica of the step (no data-path collective); the job time is the slowest
rank's, and the job value counts every rank's parameters."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms_local = [12.5, 13.25][rank]
    bench.barrier(world)
    ms = bench.max_over_ranks(ms_local, world, device="cpu")
    value = bench.job_value(1_200_000_000, ms, world)
    q.put((rank, ms, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[1] for o in out] == [13.25, 13.25]
    assert out[0][2] == pytest.approx(2 * 1_200_000_000 / 13.25e-3)


def test_single_rank_value():
    import bench
    assert bench.job_value(1000, 1.0, 1) == pytest.approx(1e6)
    assert bench.max_over_ranks(3.0, 1) == 3.0


def _fits_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    need = 10 * 2 ** 30
    # both ranks' hosts have room for both ranks' buffers: run
    a = bench.host_fits(need, world, avail=100 * 2 ** 30, device="cpu")[0]
    # rank 1's host cannot hold both: every rank skips the leg
    b = bench.host_fits(need, world, avail=[100, 30][rank] * 2 ** 30, device="cpu")[0]
    q.put((rank, a, b))
    dist.barrier()
    dist.destroy_process_group()


def test_end_to_end_leg_is_skipped_on_every_rank_or_none():
    """The end-to-end leg pins the gradients in host memory on every rank of a host at
    once; the ranks agree on running it, so that none waits in a collective another one
    skipped."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_fits_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out == [(0, True, False), (1, True, False)]
