"""The bench's multi-rank bookkeeping on CPU (gloo, world size 2).

The path is not sharded across GPUs: under torchrun every rank runs its own
replica; the only cross-rank steps are a barrier around the timed region and
the max over ranks of the elapsed time, checked here with gloo ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    out[rank] = bench.max_over_ranks(10.0 * (rank + 1), world)
    bench.barrier(world)
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == 20.0 and out[1] == 20.0


def test_reference_arm_only_rank0_works():
    class A:
        workload = "tiny"
        steps = 1
        warmup = 0
    assert bench.run_reference(A(), world=2, rank=1) is None
