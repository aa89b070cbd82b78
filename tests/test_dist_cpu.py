"""Multi-process host logic of the benchmark on CPU (gloo, world_size 2).

The attention path shards without any exchange: with N GPUs every rank runs its own replica
of the workload and only the timings meet, max-reduced across ranks.  These tests run that
host-side logic in two CPU processes."""
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
    w, r, _ = bench.dist_init()
    assert (w, r) == (world, rank) and dist.get_backend() == "gloo"
    t = bench.max_over_ranks(1.5 + rank, w)       # each rank's step time
    bench.barrier(w)
    from programming_flashattention_fwd_gb300.inputs import WORKLOADS
    wl = WORKLOADS["mha_b1_h2_s128_d64"]
    seed = (wl.with_(seed=wl.seed + 7919 * rank) if rank else wl).seed
    out[rank] = (t, seed)
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_max_over_ranks_and_replica_seeds():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
        assert p.exitcode == 0
    assert out[0][0] == out[1][0] == 2.5          # max of 1.5 and 2.5 on every rank
    assert out[0][1] != out[1][1]                 # replicas draw independent inputs


def test_single_process_helpers_are_identity():
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    bench.barrier(1)
