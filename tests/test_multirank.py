"""The bench's multi-rank plumbing on the CPU: two gloo ranks (world size 2), as
torch.distributed.run would start them for `bench.py --gpus 2`.  Each rank is an
independent replica (no collective on the data path); the ranks meet only at the barrier
around the timed region and at the max-over-ranks of the step time, and only rank 0 runs
the reference arm's oracle timing."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import bench
    import torch.distributed as dist
    w, r, local = bench.dist_setup(None)
    assert (w, r, local) == (world, rank, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    # each replica's own step time; the job's is the slowest
    out[rank] = bench.max_over_ranks(w, 1.5 + rank)
    # the reference arm: rank 0 alone would time the oracle, the others return at once
    calls = []
    orig = bench.oracle_prefill_sample
    bench.oracle_prefill_sample = lambda *a, **k: calls.append(a) or (1.0, {"rows": 1, "seconds": 1.0})
    try:
        if rank != 0:
            bench.run_reference(None, None, w, r)
            assert calls == []
    finally:
        bench.oracle_prefill_sample = orig
    bench.barrier(w)
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_agree_on_the_slowest_step():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn", join=True)
    assert dict(out) == {0: 2.5, 1: 2.5}
