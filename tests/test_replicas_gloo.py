"""The multi-GPU path of bench.py is replicas only: each rank runs its own
copy of the layer on its own tokens, and ranks share only a barrier and the
max of their timings.  Two gloo ranks on CPU check that bookkeeping: the
slowest rank's time reaches every rank, the whole-job throughput counts all
ranks' tokens, every rank draws distinct token batches, and the reference
arm runs on rank 0 only."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench
from lmoe_inputs import configs as C


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slow = bench.max_over_ranks(10.0 + 5.0 * rank, world, device="cpu")
        dist.barrier()
        seeds = bench.replica_seeds(C.workload("k3_decode_t64"), rank)
        # the reference arm: ranks other than 0 leave at once, printing nothing
        ref = bench.run_reference(None) if rank != 0 else None
        q.put((rank, slow, seeds, ref))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = {}
    for _ in range(world):
        r, slow, seeds, ref = q.get(timeout=120)
        got[r] = (slow, seeds, ref)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got[0][0] == got[1][0] == 15.0                  # the slowest rank's time, on every rank
    assert not set(got[0][1]) & set(got[1][1])            # distinct token batches per rank
    assert got[1][2] is None


def test_job_throughput_counts_every_rank():
    assert bench.job_throughput(1, 64, 100, 0.5) == pytest.approx(12800.0)
    assert bench.job_throughput(4, 64, 100, 0.5) == pytest.approx(4 * 12800.0)
    assert bench.max_over_ranks(3.5, 1) == 3.5
