"""CPU: the multi-GPU path is replicas only (sessions shard, no collective on
the data path); what the ranks share is the timing.  Two gloo ranks on the
host check the max-over-ranks reduction and the whole-job throughput, and
that the reference arm's non-zero ranks exit without work."""
import os
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # rank r took (10 + r) ms per step and (12 - r) ms end to end
        ms, e2e = bench.max_over_ranks([10.0 + rank, 12.0 - rank], dist)
        out[rank] = (ms, e2e, bench.job_throughput(world, 80, ms))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_replica():
    world, port = 2, 29517 + os.getpid() % 1000
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        ms, e2e, value = out[r]
        assert ms == 11.0 and e2e == 12.0
        assert value == pytest.approx(2 * 80 / 0.011)


def test_single_process_reduction_is_identity():
    import bench
    assert bench.max_over_ranks([3.0, 4.0]) == [3.0, 4.0]
    assert bench.job_throughput(1, 80, 10.0) == pytest.approx(8000.0)


def test_reference_arm_non_zero_rank_does_no_work(monkeypatch, capsys):
    import bench
    import synth
    monkeypatch.setenv("RANK", "1")

    class A:
        S, steps, warmup, gpus = 80, 1, 1, 2
    bench.run_reference(A(), synth.SEVEN_B)
    assert capsys.readouterr().out == ""
