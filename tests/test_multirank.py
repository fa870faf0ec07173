"""The bench's multi-GPU path on CPU: two gloo ranks, each serving its own batch, with the
slowest rank setting the time (the only collective, outside the timed region)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, queue):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        times = bench.slowest_over_ranks([1.0 + rank, 5.0 - rank, 3.0], world)
        step = bench.replica_step("llama8b_gqa_decode", rank, world)
        queue.put((rank, times, step.seed, int(step.decode.context_lens.sum())))
    finally:
        dist.destroy_process_group()


def test_two_ranks_weak_scaling_and_slowest_rank_time():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(queue.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, t0, seed0, tok0), (r1, t1, seed1, tok1) = results
    assert t0 == t1 == [2.0, 5.0, 3.0]       # the slowest rank's time, everywhere
    assert seed0 != seed1                     # each replica its own batch ...
    assert tok0 == tok1                       # ... of the same workload shape


def test_single_rank_needs_no_collective():
    import bench
    assert bench.slowest_over_ranks([1.5, 2], 1) == [1.5, 2.0]
    assert bench.replica_step("tiny_decode", 0, 1).seed == 53_000
