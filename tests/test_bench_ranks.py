"""The bench's multi-rank host logic on CPU (gloo, world_size 2): max of the
elapsed times and sum of the work over ranks, as bench.py reports them."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    assert bench.dist_env() == (world, rank, rank)
    secs, units = bench.aggregate(1.0 + rank, 10.0 * (rank + 1), world)
    q.put((rank, secs, units))
    dist.destroy_process_group()


def test_aggregate_is_max_time_and_sum_of_work():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for _, secs, units in res:
        assert secs == 2.0
        assert units == 30.0


def test_single_rank_aggregate_is_identity():
    import bench
    assert bench.aggregate(1.5, 7.0, 1) == (1.5, 7.0)


def test_reference_arm_rank_nonzero_does_nothing(monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.run_reference(bench.main.__defaults__ if False else _Args()) is None


class _Args:
    steps = 1
    warmup = 0
    cpu_seconds = 0.1


def test_flop_and_byte_counts():
    import bench
    assert bench.prefill_flops(1, 16, 8192, 128) == 4 * 16 * 8192 ** 2 * 128
    assert bench.prefill_flops(1, 1, 10, 64, causal=True) == 2 * 100 * 64
    assert bench.decode_bytes([1, 3], 14, 64) == 2 * 14 * 4 * 64 * 2
