"""The N > 1 path of the bench (independent replicas, one per GPU) reduced over
two gloo ranks on the CPU: the job's value is the tokens of all ranks over the
slowest rank's step time; no GPU is involved."""
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


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r: step 6.5 + r ms, 6 - r tokens per step, e2e step 7 + r ms
    mean_ms, tps = 6.5 + rank, 6.0 - rank
    e2e_s = (7.0 + rank) / 1e3
    out = bench.reduce_over_ranks(mean_ms, tps, e2e_s, tps / e2e_s, True)
    q.put((rank, out))
    dist.destroy_process_group()


def test_replica_reduction_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    for r in (0, 1):
        slow_ms, value, e2e = res[r]
        assert slow_ms == pytest.approx(7.5)
        assert value == pytest.approx((6.0 + 5.0) / 7.5e-3)
        assert e2e == pytest.approx((6.0 + 5.0) / 8.0e-3)


def test_single_rank_reduction_is_the_local_rate():
    import bench
    assert bench.reduce_over_ranks(5.0, 6.0, 0.006, 1000.0, False) == (5.0, 1200.0, 1000.0)
