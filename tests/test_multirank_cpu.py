"""The N>1 host logic of bench.py on CPU: two gloo ranks, each with its own
step time; both must see the slowest rank's time and the same whole-job
value (weak scaling: bytes per rank x ranks / slowest time)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 10.0 + 5.0 * rank
    slow = bench.max_over_ranks(ms)
    out[rank] = (slow, bench.job_gbs(1e9, world, slow), bench.dist_env())
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        slow, gbs, env = out[r]
        assert slow == 15.0
        assert gbs == pytest.approx(1e9 * 2 / 15e-3 / 1e9)
        assert env == (r, 2, r)


def test_single_process_is_a_no_op():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_gbs(2e9, 1, 1.0) == pytest.approx(2000.0)
