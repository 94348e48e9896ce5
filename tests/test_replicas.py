"""Host logic of the replica (one process per GPU) path, run as two gloo ranks on the CPU:
rank layout from the launcher's environment, the barrier, the max-over-ranks reduction of the
timed region and the whole-job rate.  No GPU and no kernel is involved."""
import os
import socket

import pytest
import torch.multiprocessing as mp

from relation_token_mixing_gb300 import replicas


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    env = {"WORLD_SIZE": str(world), "RANK": str(rank), "LOCAL_RANK": str(rank),
           "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)}
    os.environ.update(env)
    r = replicas.from_env()
    replicas.init(r, "gloo")
    replicas.barrier(r)
    slowest = replicas.max_over_ranks(r, times[rank])
    rate = replicas.job_rate(r, 1000.0, slowest)
    replicas.barrier(r)
    replicas.finish(r)
    out.put((rank, slowest, rate))


@pytest.mark.parametrize("world", [2])
def test_two_gloo_ranks_take_the_slowest_time(world):
    ctx = mp.get_context("spawn")
    out = ctx.SimpleQueue()
    times = [0.25, 0.75]
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    for p in procs:
        if p.is_alive():
            p.kill()
            p.join()
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(out.get() for _ in range(world))
    for rank, slowest, rate in got:
        assert slowest == max(times)
        assert rate == pytest.approx(world * 1000.0 / max(times))
    assert [g[0] for g in got] == list(range(world))


def test_single_process_defaults():
    r = replicas.from_env({})
    assert (r.world, r.rank, r.local, r.distributed) == (1, 0, 0, False)
    assert replicas.max_over_ranks(r, 3.5) == 3.5
    assert replicas.job_rate(r, 10.0, 2.0) == 5.0
    replicas.init(r, "gloo")   # no process group for one process
    replicas.barrier(r)
    replicas.finish(r)


def test_rank_layout_is_checked():
    with pytest.raises(ValueError):
        replicas.from_env({"WORLD_SIZE": "2", "RANK": "2"})
    with pytest.raises(ValueError):
        replicas.from_env({"WORLD_SIZE": "0"})
    r = replicas.from_env({"WORLD_SIZE": "4", "RANK": "3", "LOCAL_RANK": "1"})
    assert (r.world, r.rank, r.local) == (4, 3, 1)
    with pytest.raises(ValueError):
        replicas.job_rate(r, 1.0, 0.0)
