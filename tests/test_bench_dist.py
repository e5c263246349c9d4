"""The bench's multi-process path (replicas only) on CPU with gloo, world 2:
barrier, exactly K timed steps after W warm-up steps, max over ranks."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import time
    import bench
    d = bench.Dist(world, "gloo")
    calls = []

    def step():
        calls.append(1)
        time.sleep(0.01 * (rank + 1))      # rank 1 is the slower replica

    dt = bench.timed_region(step, lambda: None, d, steps=5, warmup=3)
    out[rank] = (len(calls), dt)
    d.close()


def test_two_replicas_gloo():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == 8 and res[1][0] == 8            # 3 warm-up + 5 timed steps each
    assert res[0][1] == pytest.approx(res[1][1])        # both report the max over ranks
    assert res[0][1] >= 5 * 0.02                        # ... which is the slower rank's time
