"""The benchmark's N > 1 path on CPU: two gloo ranks, as torchrun would start them.

Each rank prefills its own requests (its own seed of token ids), the timed region's length is
the slowest rank's (max over ranks), and the job's throughput counts every rank's tokens.
"""
import os
import socket
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    sys.path.insert(0, ROOT)
    import bench
    import synth

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, _ = bench.dist_env()
        local_ms = 100.0 + 50.0 * r                 # rank 1 is the slower one
        slowest = bench.slowest_rank_ms(local_ms, w, device="cpu")
        value = bench.job_tokens_per_s(2, 512, 3, w, slowest)
        ids = synth.token_ids(bench.request_seed(r), 2, 512)
        results[r] = (r, w, slowest, value, ids[0, :16].tolist())
    finally:
        dist.destroy_process_group()


def test_two_replicas_time_and_throughput():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        procs = [ctx.Process(target=_rank, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        for p in procs:
            if p.is_alive():
                p.kill()
        assert all(p.exitcode == 0 for p in procs)
        res = dict(results)
    assert sorted(res) == [0, 1]
    for r in (0, 1):
        rr, w, slowest, value, _ = res[r]
        assert (rr, w) == (r, 2)
        assert slowest == 150.0                       # both ranks see the slowest rank's time
        assert value == pytest.approx(2 * 512 * 3 * 2 / 0.150)   # every rank's tokens
    # each replica prefills its own requests
    assert not np.array_equal(res[0][4], res[1][4])


def test_one_rank_is_local():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_rank_ms(12.5, 1) == 12.5
    assert bench.job_tokens_per_s(1, 16384, 5, 1, 1000.0) == pytest.approx(16384 * 5)
