"""The multi-GPU path of bench.py is N independent replicas (observations do
not interact), so the only cross-rank steps are the timing barrier and the
max over ranks.  These tests run that aggregation on world-size-2 CPU ranks
(gloo) and check the whole-job rate and that every replica solves its own
inputs."""

import os
import socket

import numpy as np
import pytest


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world_size, port, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world_size))
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world_size)
    try:
        mine = [10.0 + rank, 5.0 - rank, 3.0 * (rank + 1)]
        got = bench.max_over_ranks(dist, mine, "cpu")
        dist.barrier()
        queue.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_world_size_2_gloo():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        results = dict(queue.get(timeout=180) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs)
    # Each element is the slowest rank's value, on every rank.
    for r in range(2):
        assert results[r] == [11.0, 5.0, 6.0]


def test_whole_job_rate_and_distinct_replica_inputs():
    import bench
    from workloads import CONFIGS, make_observations

    assert bench.whole_job_rate(2, 64, 25.0) == pytest.approx(2 * 64 / 0.025)
    assert bench.whole_job_rate(1, 1, 7.5) == pytest.approx(1 / 0.0075)
    assert bench.max_over_ranks(None, [1, 2.5], "cpu") == [1.0, 2.5]
    cfg = CONFIGS["tiny_f32"]
    obs = [make_observations(cfg.replace(seed=bench.replica_seed(cfg.seed, r)), cfg.B) for r in range(2)]
    (z0, n0), (z1, n1) = obs
    assert z0.shape == z1.shape and n0.shape == n1.shape
    assert not np.array_equal(z0, z1) and not np.array_equal(n0, n1)
    # Rank 0 keeps the configuration's own seed (the single-GPU inputs).
    z, n = make_observations(cfg, cfg.B)
    assert np.array_equal(z, z0) and np.array_equal(n, n0)
