"""bench.py's replica path over two gloo ranks on the CPU: the job time is
the slowest rank's, the job rate counts every rank's tokens."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    n, r, _ = bench._dist(backend="gloo")
    assert (n, r) == (world, rank)
    ms_local = 10.0 * (rank + 1)            # rank 1 is the slow one
    slowest = bench.max_over_ranks(ms_local, n)
    rate = bench.job_tokens_per_s(512, 100, n, ms_local)
    out[rank] = (slowest, rate)
    torch.distributed.destroy_process_group()


def test_two_gloo_replicas():
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
    for r in range(2):
        slowest, rate = out[r]
        assert slowest == 20.0
        assert rate == pytest.approx(2 * 512 * 100 / 0.020)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_tokens_per_s(10, 4, 1, 2.0) == pytest.approx(10 * 4 / 0.002)


def test_gpus_flag_against_the_rank_environment():
    """--gpus N must agree with a launcher's WORLD_SIZE (else exit code 2);
    without a launcher N = 1 runs in place and N > 1 starts N ranks itself."""
    import bench
    assert bench.replica_launch(2, [], env={"WORLD_SIZE": "1"}) == 2
    assert bench.replica_launch(1, [], env={"WORLD_SIZE": "4"}) == 2
    assert bench.replica_launch(4, [], env={"WORLD_SIZE": "4"}) is None
    assert bench.replica_launch(1, [], env={}) is None
    assert bench.replica_launch(0, [], env={}) == 2
    # two ranks started through torch.distributed.run; each parses --help
    # and exits 0 before touching a device
    assert bench.replica_launch(2, ["--help"], env={}) == 0
