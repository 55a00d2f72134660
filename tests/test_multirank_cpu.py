"""The multi-GPU path of bench.py is replicas (weak scaling): every rank runs
its own seeded copy of the workload, no collective touches the data, and the
job time is the maximum over ranks. Its host logic runs here on CPU with a
world-size-2 gloo process group."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402
import workloads  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        seconds = [0.25, 0.75][rank]          # rank 1 is the slow replica
        sec = bench.max_over_ranks(seconds, dist, "cpu")
        w = workloads.make(1, 64, 2, 16, 16, "bf16", seed=rank)  # own data per rank
        digest = float(w.q.values.astype(np.float64).sum())
        sums = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(sums, torch.tensor([digest], dtype=torch.float64))
        q.put((rank, sec, [float(x) for x in sums]))
    finally:
        dist.destroy_process_group()


def test_replicas_time_is_max_over_ranks_and_data_differs():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, sec, sums in got:
        assert sec == 0.75
        assert sums[0] != sums[1]             # seeded per rank: distinct replicas


def test_job_throughput_counts_every_replica():
    assert bench.job_tokens_per_s(16384, 1, 10, 0.01) == pytest.approx(16384 * 10 / 0.01)
    assert bench.job_tokens_per_s(16384, 4, 10, 0.01) == pytest.approx(4 * 16384 * 10 / 0.01)
    assert bench.max_over_ranks(1.5) == 1.5
