"""The N > 1 host path of bench.py on CPU: two gloo ranks, each with its own
batch, a barrier, and the slowest rank's time setting the whole-job value
(the path shards by request; there is no collective on the data path)."""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as tmp  # noqa: E402

import bench  # noqa: E402
import workloads as W  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = W.tiny_decode(bench.rank_seed(rank), "bf16")
        dist.barrier()
        local_ms = [1.25, 2.5][rank]
        ms = bench.max_over_ranks(torch, dist, local_ms, torch.device("cpu"))
        q.put((rank, ms, int(w.decode.q.sum()), bench.whole_job_gbs(10 ** 9, world, ms)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = tmp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r[1] for r in res] == [2.5, 2.5]          # both ranks see the slowest time
    assert res[0][2] != res[1][2]                      # each rank has its own batch
    assert res[0][3] == pytest.approx(2 * 1e9 / 2.5e-3 / 1e9)  # whole-job bytes / slowest time


def test_single_rank_is_identity():
    assert bench.max_over_ranks(torch, None, 0.75, torch.device("cpu")) == 0.75
    assert bench.whole_job_gbs(2 * 10 ** 9, 1, 1.0) == pytest.approx(2000.0)
