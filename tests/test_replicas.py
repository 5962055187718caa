"""The multi-GPU form of the bench is N independent replicas (no collective
on the data path): the only cross-rank steps are a barrier and the maximum
of the timed region over ranks.  Exercised here with two gloo ranks on CPU."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        elapsed = bench.max_over_ranks(1.0 + rank, torch.device("cpu"))
        q.put((rank, elapsed, bench.replica_value(1000, 10, world, elapsed)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas_agree_on_the_slowest_clock():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks see the slower rank's 2.0 s; the job value counts both replicas
    assert [o[1] for o in out] == [2.0, 2.0]
    assert out[0][2] == pytest.approx(1000 * 10 * 2 / 2.0 / 1e9)


def test_single_process_is_its_own_maximum():
    assert bench.max_over_ranks(3.5, torch.device("cpu")) == 3.5
