"""The N > 1 path of bench.py on CPU: world_size-2 gloo ranks.  The codec's
streams are independent, so ranks share nothing on the data path; what
crosses ranks is the timing (each time's maximum over ranks) and the
reference arm's rank gating (rank 0 alone runs and prints)."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    got = bench.rank_max([1.0 + rank, 10.0 - rank, 5.0], world, "cpu")
    gbs = bench.job_gbs(2e9, world, got[0])
    assert bench.dist_env()[:2] == (rank, world)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, got, gbs))


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, got, gbs in res:
        assert got == [2.0, 10.0, 5.0]                 # every rank sees the maxima
        assert gbs == pytest.approx(2 * 2e9 / 2e-3 / 1e9)  # both ranks' bytes over the slowest time


def test_single_rank_passes_values_through():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.rank_max([3.0, 4.5], 1, "cpu") == [3.0, 4.5]
    assert bench.job_gbs(1e9, 1, 1.0) == pytest.approx(1000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = type("A", (), {"workload": "llama3_70b_L80_H8_d128_S32768", "steps": 1, "warmup": 0, "gpus": 2})()
    assert bench.run_reference(args) is None
    assert capsys.readouterr().out == ""  # the other ranks exit without work or output
