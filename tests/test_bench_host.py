"""Host logic of bench.py that needs no GPU: the multi-rank aggregation over a world-size-2 gloo
group (the slowest rank's time, every rank's tokens) and the reference arm's rank-0-only rule."""
import os
import socket
import sys
import types

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [3.0, 5.0][rank]  # this rank's step time
        m = bench.max_over_ranks(ms, dist, torch.device("cpu"))
        q.put((rank, m, bench.job_tokens_per_s(1000, world, m)))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, _, _ in out] == [0, 1]
    assert all(m == 5.0 for _, m, _ in out)              # both ranks see the slowest rank
    assert out[0][2] == pytest.approx(2 * 1000 / 5e-3)   # all ranks' tokens over that time


def test_reference_arm_runs_on_rank_0_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    def no_work(*a, **k):
        raise AssertionError("rank 1 of the reference arm did work")

    monkeypatch.setattr(bench, "make_inputs", no_work)
    monkeypatch.setenv("RANK", "1")
    args = types.SimpleNamespace(workload="large_s4096", steps=1, warmup=0)
    assert bench.run_reference(args) is None  # returns before building, drawing or timing anything
