"""Host logic of the N > 1 bench path (replicas, weak scaling) on CPU ranks
with the gloo backend: the job time is the slowest rank's, the value counts
every rank's units, and the reference arm runs on rank 0 only."""
import os
import socket
import sys
import types

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out_q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(times[rank], dist, device="cpu")
        dist.barrier()
        out_q.put((rank, t, bench.whole_job_value(world, 1000, 26097152 / 1e9, t)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_max_over_ranks_and_whole_job_value(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    times = [0.010 + 0.002 * r for r in range(world)]
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    slowest = max(times)
    for _, t, v in res:
        assert t == pytest.approx(slowest)
        assert v == pytest.approx(world * 1000 * 26097152 / 1e9 / slowest)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(0.5, None) == 0.5
    assert bench.whole_job_value(1, 10, 2.0, 4.0) == 5.0


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    args = types.SimpleNamespace(config=0, steps=1, warmup=0, gpus=2)
    assert bench.run_reference(args) is None
    assert capsys.readouterr().out == ""
