"""The benchmark's multi-GPU path is replicas: every rank encodes its own
requests and rank 0 reports the whole job (the slowest rank's time, all
ranks' bytes).  Its host logic runs here as two gloo processes on the CPU."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    times, nbytes = [0.5, 0.8], [1000, 2500]
    s, b = bench.combine_ranks(times[rank], nbytes[rank], world, torch.device("cpu"))
    out.put((rank, s, b, bench.rank_seeds(rank, 4, 3)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_time_and_all_bytes():
    ctx = torch.multiprocessing.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, s, b, _ in res:
        assert s == 0.8 and b == 3500.0, rank
    (t0, w0), (t1, w1) = res[0][3], res[1][3]
    seeds = t0 + w0 + t1 + w1
    assert len(set(seeds)) == len(seeds)          # no request shared between ranks or phases


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.combine_ranks(0.25, 123, 1, None) == (0.25, 123.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.run_reference(None) is None      # returns before it reads its arguments
    assert capsys.readouterr().out == ""
