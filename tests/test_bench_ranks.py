"""Host logic of `bench.py --gpus N` (N independent replicas, one per rank):
the max-over-ranks timing reduction, the whole-job aggregate and the
reference arm's rank handling, run as world-size-2 gloo process groups on
the CPU (no GPU)."""
import importlib.util
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, values, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _bench()
        m = b.max_over_ranks(values[rank], world)
        job = b.whole_job(m, 64, world)
        dist.barrier()
        q.put((rank, m, job))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_gloo():
    world, values = 2, [0.2141, 0.2187]  # ms per step on each rank
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, values, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, m, job in got:
        assert m == pytest.approx(max(values))  # every rank sees the slowest rank's time
        assert job["us_per_step"] == pytest.approx(max(values) * 1e3 / world)
        assert job["rows_per_s"] == pytest.approx(64 * world / (max(values) * 1e-3))


def test_single_rank_is_plain():
    b = _bench()
    assert b.max_over_ranks(0.25, 1) == 0.25
    assert b.whole_job(0.25, 64, 1) == {"us_per_step": 250.0, "rows_per_s": 64 / 0.25e-3}


def test_reference_arm_other_ranks_do_no_work(monkeypatch, capsys):
    """Under torchrun only rank 0 runs and prints the reference arm."""
    b = _bench()
    monkeypatch.setenv("RANK", "1")
    args = type("A", (), {"workload": 2, "steps": 1, "warmup": 0})()
    assert b.run_reference(args) is None
    assert capsys.readouterr().out == ""
