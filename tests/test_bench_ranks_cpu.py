"""The bench's multi-rank host logic on CPU: world size 2 over gloo (the
path shards into independent replicas, so the ranks only share a timing
barrier and the max over ranks; no data-path collective)."""
import multiprocessing
import socket
import types

import pytest

import bench

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_max_over_ranks_with_two_gloo_ranks():
    import _ranks_worker

    ctx = multiprocessing.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_ranks_worker.max_over_ranks_worker, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict(queue.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # every rank sees the slowest rank's time
    assert results == {0: 1.5, 1: 1.5}


def test_single_rank_max_is_identity():
    assert bench.max_over_ranks(3.25, None, "cpu") == 3.25


def test_job_rate_is_whole_job_weak_scaling():
    # every rank processes the same units; the job takes the slowest rank's time
    assert bench.job_rate(100.0, 2.0, 1) == 50.0
    assert bench.job_rate(100.0, 2.0, 4) == 200.0


def test_reference_arm_runs_on_rank_zero_only(capsys):
    args = types.SimpleNamespace(steps=1, warmup=0)
    bench.run_reference(args, world=2, rank=1)
    assert capsys.readouterr().out == ""
