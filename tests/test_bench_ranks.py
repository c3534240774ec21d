"""The multi-rank path of bench.py (replicas only) on CPU: two gloo ranks on 127.0.0.1 agree on
the slowest rank's time and the whole-job rate; the reference arm does no work off rank 0."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, lr = bench.rank_env()
        local_ms = 10.0 + 5.0 * r  # rank 1 is the slow one
        mx = bench.max_over_ranks(local_ms, w, torch.device("cpu"))
        dist.barrier()
        q.put((r, w, lr, mx, bench.whole_job_rate(w, 4096, 20, mx)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_time_and_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, world, local, mx, rate) in enumerate(out):
        assert (rank, world, local) == (r, 2, r)
        assert mx == 15.0  # the slower rank's time, on both ranks
        assert rate == pytest.approx(2 * 4096 * 20 / 0.015)


def test_single_rank_needs_no_process_group(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.rank_env() == (1, 0, 0)
    assert bench.max_over_ranks(3.5, 1, None) == 3.5
    assert bench.whole_job_rate(1, 4096, 10, 20.0) == pytest.approx(4096 * 10 / 0.02)


def test_reference_arm_does_nothing_off_rank_zero(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")

    class Args:
        tokens, ref_tokens, steps, warmup = 4096, 4, 1, 0

    bench.run_reference(Args())  # returns before importing or building the oracle
    assert capsys.readouterr().out == ""
