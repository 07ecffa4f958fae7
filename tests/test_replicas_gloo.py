"""Host logic of the multi-GPU benchmark, on CPU with two gloo ranks.

The attention path shards into independent (batch, KV-group) units with no
exchange, so N GPUs run N independent replicas ("replicas only"); the
benchmark only needs a barrier and a max over ranks of the step time.  These
tests run that logic as world_size-2 gloo processes on 127.0.0.1."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        local_ms = [0.120, 0.135][rank]          # rank 1 is the slowest replica
        bench.barrier(ws)
        worst = bench.max_over_ranks(local_ms, ws)
        value = bench.job_value(45.097e9, worst, ws)
        q.put((rank, worst, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_and_job_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    out = sorted(q.get(timeout=10) for _ in range(2))
    for rank, worst, value in out:
        assert worst == pytest.approx(0.135)
        # two replicas, each one step of 45.097 GFLOP, slowest at 0.135 ms
        assert value == pytest.approx(2 * 45.097e9 / 0.135e-3 / 1e12)


def test_reference_arm_other_ranks_exit_without_work(capsys, monkeypatch):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")

    class Args:
        steps, warmup = 1, 0
    bench.run_reference(Args())
    assert capsys.readouterr().out == ""
