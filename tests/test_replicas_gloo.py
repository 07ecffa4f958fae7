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


def _spawned_rank(out_dir):
    """Target of bench.spawn_local_ranks: joins the job the way run_cuda
    does (gloo here, without a GPU), then records what it saw."""
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    ws, rank, local = bench.dist_setup()
    try:
        bench.barrier(ws)
        worst = bench.max_over_ranks(0.1 + 0.01 * rank, ws)
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{ws} {rank} {local} {worst:.6f}")
    finally:
        dist.destroy_process_group()


def test_gpus_flag_spawns_local_ranks(tmp_path):
    """bench.py --gpus N without torchrun starts N ranks itself; each gets
    RANK / LOCAL_RANK / WORLD_SIZE as torchrun would set them and joins one
    process group."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    rc = bench.spawn_local_ranks(2, _spawned_rank, str(tmp_path))
    assert rc == 0
    got = sorted((tmp_path / f"rank{r}.txt").read_text().split() for r in range(2))
    assert got == [["2", "0", "0", "0.110000"], ["2", "1", "1", "0.110000"]]
