"""bench.py's replica mode on CPU: two gloo ranks agree on the slowest rank's
time and report whole-job throughput (no GPU; the data path has no collective)."""
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
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        elapsed = [10.0, 25.0][rank]  # rank 1 is slower
        slowest = bench.max_over_ranks(elapsed, "cpu")
        q.put((rank, slowest, bench.job_gbs(1_000_000, world, 100, slowest)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, slowest, gbs in got:
        assert slowest == 25.0
        assert gbs == pytest.approx(2 * 1_000_000 * 100 / 25e-3 / 1e9)


def test_single_process_is_identity():
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
    assert bench.job_gbs(10**9, 1, 1, 1.0) == pytest.approx(1000.0)


def test_reference_arm_prints_only_on_rank_zero(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = bench.main.__globals__["argparse"].Namespace(config=1, steps=3, warmup=3, ref_seconds=1.0)
    assert bench.run_reference(args) is None
