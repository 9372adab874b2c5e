"""Host logic of the multi-rank bench (replicas only): max-over-ranks timing and
the whole-job aggregate, checked with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t_local = [0.25, 0.40][rank]  # seconds each rank measured
        t_max = bench.reduce_max(t_local, world)
        value = bench.aggregate(per_rank_units=10.0, world=world, t_max_s=t_max)
        q.put((rank, t_max, value))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t_max, value in got:
        assert t_max == pytest.approx(0.40)
        assert value == pytest.approx(2 * 10.0 / 0.40)


def test_single_rank_is_identity():
    assert bench.reduce_max(1.5, 1) == 1.5
    assert bench.aggregate(3.0, 1, 1.5) == pytest.approx(2.0)


def test_reference_arm_other_ranks_exit_without_work(capsys):
    args = bench.argparse.Namespace(workload="decode", steps=1, warmup=3)
    bench.run_reference(args, rank=1, world=2)
    assert capsys.readouterr().out == ""
