"""The multi-GPU path of bench.py is replicas only (heads and sequences are
independent; no data-path collective).  Its host logic -- max-over-ranks timing
and the whole-job rate -- is exercised here with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ws, r, local = bench.dist_env()
        assert (ws, r, local) == (world, rank, rank)
        # rank r "measured" 1 + r ms for prefill and 3 - r ms for decode
        pre, dec = bench.max_over_ranks([1.0 + rank, 3.0 - rank])
        rate = bench.replica_rate(4096, ws, pre)
        out.put((rank, pre, dec, rate))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_sum_the_work():
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(2))
    for rank, pre, dec, rate in res:
        assert pre == 2.0 and dec == 3.0  # slowest rank on each metric
        assert rate == pytest.approx(2 * 4096 / 2.0e-3)


def test_single_process_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
    assert bench.replica_rate(100, 1, 0.5) == pytest.approx(2e5)
