"""The multi-rank path of bench.py on CPU: two gloo ranks of a weak-scaling
run agree on the whole-job throughput, taken over the slowest rank, without any
data-path collective (each rank's replica works on its own batch)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r timed 10 + 5r ms over 4 steps of 64 tokens, e2e 20 + r ms
    v, e, t, te = bench.aggregate_over_ranks(10.0 + 5 * rank, 20.0 + rank, 64, 4, world, torch.device("cpu"))
    q.put((rank, v, e, t, te))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_weak_scaling_aggregate_over_gloo_ranks(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    slowest = 10.0 + 5 * (world - 1)
    for rank, v, e, t, te in res:
        assert t == slowest and te == 20.0 + (world - 1)
        assert v == pytest.approx(world * 64 * 4 / (slowest / 1e3))
        assert e == pytest.approx(world * 64 * 4 / (te / 1e3))
    assert len({r[1] for r in res}) == 1          # every rank reports the same job throughput


def test_single_rank_needs_no_process_group():
    import bench
    v, e, t, te = bench.aggregate_over_ranks(8.0, 16.0, 16, 2, 1, torch.device("cpu"))
    assert (t, te) == (8.0, 16.0) and v == pytest.approx(32 / 8e-3) and e == pytest.approx(32 / 16e-3)
