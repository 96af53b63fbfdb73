"""The multi-rank path of bench.py (one replica per rank, weak scaling) on
CPU with the gloo backend and two ranks: barrier, max-over-ranks timing and
the whole-job throughput."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, local = bench.dist_setup(None)
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    # rank r "took" 1 + r seconds for 1000 units
    value, slowest = bench.aggregate_throughput(1.0 + rank, 1000, w)
    # the end-to-end leg runs only where every rank's host buffer fits: one
    # rank that does not fit makes all of them skip it
    any_short = bench.max_over_ranks(1.0 if rank == 1 else 0.0, w)
    out.put((rank, value, slowest, any_short))
    bench.barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_report_whole_job_throughput():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(out.get(timeout=10) for _ in range(2))
    for rank, value, slowest, any_short in res:
        assert slowest == pytest.approx(2.0)          # the slower rank's time
        assert value == pytest.approx(2 * 1000 / 2.0)  # all units / slowest time
        assert any_short == 1.0


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate_throughput(2.0, 100, 1) == (50.0, 2.0)


def test_host_memory_is_read_for_the_end_to_end_guard():
    sys.path.insert(0, ROOT)
    import bench
    avail = bench.host_memory_available()
    assert avail is None or avail > 0
