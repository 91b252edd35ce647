"""World-size-2 gloo checks (CPU) of the benchmark's multi-process host logic.

The verification path shards by request with no collective on the data path; the only
cross-rank steps are the benchmark's barrier and its max / sum reductions of host timings.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    bench.init_dist(world, "gloo")
    r, lr, w = bench.dist_env()
    bench.barrier(w)
    mx = bench.max_over_ranks(10.0 + r, w)            # e.g. elapsed ms per rank
    sm = bench.sum_over_ranks(100.0 * (r + 1), w)     # e.g. tokens per rank
    bench.barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()
    q.put((r, mx, sm))


def test_two_rank_timing_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out == [(0, 11.0, 300.0), (1, 11.0, 300.0)]


def test_reference_arm_other_ranks_do_no_work():
    sys.path.insert(0, ROOT)
    import bench
    args = bench.parse(["--impl", "reference", "--steps", "3", "--warmup", "3"])
    assert bench.run_reference(args, rank=1, world=2) is None


def test_single_process_helpers_are_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.sum_over_ranks(2.0, 1) == 2.0
    with pytest.raises(SystemExit):
        bench.parse(["--warmup", "2"])
