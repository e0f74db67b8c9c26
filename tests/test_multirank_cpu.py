"""The benchmark's multi-rank host logic on 2 gloo ranks (CPU, no GPU).

The path shards by sequence with no exchange, so ranks only meet to agree on
the slowest rank's time; the reference arm runs on rank 0 alone.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    times = [1.0 + rank, 5.0 - rank]                 # rank 0: [1, 5]; rank 1: [2, 4]
    got = bench.reduce_max(times)
    thr = bench.job_throughput(world, 3e9, got[0])
    # A non-zero rank of the reference arm returns at once without output.
    rc = bench.run_reference(bench.parse_args(["--impl", "reference"])) if rank == 1 else None
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, got, thr, rc))


def test_two_gloo_ranks_agree_on_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, thr, rc in results:
        assert got == [2.0, 5.0]
        assert thr == pytest.approx(2 * 3e9 / 2.0 / 1e9)
    assert results[1][3] == 0


def test_single_process_reduction_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max([1.5, 2.5]) == [1.5, 2.5]
    assert bench.job_throughput(1, 2e9, 0.5) == pytest.approx(4.0)
