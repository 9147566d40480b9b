"""The bench's multi-rank logic on CPU: two gloo ranks on 127.0.0.1 agree
on the slowest rank's timings, and the whole-job value counts every rank's
copy of the workload (weak scaling)."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world),
                       "LOCAL_RANK": str(rank)})
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}",
                            rank=rank, world_size=world)
    r, w, _ = bench.dist_env()
    # rank 1 is slower at compress, rank 0 at decompress
    mine = [0.20 + 0.05 * r, 0.30 - 0.10 * r, 0.50]
    t = bench.max_over_ranks(mine, w)
    dist.barrier()
    dist.destroy_process_group()
    q.put((r, w, t, bench.whole_job_gbs(w, 10**9, 4, t[1])))


def test_two_gloo_ranks_take_the_slowest_rank():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q))
             for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, w, t, gbs in out:
        assert w == 2
        assert t == pytest.approx([0.25, 0.30, 0.50])
        # both ranks' copies over the slowest rank's decompress time
        assert gbs == pytest.approx(2 * 1e9 * 4 / 0.30 / 1e9)


def test_one_rank_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1, 2.5], 1) == [1.0, 2.5]
    assert bench.whole_job_gbs(1, 10**9, 2, 1.0) == pytest.approx(2.0)
