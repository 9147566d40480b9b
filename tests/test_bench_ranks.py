"""The bench's multi-rank logic on CPU: the layer blocks that ranks take
cover every (layer, K|V) stream of a workload exactly once, two gloo ranks
on 127.0.0.1 agree on the slowest rank's timings, and the whole-job value
counts the whole workload's bytes once over that time."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import synth  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("name", ["llama31_8b_8k", "mistral_nemo_12b_32k",
                                  "llama33_70b_16k", "qwen25_7b_paged"])
@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
def test_layer_blocks_cover_every_stream_once(name, world):
    import bench
    w = synth.WORKLOADS[name]
    seen = []
    sizes = []
    for rank in range(world):
        l0, nl = bench.layer_shard(w.layers, world, rank)
        seen += [(l, k) for l in range(l0, l0 + nl) for k in w.kv]
        sizes.append(nl)
    assert seen == w.streams()          # every stream once, in order
    assert max(sizes) - min(sizes) <= 1
    # the shards' bytes add up to the workload's
    per_stream = w.requests * w.tokens * w.D * 2
    assert sum(sizes) * len(w.kv) * per_stream == w.raw_bytes()


def test_more_ranks_than_layers_is_refused():
    import bench
    with pytest.raises(ValueError):
        bench.layer_shard(2, 4, 0)


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    import bench
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world),
                       "LOCAL_RANK": str(rank)})
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}",
                            rank=rank, world_size=world)
    r, wsize, _ = bench.dist_env()
    w = synth.WORKLOADS["llama31_8b_8k"]
    l0, nl = bench.layer_shard(w.layers, wsize, r)
    mine = [(l, k) for l in range(l0, l0 + nl) for k in w.kv]
    everyone = [None] * wsize
    dist.all_gather_object(everyone, mine)
    # rank 1 is slower at compress, rank 0 at decompress
    times = [0.20 + 0.05 * r, 0.30 - 0.10 * r, 0.50]
    t = bench.max_over_ranks(times, wsize)
    dist.barrier()
    dist.destroy_process_group()
    q.put((r, wsize, t, everyone,
           bench.job_gbs(w.raw_bytes(), 4, t[1])))


def test_two_gloo_ranks_shard_layers_and_take_the_slowest_rank():
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
    w = synth.WORKLOADS["llama31_8b_8k"]
    for r, wsize, t, everyone, gbs in out:
        assert wsize == 2
        assert t == pytest.approx([0.25, 0.30, 0.50])
        # rank 0 holds layers 0..15, rank 1 layers 16..31; together every
        # stream exactly once
        assert everyone[0][0] == (0, 0) and everyone[1][0] == (16, 0)
        assert everyone[0] + everyone[1] == w.streams()
        # the whole workload once, over the slowest rank's decompress time
        assert gbs == pytest.approx(w.raw_bytes() * 4 / 0.30 / 1e9)


def test_one_rank_is_the_identity():
    import bench
    assert bench.max_over_ranks([1, 2.5], 1) == [1.0, 2.5]
    assert bench.job_gbs(10**9, 2, 1.0) == pytest.approx(2.0)
    assert bench.layer_shard(32, 1, 0) == (0, 32)
