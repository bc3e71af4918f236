"""Window sharding and the max-over-ranks timing reduction, on CPU with gloo
(world size 2), the host logic of the multi-GPU bench path."""
import os
import socket

import pytest

from bidirectional_lstm_stack_gb300.sharding import max_over_ranks, window_shard


@pytest.mark.parametrize("total", [0, 1, 2, 7, 32, 256, 257])
@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_shards_cover_every_window_once(total, world):
    seen = []
    sizes = []
    for r in range(world):
        a, b = window_shard(total, r, world)
        seen.extend(range(a, b))
        sizes.append(b - a)
    assert seen == list(range(total))
    assert max(sizes) - min(sizes) <= 1


def test_shard_rejects_bad_rank():
    with pytest.raises(ValueError):
        window_shard(4, 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        shard = window_shard(32 * world, rank, world)
        t = max_over_ranks(1.5 + rank)
        q.put((rank, shard, t))
    finally:
        dist.destroy_process_group()


def test_gloo_world_two_shards_and_max():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got[0][1] == (0, 32) and got[1][1] == (32, 64)
    assert got[0][2] == got[1][2] == 2.5
