"""Two ranks on the CPU (gloo): token sharding covers the batch exactly, the
sharded results equal the whole-batch results, and the benchmark's
max-over-ranks timing reduction works."""
import socket

import pytest
import torch.multiprocessing as mp

from transformer_rope_positional_gb300 import shard


def test_token_ranges_tile_the_batch():
    for total in (0, 1, 5, 37, 1024):
        for world in (1, 2, 3, 8):
            ranges = [shard.token_range(total, r, world) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == total
            assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
            sizes = [b - a for a, b in ranges]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        shard.token_range(10, 2, 2)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def test_two_rank_shards_match_whole_batch():
    import gloo_worker

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    mp.spawn(gloo_worker.run, args=(2, _free_port(), q), nprocs=2, join=True)
    assert q.get(timeout=60) is True
