"""Token sharding for runs with one process per GPU.

Both operators treat tokens independently (a token's rows read only that
token's cos/sin or cache rows), so a batch splits across ranks into contiguous
token ranges with no exchange at all: each rank applies the operator to its own
range on its own GPU.  These helpers compute the ranges and cut the inputs.
"""
from __future__ import annotations

from typing import Tuple

import torch


def token_range(total: int, rank: int, world: int) -> Tuple[int, int]:
    """Contiguous range [start, end) of ``total`` tokens owned by ``rank``;
    the ranges of ranks 0..world-1 tile [0, total), sizes differing by at most 1."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("rank %d outside a world of %d" % (rank, world))
    base, extra = divmod(total, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def shard_cache_inputs(positions: torch.Tensor, query: torch.Tensor, key: torch.Tensor, rank: int,
                       world: int):
    """This rank's tokens of the cache-indexed operator's inputs (views).

    positions is [T] (rope) or [m, T] (mrope); query/key are [T, ...].  The
    cos/sin cache is not sharded: every rank keeps the whole table."""
    T = query.shape[0]
    a, b = token_range(T, rank, world)
    return positions[..., a:b], query[a:b], key[a:b]


def shard_inplace_inputs(x: torch.Tensor, cos: torch.Tensor, sin: torch.Tensor, rank: int, world: int):
    """This rank's part of the in-place operator's inputs: x [B, S, N, D] is cut
    along B when B >= world, else along S; cos/sin follow the cut on the dims
    they do not broadcast.  A cut along S with B > 1 is a strided view: move it
    to the rank's device with ``.contiguous()`` (the operator takes contiguous
    tensors) and gather the results back the same way."""
    B, S = x.shape[0], x.shape[1]
    if B >= world:
        a, b = token_range(B, rank, world)
        cut = (lambda t: t[a:b]) if cos.shape[0] != 1 else (lambda t: t)
        return x[a:b], cut(cos), cut(sin)
    a, b = token_range(S, rank, world)
    cut = (lambda t: t[:, a:b]) if cos.shape[1] != 1 else (lambda t: t)
    return x[:, a:b], cut(cos), cut(sin)
