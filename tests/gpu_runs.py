"""Helpers that run one workload through the CUDA library and through the
oracle, for the parity tests.  Every device tensor of a GPU call sits between
guard bands (tests/guard.py) that are checked after the call."""
import torch

import oracle
import transformer_rope_positional_gb300 as R
from guard import Guards


def gpu_inplace(case, stream=None):
    g = Guards()
    x, c, s = g.put(case.x, "x"), g.put(case.cos, "cos"), g.put(case.sin, "sin")
    R.rope_inplace_partial(x, c, s, case.rotary_mode, [case.start, case.end], stream=stream)
    g.check()
    return x.cpu()


def oracle_inplace(case):
    return oracle.inplace_partial_rotary_mul(case.x, case.cos, case.sin, case.start, case.end)


def gpu_cache(case, positions=None):
    g = Guards()
    pos = g.put(case.positions if positions is None else positions, "positions")
    q, k, c = g.put(case.query, "query"), g.put(case.key, "key"), g.put(case.cache, "cache")
    R.rope_with_sin_cos_cache(pos, q, k, c, case.head_size, case.rotary_dim, case.is_neox, case.mrope_section)
    g.check()
    return q.cpu(), k.cpu()


def oracle_cache(case, positions=None):
    pos = case.positions if positions is None else positions
    return oracle.rope_with_sin_cos_cache(pos, case.query, case.key, case.cache, case.head_size,
                                          case.is_neox, case.mrope_section)


def _all_cores(fn, shards):
    import concurrent.futures as cf

    import bench
    with cf.ThreadPoolExecutor(max_workers=bench.usable_cores()) as pool:
        return list(pool.map(fn, shards))


def oracle_inplace_all_cores(case, rotary_mode=None, backward=False):
    """The oracle on the whole workload, token shards spread over every usable
    core (bit-exact with one call; tests/test_bench_host.py checks that)."""
    import bench
    mode = case.rotary_mode if rotary_mode is None else rotary_mode
    shards = bench.oracle_shards(case, 4 * bench.usable_cores())
    outs = _all_cores(lambda s: oracle.inplace_partial_rotary_mul(s.x, s.cos, s.sin, s.start, s.end, mode, backward),
                      shards)
    return torch.cat(outs, 1)


def oracle_cache_all_cores(case, cache_mode=0):
    """(query, key, skipped) of the oracle on the whole workload, over every core."""
    import bench
    shards = bench.oracle_shards(case, 4 * bench.usable_cores())
    outs = _all_cores(lambda s: oracle.rope_with_sin_cos_cache(s.positions, s.query, s.key, s.cache, s.head_size,
                                                               s.is_neox, s.mrope_section, cache_mode), shards)
    return torch.cat([o[0] for o in outs]), torch.cat([o[1] for o in outs]), sum(o[2] for o in outs)
