"""Worker for the two-rank gloo test (CPU only): each rank takes its token
shard, runs the oracle on it, and the ranks check the pieces against the
whole-batch result and the timing reduction the benchmark uses."""
import os

import torch
import torch.distributed as dist


def run(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle
        import workloads as W
        from transformer_rope_positional_gb300 import shard

        # cache-indexed operator, mrope, ragged token count
        c = W.cache_case("gloo", 90, 37, 3, 1, 64, 64, 200, torch.bfloat16, True, mrope_section=[8, 12, 12])
        pos, q, k = shard.shard_cache_inputs(c.positions, c.query, c.key, rank, world)
        qo, ko, _ = oracle.rope_with_sin_cos_cache(pos.contiguous(), q.contiguous(), k.contiguous(), c.cache, 64,
                                                   True, c.mrope_section)
        pieces = [None] * world
        dist.all_gather_object(pieces, (qo, ko))
        # in-place operator, sharded along S (B = 1 < world)
        ic = W.inplace_case("gloo_inplace", 91, (1, 9, 3, 32), 8, 24, torch.float16, torch.float32)
        x, cs, sn = shard.shard_inplace_inputs(ic.x, ic.cos, ic.sin, rank, world)
        xo = oracle.inplace_partial_rotary_mul(x.contiguous(), cs.contiguous(), sn.contiguous(), 8, 24)
        xpieces = [None] * world
        dist.all_gather_object(xpieces, xo)
        # the benchmark's max-over-ranks reduction
        mx = bench.max_over_ranks(float(rank + 1) * 1.5, world, torch.device("cpu"))
        if rank == 0:
            qw, kw, _ = oracle.rope_with_sin_cos_cache(c.positions, c.query, c.key, c.cache, 64, True,
                                                       c.mrope_section)
            xw = oracle.inplace_partial_rotary_mul(ic.x, ic.cos, ic.sin, 8, 24)
            ok = (torch.equal(torch.cat([p[0] for p in pieces]).view(torch.int16), qw.view(torch.int16))
                  and torch.equal(torch.cat([p[1] for p in pieces]).view(torch.int16), kw.view(torch.int16))
                  and torch.equal(torch.cat(xpieces, dim=1).view(torch.int16), xw.view(torch.int16))
                  and mx == 1.5 * world)
            out.put(bool(ok))
        dist.barrier()
    finally:
        dist.destroy_process_group()
