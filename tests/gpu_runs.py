"""Helpers that run one workload through the CUDA library and through the
oracle, for the parity tests."""
import torch

import oracle
import transformer_rope_positional_gb300 as R


def gpu_inplace(case, stream=None):
    x = case.x.cuda()
    c = case.cos.cuda()
    s = case.sin.cuda()
    R.rope_inplace_partial(x, c, s, case.rotary_mode, [case.start, case.end], stream=stream)
    torch.cuda.synchronize()
    return x.cpu()


def oracle_inplace(case):
    return oracle.inplace_partial_rotary_mul(case.x, case.cos, case.sin, case.start, case.end)


def gpu_cache(case, positions=None):
    pos = (case.positions if positions is None else positions).cuda()
    q = case.query.cuda()
    k = case.key.cuda()
    c = case.cache.cuda()
    R.rope_with_sin_cos_cache(pos, q, k, c, case.head_size, case.rotary_dim, case.is_neox, case.mrope_section)
    torch.cuda.synchronize()
    return q.cpu(), k.cpu()


def oracle_cache(case, positions=None):
    pos = case.positions if positions is None else positions
    return oracle.rope_with_sin_cos_cache(pos, case.query, case.key, case.cache, case.head_size,
                                          case.is_neox, case.mrope_section)
