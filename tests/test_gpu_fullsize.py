"""The five named workloads at full size, through the same library calls the
benchmark times.

The oracle recomputes a sample of tokens one by one (tokens are independent
under both operators); properties that hold at any size -- untouched columns
bit-exact, no device error -- are checked on the whole output.
"""
import pytest
import torch

import oracle
import workloads as W
from gpu_runs import gpu_cache, gpu_inplace, oracle_inplace
from parity import assert_matches, same_bits
import transformer_rope_positional_gb300 as R

pytestmark = pytest.mark.gpu

SAMPLE = 384


def _sample(n, seed):
    idx = W.uniform_int(W.stream_seed(seed, 9), SAMPLE, 0, n)
    return torch.unique(torch.cat([idx, torch.tensor([0, n - 1])]))


@pytest.mark.parametrize("variant", ["slice", "full", "noop"])
def test_small_f32_workload_whole(rope_gpu, variant):
    case = W.inplace_f32_small(variant)
    got = gpu_inplace(case)
    assert_matches(got, oracle_inplace(case), case.name)


def test_mixed_bf16_workload_full_size(rope_gpu):
    case = W.inplace_bf16_mixed()
    got = gpu_inplace(case)
    assert R.get_device_error() == 0
    B, S, N, D = case.x.shape
    # columns [0, 64) are outside the slice: bit-exact over the whole tensor
    assert same_bits(got[..., :64], case.x[..., :64])
    tok = _sample(B * S, 101)
    for t in tok.tolist():
        b, s = divmod(t, S)
        sub = W.InplaceCase("tok", case.x[b:b + 1, s:s + 1].contiguous(), case.cos[:, s:s + 1].contiguous(),
                            case.sin[:, s:s + 1].contiguous(), case.start, case.end)
        ref = oracle.inplace_partial_rotary_mul(sub.x, sub.cos, sub.sin, sub.start, sub.end)
        assert_matches(got[b:b + 1, s:s + 1], ref, "token %d" % t)


def _check_cache_sampled(case, seed):
    qg, kg = gpu_cache(case)
    assert R.get_device_error() == 0
    T = case.tokens
    tok = _sample(T, seed)
    pos = case.positions[..., tok].contiguous()
    qo, ko, skipped = oracle.rope_with_sin_cos_cache(pos, case.query[tok], case.key[tok], case.cache,
                                                     case.head_size, case.is_neox, case.mrope_section)
    assert skipped == 0
    assert_matches(qg[tok], qo, case.name + " query")
    assert_matches(kg[tok], ko, case.name + " key")
    return qg, kg


def test_neox_bf16_workload_full_size(rope_gpu):
    _check_cache_sampled(W.cache_neox_bf16(), 102)


def test_gptj_f16_partial_workload_full_size(rope_gpu):
    case = W.cache_gptj_f16_partial()
    qg, kg = _check_cache_sampled(case, 103)
    hs, r = case.head_size, case.rotary_dim
    for got, x in ((qg, case.query), (kg, case.key)):
        assert same_bits(got.view(case.tokens, -1, hs)[..., r:], x.view(case.tokens, -1, hs)[..., r:])


def test_mrope_workload_full_size(rope_gpu):
    _check_cache_sampled(W.mrope_neox_bf16(), 104)


@pytest.mark.parametrize("run", [("half", False), ("interleave", True)], ids=["half_fwd", "interleave_bwd"])
def test_mixed_bf16_workload_full_size_other_modes(rope_gpu, run):
    mode, backward = run
    case = W.inplace_bf16_mixed()
    x = case.x.cuda()
    fn = R.rope_inplace_partial_backward if backward else R.rope_inplace_partial
    fn(x, case.cos.cuda(), case.sin.cuda(), mode, [case.start, case.end])
    got = x.cpu()
    B, S, N, D = case.x.shape
    assert same_bits(got[..., :64], case.x[..., :64])
    for t in _sample(B * S, 105).tolist():
        b, s = divmod(t, S)
        ref = oracle.inplace_partial_rotary_mul(case.x[b:b + 1, s:s + 1].contiguous(),
                                                case.cos[:, s:s + 1].contiguous(), case.sin[:, s:s + 1].contiguous(),
                                                case.start, case.end, rotary_mode=R._capi.MODES[mode],
                                                backward=backward)
        assert_matches(got[b:b + 1, s:s + 1], ref, "token %d" % t)


def test_unaligned_slice_full_size(rope_gpu):
    """The [4,4096,32,128] bf16 workload with the slice [4,68): 8-byte vectors,
    and a slice that crosses a 128-byte line of every row."""
    full = W.inplace_bf16_mixed()
    case = W.inplace_case("inplace_bf16x_f32cs_4x4096x32x128_slice4_68", 1, tuple(full.x.shape), 4, 68,
                          torch.bfloat16, torch.float32)
    got = gpu_inplace(case)
    assert R.get_device_error() == 0
    assert same_bits(got[..., :4], case.x[..., :4]) and same_bits(got[..., 68:], case.x[..., 68:])
    B, S, N, D = case.x.shape
    for t in _sample(B * S, 106).tolist():
        b, s = divmod(t, S)
        ref = oracle.inplace_partial_rotary_mul(case.x[b:b + 1, s:s + 1].contiguous(), case.cos[:, s:s + 1],
                                                case.sin[:, s:s + 1], 4, 68)
        assert_matches(got[b:b + 1, s:s + 1], ref, "token %d" % t)


def test_mrope_interleaved_splice_full_size(rope_gpu):
    """The mrope workload through the V2 interleaved splice (cacheMode 1)."""
    case = W.mrope_neox_bf16()
    q, k = case.query.cuda(), case.key.cuda()
    R.rope_with_sin_cos_cache(case.positions.cuda(), q, k, case.cache.cuda(), case.head_size, case.rotary_dim,
                              case.is_neox, case.mrope_section, cache_mode=1)
    torch.cuda.synchronize()
    assert R.get_device_error() == 0
    tok = _sample(case.tokens, 107)
    qo, ko, skipped = oracle.rope_with_sin_cos_cache(case.positions[..., tok].contiguous(), case.query[tok],
                                                     case.key[tok], case.cache, case.head_size, case.is_neox,
                                                     case.mrope_section, cache_mode=1)
    assert skipped == 0
    assert_matches(q[tok.cuda()].cpu(), qo, "interleaved splice query")
    assert_matches(k[tok.cuda()].cpu(), ko, "interleaved splice key")
