"""The five named workloads at full size, through the same library calls the
benchmark times, compared with the oracle on every token: the oracle runs over
the whole workload, token shards spread over all host cores (tokens are
independent under both operators).  Untouched columns are compared bit-exact
over the whole tensor, and every device tensor sits between guard bands."""
import pytest
import torch

import workloads as W
from gpu_runs import gpu_cache, gpu_inplace, oracle_cache_all_cores, oracle_inplace, oracle_inplace_all_cores
from guard import Guards
from parity import assert_matches, assert_matches_rows, same_bits
import transformer_rope_positional_gb300 as R

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("variant", ["slice", "full", "noop"])
def test_small_f32_workload_whole(rope_gpu, variant):
    case = W.inplace_f32_small(variant)
    got = gpu_inplace(case)
    assert_matches(got, oracle_inplace(case), case.name)


def test_mixed_bf16_workload_full_size(rope_gpu):
    case = W.inplace_bf16_mixed()
    got = gpu_inplace(case)
    assert R.get_device_error() == 0
    # columns [0, 64) are outside the slice: bit-exact over the whole tensor
    assert same_bits(got[..., :64], case.x[..., :64])
    assert_matches_rows(got, oracle_inplace_all_cores(case), case.name)


def _check_cache_all_tokens(case):
    qg, kg = gpu_cache(case)
    assert R.get_device_error() == 0
    qo, ko, skipped = oracle_cache_all_cores(case)
    assert skipped == 0
    assert_matches_rows(qg, qo, case.name + " query")
    assert_matches_rows(kg, ko, case.name + " key")
    return qg, kg


def test_neox_bf16_workload_full_size(rope_gpu):
    _check_cache_all_tokens(W.cache_neox_bf16())


def test_gptj_f16_partial_workload_full_size(rope_gpu):
    case = W.cache_gptj_f16_partial()
    qg, kg = _check_cache_all_tokens(case)
    hs, r = case.head_size, case.rotary_dim
    for got, x in ((qg, case.query), (kg, case.key)):
        assert same_bits(got.view(case.tokens, -1, hs)[..., r:], x.view(case.tokens, -1, hs)[..., r:])


def test_mrope_workload_full_size(rope_gpu):
    _check_cache_all_tokens(W.mrope_neox_bf16())


@pytest.mark.parametrize("run", [("half", False), ("interleave", True)], ids=["half_fwd", "interleave_bwd"])
def test_mixed_bf16_workload_full_size_other_modes(rope_gpu, run):
    mode, backward = run
    case = W.inplace_bf16_mixed()
    g = Guards()
    x = g.put(case.x, "x")
    fn = R.rope_inplace_partial_backward if backward else R.rope_inplace_partial
    fn(x, g.put(case.cos, "cos"), g.put(case.sin, "sin"), mode, [case.start, case.end])
    g.check()
    got = x.cpu()
    assert same_bits(got[..., :64], case.x[..., :64])
    ref = oracle_inplace_all_cores(case, R._capi.MODES[mode], backward)
    assert_matches_rows(got, ref, "%s %s" % (mode, "backward" if backward else "forward"))


def test_unaligned_slice_full_size(rope_gpu):
    """The [4,4096,32,128] bf16 workload with the slice [4,68): 8-byte vectors,
    and a slice that crosses a 128-byte line of every row."""
    full = W.inplace_bf16_mixed()
    case = W.inplace_case("inplace_bf16x_f32cs_4x4096x32x128_slice4_68", 1, tuple(full.x.shape), 4, 68,
                          torch.bfloat16, torch.float32)
    got = gpu_inplace(case)
    assert R.get_device_error() == 0
    assert same_bits(got[..., :4], case.x[..., :4]) and same_bits(got[..., 68:], case.x[..., 68:])
    assert_matches_rows(got, oracle_inplace_all_cores(case), case.name)


def test_mrope_interleaved_splice_full_size(rope_gpu):
    """The mrope workload through the V2 interleaved splice (cacheMode 1)."""
    case = W.mrope_neox_bf16()
    g = Guards()
    q, k = g.put(case.query, "query"), g.put(case.key, "key")
    R.rope_with_sin_cos_cache(g.put(case.positions, "positions"), q, k, g.put(case.cache, "cache"), case.head_size,
                              case.rotary_dim, case.is_neox, case.mrope_section, cache_mode=1)
    g.check()
    assert R.get_device_error() == 0
    qo, ko, skipped = oracle_cache_all_cores(case, cache_mode=1)
    assert skipped == 0
    assert_matches_rows(q.cpu(), qo, "interleaved splice query")
    assert_matches_rows(k.cpu(), ko, "interleaved splice key")
