"""Parity of the V2 cache-indexed entry point: interleaved mrope splice
(cacheMode 1), strided query/key rows, separate outputs."""
import pytest
import torch

import oracle
import transformer_rope_positional_gb300 as R
import workloads as W
from parity import assert_matches, same_bits

pytestmark = pytest.mark.gpu

DTYPES = [torch.float32, torch.float16, torch.bfloat16]
SECTIONS = [[24, 20, 20], [16, 24, 24], [11, 11, 10], [8, 12, 12]]


def _gpu(case, positions=None, **kw):
    pos = (case.positions if positions is None else positions).cuda()
    q, k = case.query.cuda(), case.key.cuda()
    R.rope_with_sin_cos_cache(pos, q, k, case.cache.cuda(), case.head_size, case.rotary_dim, case.is_neox,
                              case.mrope_section, **kw)
    torch.cuda.synchronize()
    return q.cpu(), k.cpu()


@pytest.mark.parametrize("section", SECTIONS, ids=["_".join(map(str, s)) for s in SECTIONS])
@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("neox", [True, False], ids=["neox", "gptj"])
def test_interleaved_splice(rope_gpu, section, dt, neox):
    R_ = 2 * sum(section)
    case = W.cache_case("v2", 111, 53, 3, 2, R_, R_, 300, dt, neox, mrope_section=section)
    qg, kg = _gpu(case, cache_mode=1)
    qo, ko, sk = oracle.rope_with_sin_cos_cache(case.positions, case.query, case.key, case.cache, R_, neox,
                                                section, cache_mode=1)
    assert sk == 0
    assert_matches(qg, qo, "query")
    assert_matches(kg, ko, "key")
    assert R.get_device_error() == 0


def test_interleaved_splice_equal_rows_is_rope(rope_gpu):
    case = W.cache_case("v2eq", 112, 200, 4, 2, 128, 128, 500, torch.bfloat16, True)
    qa, ka = _gpu(case)
    pos3 = case.positions[None, :].expand(3, -1).contiguous()
    case.mrope_section = [24, 20, 20]
    qb, kb = _gpu(case, positions=pos3, cache_mode=1)
    assert same_bits(qa, qb) and same_bits(ka, kb)


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("neox", [True, False], ids=["neox", "gptj"])
def test_strided_views_of_fused_qkv(rope_gpu, dt, neox):
    T, hq, hk, hv = 77, 4, 2, 2
    hs, R_ = (64, 32) if dt == torch.float32 else (128, 64)
    qkv = W.normal(113, (T, (hq + hk + hv) * hs), dt)
    case = W.cache_case("fused", 114, T, hq, hk, hs, R_, 256, dt, neox)
    dev = qkv.cuda()
    q = dev[:, :hq * hs]
    k = dev[:, hq * hs:(hq + hk) * hs]
    R.rope_with_sin_cos_cache(case.positions.cuda(), q, k, case.cache.cuda(), hs, R_, neox)
    torch.cuda.synchronize()
    out = dev.cpu()
    qo, ko, _ = oracle.rope_with_sin_cos_cache(case.positions, qkv[:, :hq * hs].contiguous(),
                                               qkv[:, hq * hs:(hq + hk) * hs].contiguous(), case.cache, hs, neox)
    assert_matches(out[:, :hq * hs].contiguous(), qo, "q view")
    assert_matches(out[:, hq * hs:(hq + hk) * hs].contiguous(), ko, "k view")
    assert same_bits(out[:, (hq + hk) * hs:], qkv[:, (hq + hk) * hs:])  # v untouched


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("neox", [True, False], ids=["neox", "gptj"])
def test_out_of_place(rope_gpu, dt, neox):
    hs, R_ = (64, 32) if dt == torch.float32 else (256, 64)
    case = W.cache_case("oop", 115, 91, 3, 1, hs, R_, 300, dt, neox)
    q, k = case.query.cuda(), case.key.cuda()
    qo = torch.full_like(q, float("nan"))
    ko = torch.full_like(k, float("nan"))
    R.rope_with_sin_cos_cache(case.positions.cuda(), q, k, case.cache.cuda(), hs, R_, neox, query_out=qo,
                              key_out=ko)
    torch.cuda.synchronize()
    assert same_bits(q.cpu(), case.query) and same_bits(k.cpu(), case.key)  # inputs untouched
    qr, kr, _ = oracle.rope_with_sin_cos_cache(case.positions, case.query, case.key, case.cache, hs, neox)
    assert_matches(qo.cpu(), qr, "query_out")
    assert_matches(ko.cpu(), kr, "key_out")
    # pass-through columns copied bit-exactly
    assert same_bits(qo.cpu().view(91, -1, hs)[..., R_:], case.query.view(91, -1, hs)[..., R_:])


def test_out_of_place_strided_interleaved_together(rope_gpu):
    T, hq, hk, hs = 64, 4, 2, 128
    section = [24, 20, 20]
    case = W.cache_case("all", 116, T, hq, hk, hs, hs, 400, torch.bfloat16, True, mrope_section=section)
    qkv = torch.cat([case.query, case.key, W.normal(117, (T, 2 * hs), torch.bfloat16)], dim=1).cuda()
    q, k = qkv[:, :hq * hs], qkv[:, hq * hs:(hq + hk) * hs]
    qo = torch.empty(T, hq * hs, dtype=torch.bfloat16, device="cuda")
    ko = torch.empty(T, hk * hs, dtype=torch.bfloat16, device="cuda")
    before = qkv.cpu()
    R.rope_with_sin_cos_cache(case.positions.cuda(), q, k, case.cache.cuda(), hs, hs, True, section, cache_mode=1,
                              query_out=qo, key_out=ko)
    torch.cuda.synchronize()
    assert same_bits(qkv.cpu(), before)
    qr, kr, _ = oracle.rope_with_sin_cos_cache(case.positions, case.query, case.key, case.cache, hs, True, section,
                                               cache_mode=1)
    assert_matches(qo.cpu(), qr, "query_out")
    assert_matches(ko.cpu(), kr, "key_out")


def test_output_equal_to_input_means_in_place(rope_gpu):
    case = W.cache_case("alias", 118, 33, 2, 2, 64, 64, 100, torch.float16, True)
    q, k = case.query.cuda(), case.key.cuda()
    R.rope_with_sin_cos_cache(case.positions.cuda(), q, k, case.cache.cuda(), 64, query_out=q, key_out=k)
    torch.cuda.synchronize()
    qr, kr, _ = oracle.rope_with_sin_cos_cache(case.positions, case.query, case.key, case.cache, 64, True)
    assert_matches(q.cpu(), qr, "q")
    assert_matches(k.cpu(), kr, "k")


def test_overlapping_output_rejected(rope_gpu):
    case = W.cache_case("overlap", 119, 8, 2, 2, 64, 64, 100, torch.float16, True)
    buf = torch.zeros(8 * 512, dtype=torch.float16, device="cuda")
    q = buf[:8 * 128].view(8, 128)
    with pytest.raises(R.RopeError):
        R.rope_with_sin_cos_cache(case.positions.cuda(), q, case.key.cuda(), case.cache.cuda(), 64,
                                  query_out=buf[64:64 + 8 * 128].view(8, 128), key_out=torch.empty_like(q))


def test_out_of_place_out_of_range_token_leaves_output_unwritten(rope_gpu):
    case = W.cache_case("oob_oop", 120, 6, 1, 1, 64, 64, 20, torch.bfloat16, True)
    pos = case.positions.clone()
    pos[3] = 20
    q, k = case.query.cuda(), case.key.cuda()
    qo = torch.full_like(q, 7.0)
    ko = torch.full_like(k, 7.0)
    R.rope_with_sin_cos_cache(pos.cuda(), q, k, case.cache.cuda(), 64, query_out=qo, key_out=ko)
    assert R.get_device_error() == R.ROPE_DEVICE_POSITION_OUT_OF_RANGE
    assert torch.all(qo[3].cpu() == 7.0) and torch.all(ko[3].cpu() == 7.0)
    qr, _, sk = oracle.rope_with_sin_cos_cache(pos, case.query, case.key, case.cache, 64, True)
    assert sk == 1
    keep = [0, 1, 2, 4, 5]
    assert_matches(qo.cpu()[keep], qr[keep], "other tokens")
