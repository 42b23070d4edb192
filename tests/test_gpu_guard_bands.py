"""Guard bands (tests/guard.py) around every tensor of the calls most exposed to
a stray store: the V2 operator's separate outputs (whole rows written, pass-
through columns copied), q/k as strided row views of one fused QKV buffer (the
V heads between and after them must stay untouched), and the in-place operator
at misaligned addresses (narrower vector paths and the scalar pair kernel).
The fused QKV op's paged-cache scatter runs guarded in every test of
test_gpu_qkv.py.  Each case also checks parity with the oracle."""
import pytest
import torch

import oracle
import transformer_rope_positional_gb300 as R
import workloads as W
from guard import Guards
from parity import assert_matches, same_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("neox,hs,rot", [(True, 128, 64), (False, 256, 64), (True, 64, 64)])
@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_separate_outputs(rope_gpu, neox, hs, rot, dt):
    case = W.cache_case("guard_out", 201, 333, 3, 2, hs, rot, 500, dt, neox)
    g = Guards()
    q, k = g.put(case.query, "query"), g.put(case.key, "key")
    qo, ko = g.empty(case.query.shape, dt, "query_out"), g.empty(case.key.shape, dt, "key_out")
    R.rope_with_sin_cos_cache(g.put(case.positions, "positions"), q, k, g.put(case.cache, "cache"), hs, rot, neox,
                              query_out=qo, key_out=ko)
    g.check()
    want_q, want_k, _ = oracle.rope_with_sin_cos_cache(case.positions, case.query, case.key, case.cache, hs, neox)
    assert_matches(qo.cpu(), want_q, "query_out")
    assert_matches(ko.cpu(), want_k, "key_out")
    assert same_bits(q.cpu(), case.query) and same_bits(k.cpu(), case.key)  # inputs untouched


@pytest.mark.parametrize("neox", [True, False], ids=["neox", "gptj"])
@pytest.mark.parametrize("out", [False, True], ids=["in_place", "separate_outputs"])
def test_views_of_a_fused_qkv_buffer(rope_gpu, neox, out):
    T, hs, rot, nq, nk, nv = 257, 128, 64, 4, 2, 2
    case = W.cache_case("guard_views", 202, T, nq, nk, hs, rot, 400, torch.float16, neox)
    v = W.normal(203, (T, nv * hs), torch.float16)
    fused = torch.cat([case.query, case.key, v], dim=1)
    g = Guards()
    buf = g.put(fused, "fused qkv")
    q, k = buf[:, :nq * hs], buf[:, nq * hs:(nq + nk) * hs]
    kw = {}
    if out:
        kw = dict(query_out=g.empty(case.query.shape, torch.float16, "query_out"),
                  key_out=g.empty(case.key.shape, torch.float16, "key_out"))
    R.rope_with_sin_cos_cache(g.put(case.positions, "positions"), q, k, g.put(case.cache, "cache"), hs, rot, neox,
                              **kw)
    g.check()
    want_q, want_k, _ = oracle.rope_with_sin_cos_cache(case.positions, case.query, case.key, case.cache, hs, neox)
    got = buf.cpu()
    assert same_bits(got[:, (nq + nk) * hs:], v), "V heads changed"
    if out:
        assert same_bits(got, fused), "inputs changed"
        assert_matches(kw["query_out"].cpu(), want_q, "query_out")
        assert_matches(kw["key_out"].cpu(), want_k, "key_out")
    else:
        assert_matches(got[:, :nq * hs].contiguous(), want_q, "query")
        assert_matches(got[:, nq * hs:(nq + nk) * hs].contiguous(), want_k, "key")


def test_interleaved_splice_views_and_outputs_together(rope_gpu):
    T, hs = 190, 128
    section = [24, 20, 20]
    case = W.cache_case("guard_mrope", 204, T, 3, 1, hs, hs, 300, torch.bfloat16, True, mrope_section=section)
    extra = W.normal(205, (T, 2 * hs), torch.bfloat16)
    g = Guards()
    buf = g.put(torch.cat([case.query, case.key, extra], dim=1), "fused qkv")
    q, k = buf[:, :3 * hs], buf[:, 3 * hs:4 * hs]
    qo, ko = g.empty(case.query.shape, torch.bfloat16, "query_out"), g.empty(case.key.shape, torch.bfloat16, "key_out")
    R.rope_with_sin_cos_cache(g.put(case.positions, "positions"), q, k, g.put(case.cache, "cache"), hs, hs, True,
                              section, cache_mode=1, query_out=qo, key_out=ko)
    g.check()
    want_q, want_k, _ = oracle.rope_with_sin_cos_cache(case.positions, case.query, case.key, case.cache, hs, True,
                                                       section, cache_mode=1)
    assert_matches(qo.cpu(), want_q, "query_out")
    assert_matches(ko.cpu(), want_k, "key_out")


# x at byte offsets that leave it 2-, 4- or 8-byte aligned (cos/sin stay
# 16-byte aligned): bf16 +2, f16 +6 and f32 +4 take the scalar pair kernel,
# bf16 +4 and f32 +8 2-element vectors, bf16 +8 4-element vectors
@pytest.mark.parametrize("dt,offset", [(torch.bfloat16, 2), (torch.bfloat16, 4), (torch.bfloat16, 8),
                                       (torch.float16, 6), (torch.float32, 4), (torch.float32, 8)])
@pytest.mark.parametrize("mode", [1, 0], ids=["interleave", "half"])
@pytest.mark.parametrize("backward", [False, True], ids=["fwd", "bwd"])
def test_inplace_at_misaligned_addresses(rope_gpu, dt, offset, mode, backward):
    case = W.inplace_case("guard_inplace", 206, (2, 33, 5, 64), 8, 56, dt, torch.float32, cs_kind="randn")
    g = Guards()
    x = g.put(case.x, "x", offset=offset)
    c, s = g.put(case.cos, "cos", offset=16), g.put(case.sin, "sin", offset=32)
    fn = R.rope_inplace_partial_backward if backward else R.rope_inplace_partial
    fn(x, c, s, mode, [case.start, case.end])
    g.check()
    want = oracle.inplace_partial_rotary_mul(case.x, case.cos, case.sin, case.start, case.end, mode, backward)
    assert_matches(x.cpu(), want, "x")


def test_out_of_range_tokens_write_nothing(rope_gpu):
    case = W.cache_case("guard_bad_pos", 207, 64, 2, 2, 64, 64, 100, torch.float32, True)
    pos = case.positions.clone()
    pos[::5] = 100  # == maxSeqLen: out of range
    g = Guards()
    qo, ko = g.empty(case.query.shape, torch.float32, "query_out"), g.empty(case.key.shape, torch.float32, "key_out")
    R.rope_with_sin_cos_cache(g.put(pos, "positions"), g.put(case.query, "query"), g.put(case.key, "key"),
                              g.put(case.cache, "cache"), 64, 64, True, query_out=qo, key_out=ko)
    g.check()
    assert R.get_device_error() == R.ROPE_DEVICE_POSITION_OUT_OF_RANGE
    want_q, _, skipped = oracle.rope_with_sin_cos_cache(pos, case.query, case.key, case.cache, 64, True)
    assert skipped == 13
    got = qo.cpu()
    canary = g.empty((1,), torch.float32).cpu()
    assert same_bits(got[::5], canary.expand(13, got.shape[1]).contiguous())  # rows of skipped tokens unwritten
    keep = torch.ones(64, dtype=torch.bool)
    keep[::5] = False
    assert_matches(got[keep], want_q[keep], "query_out")
