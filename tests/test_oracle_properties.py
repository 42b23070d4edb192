"""Randomised pins of the CPU oracle (hypothesis): over random shapes, slices,
dtypes, broadcast layouts, head layouts and mrope sections, the oracle agrees
with the textbook complex-number form of RoPE, leaves every column outside the
rotated span bit-exact, and its backward undoes its forward.  The fixed-shape
pins in test_oracle_pins.py hold at chosen points; these hold anywhere the
generator reaches, so an index slip that only shows at an odd start, a
broadcast dim or an uneven section fails here.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from test_oracle_pins import _complex_cache, _complex_interleave, _same_bits, _ulp_dist

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")
given, settings = hyp.given, hyp.settings

DTYPES = [torch.float32, torch.float16, torch.bfloat16]
SETTINGS = dict(max_examples=150, deadline=None, derandomize=True)


@st.composite
def inplace_problems(draw):
    B, S, N = draw(st.integers(1, 3)), draw(st.integers(1, 6)), draw(st.integers(1, 4))
    D = 2 * draw(st.integers(1, 32))
    start = draw(st.integers(0, D - 2))
    L = 2 * draw(st.integers(1, (D - start) // 2))
    dt = draw(st.sampled_from(DTYPES))
    cs_dt = torch.float32 if dt == torch.float32 else draw(st.sampled_from([dt, torch.float32]))
    cs_shape = tuple(draw(st.sampled_from([1, n])) for n in (B, S, N)) + (L,)
    seed = draw(st.integers(0, 10_000))
    return (B, S, N, D), start, start + L, dt, cs_dt, cs_shape, seed


@settings(**SETTINGS)
@given(inplace_problems())
def test_inplace_matches_complex_form_anywhere(problem):
    shape, start, end, dt, cs_dt, cs_shape, seed = problem
    case = W.inplace_case("prop", seed, shape, start, end, dt, cs_dt, cs_shape=cs_shape)
    y = oracle.inplace_partial_rotary_mul(case.x, case.cos, case.sin, start, end)
    ref = oracle.round_to(_complex_interleave(case.x, case.cos, case.sin, start, end), dt)
    assert _ulp_dist(y[..., start:end], ref[..., start:end]).max() <= 1
    assert _same_bits(y[..., :start], case.x[..., :start]) and _same_bits(y[..., end:], case.x[..., end:])


@settings(**SETTINGS)
@given(inplace_problems(), st.sampled_from([0, 1]))
def test_inplace_backward_undoes_forward_anywhere(problem, mode):
    shape, start, end, _, _, cs_shape, seed = problem
    case = W.inplace_case("prop", seed, shape, start, end, torch.float32, torch.float32, cs_shape=cs_shape)
    cos, sin = case.cos, case.sin  # equal on (2p, 2p + 1): a rotation of the interleaved pairs
    if mode == 0:  # half mode pairs (i, i + L/2): the same angles laid out on the two halves
        cos = torch.cat([cos[..., 0::2], cos[..., 0::2]], dim=-1).contiguous()
        sin = torch.cat([sin[..., 0::2], sin[..., 0::2]], dim=-1).contiguous()
    y = oracle.inplace_partial_rotary_mul(case.x, cos, sin, start, end, rotary_mode=mode)
    x2 = oracle.inplace_partial_rotary_mul(y, cos, sin, start, end, rotary_mode=mode, backward=True)
    # a rotation's transpose is its inverse: two binary32 roundings per element
    assert np.allclose(x2.double().numpy(), case.x.double().numpy(), rtol=8 * 2.0 ** -23, atol=1e-6)


@st.composite
def cache_problems(draw):
    dt = draw(st.sampled_from(DTYPES))
    head_size = draw(st.sampled_from([16, 32, 64, 96, 128]))
    R = 2 * draw(st.integers(1, head_size // 2))
    is_neox = draw(st.booleans())
    section = None
    if draw(st.booleans()):  # mrope: 3 or 4 sections, the first non-empty, summing to R/2
        m = draw(st.sampled_from([3, 4]))
        cuts = sorted(draw(st.lists(st.integers(0, R // 2), min_size=m - 1, max_size=m - 1)))
        parts = [b - a for a, b in zip([0] + cuts, cuts + [R // 2])]
        if parts[0] > 0:
            section = parts
    T, hq, hk = draw(st.integers(1, 20)), draw(st.integers(1, 4)), draw(st.integers(1, 3))
    return dt, head_size, R, is_neox, section, T, hq, hk, draw(st.integers(0, 10_000))


@settings(**SETTINGS)
@given(cache_problems())
def test_cache_matches_complex_form_anywhere(problem):
    dt, hs, R, is_neox, section, T, hq, hk, seed = problem
    c = W.cache_case("prop", seed, T, hq, hk, hs, R, 97, dt, is_neox, mrope_section=section)
    qo, ko, skipped = oracle.rope_with_sin_cos_cache(c.positions, c.query, c.key, c.cache, hs, is_neox, section)
    assert skipped == 0
    rows = c.positions.numpy() if section else c.positions.numpy()[None, :]
    for got, x in ((qo, c.query), (ko, c.key)):
        ref = oracle.round_to(_complex_cache(x, rows, c.cache, hs, R, is_neox, section), dt)
        assert _ulp_dist(got, ref).max() <= 1
        heads_got, heads_x = got.reshape(T, -1, hs), x.reshape(T, -1, hs)
        assert _same_bits(heads_got[..., R:], heads_x[..., R:])


@st.composite
def qkv_problems(draw):
    dt = draw(st.sampled_from(DTYPES))
    D = draw(st.sampled_from([16, 32, 64, 96, 128]))
    nq, nk, nv = draw(st.integers(0, 5)), draw(st.integers(0, 3)), draw(st.integers(0, 3))
    if nq + nk + nv == 0:
        nq = 1
    B = draw(st.integers(1, 6))
    qlens = draw(st.lists(st.integers(0, 9), min_size=B, max_size=B))
    if sum(qlens) == 0:
        qlens[0] = 1
    ctx = draw(st.lists(st.integers(0, 60), min_size=B, max_size=B))
    block = draw(st.sampled_from([1, 3, 4, 16]))
    pad = draw(st.sampled_from([0, 0, 2, 5]))
    return dt, D, nq, nk, nv, qlens, ctx, block, pad, draw(st.integers(0, 10_000))


@settings(**SETTINGS)
@given(qkv_problems())
def test_fused_qkv_matches_independent_composition_anywhere(problem):
    from test_oracle_pins import _qkv_reference
    dt, D, nq, nk, nv, qlens, ctx, block, pad, seed = problem
    case = W.qkv_case("prop", seed, qlens, ctx, nq, nk, nv, D, block, dt, pad_every=pad)
    qo, kc, vc, bad_pos, bad_slot = oracle.qkv_rmsnorm_rope_cache(
        case.qkv, case.nq, case.nk, case.nv, case.q_gamma, case.k_gamma, case.eps, case.cache, case.seq_lens,
        case.query_start_loc, case.slot_mapping, case.q_out, case.k_cache, case.v_cache)
    assert bad_pos == 0 and bad_slot == 0
    rq, rk, rv = _qkv_reference(case)
    # one rounding on each side of a float64 computation: within one ulp (a
    # branch with no heads gives an empty tensor, nothing to compare)
    for got, ref in ((qo, rq), (kc, rk)):
        if got.numel():
            assert _ulp_dist(got, oracle.round_to(ref, dt)).max() <= 1
    assert _same_bits(vc, oracle.round_to(rv, dt))
