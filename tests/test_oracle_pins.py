"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each pin is chosen so that a plausible slip in ``oracle/rope_oracle.c`` (a
dropped term, a wrong sign, a wrong pair index, a transposed operand, a wrong
section boundary, a rounding mistake) fails at least one test:

* number formats: exhaustive decoding against numpy/torch, rounding against
  numpy's double->half and torch's float->bfloat16 conversions;
* hand-worked cases stored under ``tests/golden`` with their page citations;
* the textbook complex-number form of RoPE (a pair (u, v) rotated by angle a is
  (u + iv) * exp(ia)), computed with numpy complex arithmetic;
* invariants: identity, per-pair norm, rotate then un-rotate, NeoX vs GPT-J
  under the even/odd permutation, mrope with equal rows vs rope, no-op and
  pass-through bytes.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
DTYPES = [torch.float32, torch.float16, torch.bfloat16]


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _same_bits(a: torch.Tensor, b: torch.Tensor) -> bool:
    bits = {4: torch.int32, 2: torch.int16}[a.element_size()]
    return torch.equal(a.contiguous().view(bits), b.contiguous().view(bits))


def _ulp_dist(a: torch.Tensor, b: torch.Tensor) -> np.ndarray:
    """Distance in units in the last place between two same-dtype tensors
    (+0 and -0 are equal; NaN against NaN is 0, NaN against a number is huge)."""
    bits = {4: np.int64, 2: np.int64}[a.element_size()]
    view = {4: torch.int32, 2: torch.int16}[a.element_size()]
    ia = a.contiguous().view(view).numpy().astype(bits)
    ib = b.contiguous().view(view).numpy().astype(bits)
    nbits = 8 * a.element_size()
    mask = (1 << nbits) - 1
    ia &= mask
    ib &= mask
    sign = 1 << (nbits - 1)

    def ordered(u):
        return np.where(u & sign, -(u & (sign - 1)), u)

    d = np.abs(ordered(ia) - ordered(ib))
    na = torch.isnan(a.float()).numpy()
    nb = torch.isnan(b.float()).numpy()
    d = np.where(na & nb, 0, d)
    d = np.where(na ^ nb, 1 << 40, d)
    return d.reshape(tuple(a.shape))


# ----------------------------------------------------------------------------
# number formats
# ----------------------------------------------------------------------------

def test_decode_binary16_exhaustive():
    bits = np.arange(1 << 16, dtype=np.uint32)
    got = np.array([oracle.decode(int(b), torch.float16) for b in bits])
    ref = bits.astype(np.uint16).view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


def test_decode_bfloat16_exhaustive():
    bits = np.arange(1 << 16, dtype=np.uint32)
    got = np.array([oracle.decode(int(b), torch.bfloat16) for b in bits])
    ref = torch.from_numpy(bits.astype(np.uint16).view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


def test_decode_binary32_sampled():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 32, size=20000, dtype=np.uint64).astype(np.uint32)
    bits[:8] = [0, 0x80000000, 1, 0x807FFFFF, 0x7F800000, 0xFF800000, 0x7F7FFFFF, 0x00800000]
    got = np.array([oracle.decode(int(b), torch.float32) for b in bits])
    with np.errstate(invalid="ignore"):
        ref = bits.view(np.float32).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def _interesting_doubles(n, lo_exp, hi_exp, seed):
    rng = np.random.default_rng(seed)
    mags = np.ldexp(rng.uniform(1.0, 2.0, n), rng.integers(lo_exp, hi_exp, n))
    return mags * rng.choice([-1.0, 1.0], n)


def test_encode_binary16_against_numpy():
    vals = list(_interesting_doubles(30000, -27, 17, 1))
    # exact ties between neighbouring halves, around 1, in the subnormals and at overflow
    for b in [0x3C00, 0x3C01, 0x0001, 0x0002, 0x03FF, 0x7BFE, 0x7BFF, 0x0400]:
        lo = float(np.uint16(b).view(np.float16))
        hi = float(np.uint16(b + 1).view(np.float16))
        vals += [(lo + hi) / 2, -(lo + hi) / 2, np.nextafter((lo + hi) / 2, 0.0)]
    vals += [0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e9, -1e9, 2.0 ** -25, 2.0 ** -26, 1e-30,
             math.inf, -math.inf]
    got = np.array([oracle.encode(v, torch.float16) for v in vals], dtype=np.uint32)
    with np.errstate(over="ignore"):
        ref = np.array(vals, dtype=np.float64).astype(np.float16).view(np.uint16).astype(np.uint32)
    assert np.array_equal(got, ref)


def test_encode_bfloat16_against_torch():
    # binary32-representable inputs, so torch's float->bfloat16 rounding is a single rounding
    f32 = _interesting_doubles(30000, -140, 127, 2).astype(np.float32)
    extra = []
    for b in [0x3F80, 0x3F81, 0x0001, 0x007F, 0x7F7E, 0x4049]:
        lo = np.uint32(b << 16).view(np.float32)
        hi = np.uint32((b + 1) << 16).view(np.float32)
        mid = np.float32((np.float64(lo) + np.float64(hi)) / 2)
        extra += [mid, -mid]
    f32 = np.concatenate([f32, np.array(extra, dtype=np.float32),
                          np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38], dtype=np.float32)])
    got = np.array([oracle.encode(float(v), torch.bfloat16) for v in f32], dtype=np.uint32)
    ref = torch.from_numpy(f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref.astype(np.uint32))


def test_encode_binary32_against_numpy():
    vals = _interesting_doubles(30000, -155, 128, 3)
    got = np.array([oracle.encode(float(v), torch.float32) for v in vals], dtype=np.uint32)
    ref = vals.astype(np.float32).view(np.uint32)
    assert np.array_equal(got, ref)


def test_encode_nan_stays_nan():
    for dt in DTYPES:
        bits = oracle.encode(float("nan"), dt)
        assert math.isnan(oracle.decode(bits, dt))


# ----------------------------------------------------------------------------
# in-place partial interleave operator
# ----------------------------------------------------------------------------

def test_inplace_hand_cases():
    g = _load("inplace_pair_hand_cases.json")
    for case in g["cases"]:
        x = torch.tensor(case["x"], dtype=torch.float32).reshape(1, 1, 1, 2)
        c = torch.tensor(case["cos"], dtype=torch.float32).reshape(1, 1, 1, 2)
        s = torch.tensor(case["sin"], dtype=torch.float32).reshape(1, 1, 1, 2)
        y = oracle.inplace_partial_rotary_mul(x, c, s, 0, 0)
        assert y.reshape(-1).tolist() == case["y"], case


def _complex_interleave(x, cos, sin, start, end):
    """Textbook complex form: pair (x[2p], x[2p+1]) times exp(i*angle); needs cos/sin
    equal on the two members of a pair (a true rotation)."""
    x = x.double().numpy().copy()
    L = end - start
    c = np.broadcast_to(cos.double().numpy(), x.shape[:3] + (L,))
    s = np.broadcast_to(sin.double().numpy(), x.shape[:3] + (L,))
    z = x[..., start:end:2] + 1j * x[..., start + 1:end:2]
    w = c[..., 0::2] + 1j * s[..., 0::2]
    r = z * w
    x[..., start:end:2] = r.real
    x[..., start + 1:end:2] = r.imag
    return x


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("cs_dt", [None, torch.float32])
@pytest.mark.parametrize("cs_shape", [(1, 5, 1, 16), (2, 5, 3, 16), (2, 1, 3, 16), (1, 1, 1, 16)])
def test_inplace_matches_complex_form(dt, cs_dt, cs_shape):
    cs_dt = cs_dt or dt
    case = W.inplace_case("t", 11, (2, 5, 3, 24), 6, 22, dt, cs_dt, cs_shape=cs_shape)
    y = oracle.inplace_partial_rotary_mul(case.x, case.cos, case.sin, 6, 22)
    ref = oracle.round_to(_complex_interleave(case.x, case.cos, case.sin, 6, 22), dt)
    assert _ulp_dist(y, ref).max() <= 1


def test_inplace_identity():
    for dt in DTYPES:
        x = W.normal(5, (2, 3, 4, 16), dt)
        c = torch.ones(1, 3, 1, 16, dtype=dt)
        s = torch.zeros(1, 3, 1, 16, dtype=dt)
        y = oracle.inplace_partial_rotary_mul(x, c, s, 0, 16)
        assert torch.equal(y.float(), x.float())


def test_inplace_noop_and_whole_axis():
    case = W.inplace_f32_small("slice")
    y = oracle.inplace_partial_rotary_mul(case.x, case.cos, case.sin, 8, 8)
    assert _same_bits(y, case.x)
    full = W.inplace_f32_small("full")
    a = oracle.inplace_partial_rotary_mul(full.x, full.cos, full.sin, 0, 0)
    b = oracle.inplace_partial_rotary_mul(full.x, full.cos, full.sin, 0, 64)
    assert _same_bits(a, b)
    assert not _same_bits(a, full.x)


def test_inplace_columns_outside_slice_untouched():
    case = W.inplace_case("t", 3, (2, 4, 3, 32), 10, 26, torch.float16, torch.float32)
    x = case.x.clone()
    payload = torch.tensor([0x7E01 + i for i in range(32)], dtype=torch.int32).to(torch.int16)
    x.view(torch.int16)[..., :10] = payload[:10]
    x.view(torch.int16)[..., 26:] = payload[26:]
    y = oracle.inplace_partial_rotary_mul(x, case.cos, case.sin, 10, 26)
    assert _same_bits(y[..., :10], x[..., :10])
    assert _same_bits(y[..., 26:], x[..., 26:])
    assert not _same_bits(y[..., 10:26], x[..., 10:26])


def test_inplace_pair_norm_and_inverse():
    case = W.inplace_f32_small("slice")
    y = oracle.inplace_partial_rotary_mul(case.x, case.cos, case.sin, 16, 48)
    xs = case.x[..., 16:48].double().numpy()
    ys = y[..., 16:48].double().numpy()
    nx = np.hypot(xs[..., 0::2], xs[..., 1::2])
    ny = np.hypot(ys[..., 0::2], ys[..., 1::2])
    assert np.allclose(ny, nx, rtol=4 * 2.0 ** -23, atol=0)
    back = oracle.inplace_partial_rotary_mul(y, case.cos, -case.sin, 16, 48)
    assert np.allclose(back.double().numpy(), case.x.double().numpy(), rtol=8 * 2.0 ** -23, atol=1e-7)


def test_inplace_literal_cat_is_not_a_rotation():
    """Documents reading (1): taking the formula's cat literally mixes x[j] with
    x[2j+1] and does not keep pair norms, which the interleave reading does."""
    case = W.inplace_f32_small("slice")
    xs = case.x[..., 16:48].double().numpy()
    c = np.broadcast_to(case.cos.double().numpy(), xs.shape)
    s = np.broadcast_to(case.sin.double().numpy(), xs.shape)
    rot = np.concatenate([-xs[..., 1::2], xs[..., 0::2]], axis=-1)
    lit = xs * c + rot * s
    n_in = np.hypot(xs[..., 0::2], xs[..., 1::2])
    n_lit = np.hypot(lit[..., 0::2], lit[..., 1::2])
    assert not np.allclose(n_lit, n_in, rtol=1e-3)


def test_inplace_element_index_mapping():
    """Unit vectors against distinct per-element cos/sin: e_{2p} -> (c[2p], s[2p+1]);
    e_{2p+1} -> (-s[2p], c[2p+1])."""
    L = 8
    c = torch.arange(1, L + 1, dtype=torch.float32).reshape(1, 1, 1, L) / 16
    s = torch.arange(101, 101 + L, dtype=torch.float32).reshape(1, 1, 1, L) / 128
    for j in range(L):
        x = torch.zeros(1, 1, 1, L)
        x[..., j] = 1.0
        y = oracle.inplace_partial_rotary_mul(x, c, s, 0, L).reshape(-1)
        p, odd = divmod(j, 2)
        want = torch.zeros(L)
        if odd == 0:
            want[2 * p], want[2 * p + 1] = c[0, 0, 0, 2 * p], s[0, 0, 0, 2 * p + 1]
        else:
            want[2 * p], want[2 * p + 1] = -s[0, 0, 0, 2 * p], c[0, 0, 0, 2 * p + 1]
        assert torch.equal(y, want), j


def test_inplace_broadcast_equals_expanded():
    case = W.inplace_case("t", 7, (3, 4, 5, 16), 0, 16, torch.bfloat16, torch.bfloat16,
                          cs_shape=(3, 1, 5, 16), cs_kind="randn")
    a = oracle.inplace_partial_rotary_mul(case.x, case.cos, case.sin, 0, 16)
    ce = case.cos.expand(3, 4, 5, 16).contiguous()
    se = case.sin.expand(3, 4, 5, 16).contiguous()
    b = oracle.inplace_partial_rotary_mul(case.x, ce, se, 0, 16)
    assert _same_bits(a, b)


def test_inplace_closed_form_rotation():
    """x = e_{2p} at position pos -> (cos(pos*theta_p), sin(pos*theta_p)) with
    theta_p = 10000^(-2p/L), against numpy's cos/sin in binary64."""
    case = W.inplace_f32_small("slice")
    L = 32
    x = torch.zeros(1, 16, 1, L)
    for p in range(L // 2):
        x.zero_()
        x[..., 2 * p] = 1.0
        y = oracle.inplace_partial_rotary_mul(x, case.cos, case.sin, 0, L)
        ang = np.arange(16) * 10000.0 ** (-2.0 * p / L)
        assert np.allclose(y[0, :, 0, 2 * p].double().numpy(), np.cos(ang), rtol=0, atol=2.0 ** -24)
        assert np.allclose(y[0, :, 0, 2 * p + 1].double().numpy(), np.sin(ang), rtol=0, atol=2.0 ** -24)


# ----------------------------------------------------------------------------
# cache-indexed operator
# ----------------------------------------------------------------------------

def test_cache_worked_example():
    g = _load("rope_cache_worked_example_bf16.json")
    dt = torch.bfloat16
    q = torch.full(g["query_shape"], g["fill"], dtype=dt)
    k = torch.full(g["key_shape"], g["fill"], dtype=dt)
    cache = torch.full(g["cache_shape"], g["fill"], dtype=dt)
    pos = torch.tensor(g["positions"], dtype=torch.int64)
    qo, ko, skipped = oracle.rope_with_sin_cos_cache(pos, q, k, cache, g["head_size"], g["is_neox"])
    assert skipped == 0
    for t in (qo, ko):
        for row in t:
            assert row.float().tolist() == [float(v) for v in g["expected_row"]]


def _complex_cache(x, pos_rows, cache, head_size, R, is_neox, section=None):
    x = x.double().numpy().copy()
    T = x.shape[0]
    half = R // 2
    tab = cache.double().numpy()
    if section is None:
        cos = tab[pos_rows[0], :half]
        sin = tab[pos_rows[0], half:]
    else:
        owner = np.repeat(np.arange(len(section)), section)  # section of each cos index
        rows = np.asarray(pos_rows)[owner, :].T               # [T, half] position per index
        idx = np.arange(half)[None, :]
        cos = tab[rows, idx]
        sin = tab[rows, half + idx]
    heads = x.reshape(T, -1, head_size)
    if is_neox:
        z = heads[..., :half] + 1j * heads[..., half:R]
    else:
        z = heads[..., 0:R:2] + 1j * heads[..., 1:R:2]
    r = z * (cos + 1j * sin)[:, None, :]
    if is_neox:
        heads[..., :half], heads[..., half:R] = r.real, r.imag
    else:
        heads[..., 0:R:2], heads[..., 1:R:2] = r.real, r.imag
    return heads.reshape(T, -1)


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("is_neox", [True, False])
def test_cache_matches_complex_form(dt, is_neox):
    c = W.cache_case("t", 21, 37, 3, 2, 64, 32, 300, dt, is_neox)
    qo, ko, sk = oracle.rope_with_sin_cos_cache(c.positions, c.query, c.key, c.cache, 64, is_neox)
    assert sk == 0
    pr = c.positions.numpy()[None, :]
    for got, x in ((qo, c.query), (ko, c.key)):
        ref = oracle.round_to(_complex_cache(x, pr, c.cache, 64, 32, is_neox), dt)
        assert _ulp_dist(got, ref).max() <= 1
        # pass-through columns [R, head_size) of every head
        assert _same_bits(got.reshape(37, -1, 64)[..., 32:], x.reshape(37, -1, 64)[..., 32:])


@pytest.mark.parametrize("section", [[16, 24, 24], [11, 11, 10], [16, 16, 16, 16]])
def test_mrope_matches_complex_form(section):
    R = 2 * sum(section)
    m = len(section)
    c = W.cache_case("t", 22, 29, 2, 1, R, R, 500, torch.float32, True, mrope_section=section)
    qo, ko, sk = oracle.rope_with_sin_cos_cache(c.positions, c.query, c.key, c.cache, R, True, section)
    assert sk == 0 and c.positions.shape == (m, 29)
    for got, x in ((qo, c.query), (ko, c.key)):
        ref = oracle.round_to(_complex_cache(x, c.positions.numpy(), c.cache, R, R, True, section),
                              torch.float32)
        assert _ulp_dist(got, ref).max() <= 1


def test_mrope_section_map_hand_case():
    g = _load("mrope_section_map_hand_case.json")
    R = g["rotary_dim"]
    half = R // 2
    cache = torch.zeros(5, R)
    for r in range(5):
        cache[r, :half] = torch.arange(half) + 10 * r
    q = torch.ones(1, R)
    k = torch.ones(1, R)
    for key, spec in g["sections"].items():
        sec = [int(v) for v in key.split(",")]
        pos = torch.tensor(g["positions"], dtype=torch.int64)
        if sec[0] == 0:
            pos = pos[0]
        qo, ko, _ = oracle.rope_with_sin_cos_cache(pos, q, k, cache, R, True, sec)
        want = spec["expected_cos"] * 2
        assert qo.reshape(-1).tolist() == want and ko.reshape(-1).tolist() == want, key
    fr = g["four_rows"]
    qo, _, _ = oracle.rope_with_sin_cos_cache(torch.tensor(fr["positions"]), q, k, cache, R, True,
                                              fr["section"])
    assert qo.reshape(-1).tolist() == fr["expected_cos"] * 2


def test_mrope_equal_rows_is_rope():
    c = W.cache_case("t", 23, 41, 3, 2, 128, 128, 700, torch.bfloat16, True)
    pos3 = c.positions[None, :].expand(3, -1).contiguous()
    a = oracle.rope_with_sin_cos_cache(c.positions, c.query, c.key, c.cache, 128, True)
    b = oracle.rope_with_sin_cos_cache(pos3, c.query, c.key, c.cache, 128, True, [16, 24, 24])
    assert _same_bits(a[0], b[0]) and _same_bits(a[1], b[1])


def test_neox_equals_gptj_under_even_odd_permutation():
    R, hs = 64, 96
    c = W.cache_case("t", 24, 19, 2, 3, hs, R, 128, torch.float16, False)

    def deinterleave(x):  # rotary dims: evens first, then odds (the NeoX halves)
        h = x.reshape(x.shape[0], -1, hs).clone()
        h[..., :R] = torch.cat([h[..., 0:R:2], h[..., 1:R:2]], dim=-1)
        return h.reshape(x.shape[0], -1)

    qj, kj, _ = oracle.rope_with_sin_cos_cache(c.positions, c.query, c.key, c.cache, hs, False)
    qn, kn, _ = oracle.rope_with_sin_cos_cache(c.positions, deinterleave(c.query),
                                               deinterleave(c.key), c.cache, hs, True)
    assert _same_bits(qn, deinterleave(qj)) and _same_bits(kn, deinterleave(kj))


def test_cache_identity_and_inverse():
    c = W.cache_case("t", 25, 23, 2, 2, 64, 64, 256, torch.float32, True)
    ident = torch.cat([torch.ones(256, 32), torch.zeros(256, 32)], dim=1)
    qo, ko, _ = oracle.rope_with_sin_cos_cache(c.positions, c.query, c.key, ident, 64, True)
    assert torch.equal(qo, c.query) and torch.equal(ko, c.key)
    inv = c.cache.clone()
    inv[:, 32:] = -inv[:, 32:]
    q1, k1, _ = oracle.rope_with_sin_cos_cache(c.positions, c.query, c.key, c.cache, 64, True)
    q2, _, _ = oracle.rope_with_sin_cos_cache(c.positions, q1, k1, inv, 64, True)
    assert np.allclose(q2.double().numpy(), c.query.double().numpy(), rtol=8 * 2.0 ** -23, atol=1e-7)
    h1 = q1.double().numpy().reshape(23, -1, 64)
    h0 = c.query.double().numpy().reshape(23, -1, 64)
    assert np.allclose(np.hypot(h1[..., :32], h1[..., 32:]), np.hypot(h0[..., :32], h0[..., 32:]),
                       rtol=4 * 2.0 ** -23)


def test_cache_closed_form_basis_vectors():
    """NeoX, x = e_i at position p -> cos(p*theta_i) at i and sin(p*theta_i) at i + R/2."""
    R = 32
    cache = W.cos_sin_cache(64, R, 10000.0, torch.float32)
    pos = torch.tensor([0, 5, 63], dtype=torch.int64)
    for i in range(R // 2):
        q = torch.zeros(3, R)
        q[:, i] = 1.0
        qo, _, _ = oracle.rope_with_sin_cos_cache(pos, q, q.clone(), cache, R, True)
        ang = pos.double().numpy() * 10000.0 ** (-2.0 * i / R)
        assert np.allclose(qo[:, i].double().numpy(), np.cos(ang), atol=2.0 ** -24, rtol=0)
        assert np.allclose(qo[:, i + R // 2].double().numpy(), np.sin(ang), atol=2.0 ** -24, rtol=0)


def test_cache_out_of_range_positions_left_untouched():
    c = W.cache_case("t", 26, 6, 1, 1, 32, 32, 16, torch.bfloat16, True)
    pos = c.positions.clone()
    pos[1] = 16
    pos[4] = -1
    qo, ko, sk = oracle.rope_with_sin_cos_cache(pos, c.query, c.key, c.cache, 32, True)
    assert sk == 2
    for t in (1, 4):
        assert _same_bits(qo[t], c.query[t]) and _same_bits(ko[t], c.key[t])


def test_special_values_propagate():
    q = torch.tensor([[float("inf"), 1.0, float("nan"), 2.0]], dtype=torch.float32)
    cache = torch.tensor([[0.5, 0.25, 0.5, 0.75]], dtype=torch.float32)  # cos=(.5,.25) sin=(.5,.75)
    qo, _, _ = oracle.rope_with_sin_cos_cache(torch.tensor([0]), q, q.clone(), cache, 4, True)
    # pair (inf, nan) and pair (1, 2)
    assert math.isnan(qo[0, 0]) and math.isnan(qo[0, 2])
    assert qo[0, 1].item() == 1.0 * 0.25 - 2.0 * 0.75 and qo[0, 3].item() == 2.0 * 0.25 + 1.0 * 0.75


# ----------------------------------------------------------------------------
# in-place operator: half mode (rotary_mode 0) and backward
# ----------------------------------------------------------------------------

def test_half_mode_and_backward_hand_cases():
    g = _load("inplace_half_and_backward_hand_cases.json")

    def t(v):
        return torch.tensor(v, dtype=torch.float32).reshape(1, 1, 1, -1)

    hf = g["half_forward"]
    y = oracle.inplace_partial_rotary_mul(t(hf["x"]), t(hf["cos"]), t(hf["sin"]), 0, 0, rotary_mode=0)
    assert y.reshape(-1).tolist() == hf["y"]
    hb = g["half_backward"]
    dx = oracle.inplace_partial_rotary_mul(t(hb["g"]), t(hb["cos"]), t(hb["sin"]), 0, 0, rotary_mode=0,
                                           backward=True)
    assert dx.reshape(-1).tolist() == hb["dx"]
    ib = g["interleave_backward"]
    dx = oracle.inplace_partial_rotary_mul(t(ib["g"]), t(ib["cos"]), t(ib["sin"]), 0, 0, rotary_mode=1,
                                           backward=True)
    assert dx.reshape(-1).tolist() == ib["dx"]


def _half_rotation_tables(rows, L, base=10000.0):
    """cos/sin for half mode: index i and i + L/2 share the angle rows*theta_i."""
    i = np.arange(L) % (L // 2)
    theta = base ** (-2.0 * i / L)
    ang = np.arange(rows, dtype=np.float64)[:, None] * theta[None, :]
    return np.cos(ang), np.sin(ang)


@pytest.mark.parametrize("dt", DTYPES)
def test_half_mode_matches_complex_form(dt):
    B, S, N, D, st, en = 2, 6, 3, 40, 8, 32
    L = en - st
    x = W.normal(77, (B, S, N, D), dt)
    c, s = _half_rotation_tables(S, L)
    cos = torch.from_numpy(c).float().to(dt).reshape(1, S, 1, L)
    sin = torch.from_numpy(s).float().to(dt).reshape(1, S, 1, L)
    y = oracle.inplace_partial_rotary_mul(x, cos, sin, st, en, rotary_mode=0)
    xd = x.double().numpy().copy()
    h = L // 2
    z = xd[..., st:st + h] + 1j * xd[..., st + h:en]
    w = np.broadcast_to(cos.double().numpy()[..., :h] + 1j * sin.double().numpy()[..., :h], z.shape)
    r = z * w
    xd[..., st:st + h] = r.real
    xd[..., st + h:en] = r.imag
    assert _ulp_dist(y, oracle.round_to(xd, dt)).max() <= 1


def test_half_mode_equals_interleave_under_permutation():
    """Half mode on the de-interleaved slice (evens, then odds) equals the
    de-interleaved interleave-mode result, with cos/sin permuted the same way."""
    case = W.inplace_case("perm", 78, (2, 5, 3, 32), 0, 32, torch.float32, torch.float32,
                          cs_shape=(2, 5, 3, 32), cs_kind="randn")
    perm = torch.cat([torch.arange(0, 32, 2), torch.arange(1, 32, 2)])
    yi = oracle.inplace_partial_rotary_mul(case.x, case.cos, case.sin, 0, 32, rotary_mode=1)
    yh = oracle.inplace_partial_rotary_mul(case.x[..., perm].contiguous(), case.cos[..., perm].contiguous(),
                                           case.sin[..., perm].contiguous(), 0, 32, rotary_mode=0)
    assert _same_bits(yh, yi[..., perm].contiguous())


def _torch_forward(x, cos, sin, start, end, mode):
    """The forward formula in torch float64 ops, for autograd."""
    L = end - start
    xs = x[..., start:end]
    if mode == 1:
        rot = torch.stack((-xs[..., 1::2], xs[..., 0::2]), dim=-1).reshape(xs.shape)
    else:
        rot = torch.cat((-xs[..., L // 2:], xs[..., :L // 2]), dim=-1)
    y = x.clone()
    y[..., start:end] = xs * cos + rot * sin
    return y


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_backward_is_the_gradient_of_the_forward(mode, dt):
    case = W.inplace_case("grad", 79, (2, 4, 3, 48), 8, 40, dt, torch.float32, cs_shape=(2, 4, 1, 32),
                          cs_kind="randn")
    gy = W.normal(80, case.x.shape, dt)
    x = case.x.double().requires_grad_(True)
    y = _torch_forward(x, case.cos.double(), case.sin.double(), 8, 40, mode)
    (y * gy.double()).sum().backward()
    ref = oracle.round_to(x.grad.numpy(), dt)
    got = oracle.inplace_partial_rotary_mul(gy, case.cos, case.sin, 8, 40, rotary_mode=mode, backward=True)
    assert _ulp_dist(got, ref).max() <= 1


@pytest.mark.parametrize("mode", [0, 1])
def test_backward_adjoint_identity(mode):
    """<F x, g> == <x, F^T g> for random x, g and free cos/sin (float64 sums of
    float32 results; the tolerance covers the two output roundings)."""
    case = W.inplace_case("adj", 81, (3, 5, 2, 64), 0, 64, torch.float32, torch.float32, cs_shape=(3, 5, 2, 64),
                          cs_kind="randn")
    g = W.normal(82, case.x.shape, torch.float32)
    fx = oracle.inplace_partial_rotary_mul(case.x, case.cos, case.sin, 0, 64, rotary_mode=mode).double()
    ftg = oracle.inplace_partial_rotary_mul(g, case.cos, case.sin, 0, 64, rotary_mode=mode, backward=True).double()
    lhs = float((fx * g.double()).sum())
    rhs = float((case.x.double() * ftg).sum())
    scale = float((fx.abs() * g.double().abs()).sum())
    assert abs(lhs - rhs) <= 4 * 2.0 ** -24 * scale


@pytest.mark.parametrize("mode", [0, 1])
def test_backward_of_rotation_is_the_inverse_rotation(mode):
    L = 32
    if mode == 1:
        case = W.inplace_f32_small("slice")
        cos, sin = case.cos, case.sin
    else:
        c, s = _half_rotation_tables(16, L)
        cos = torch.from_numpy(c).float().reshape(1, 16, 1, L)
        sin = torch.from_numpy(s).float().reshape(1, 16, 1, L)
    g = W.normal(83, (1, 16, 2, 64), torch.float32)
    a = oracle.inplace_partial_rotary_mul(g, cos, sin, 16, 48, rotary_mode=mode, backward=True)
    b = oracle.inplace_partial_rotary_mul(g, cos, -sin, 16, 48, rotary_mode=mode)
    assert _same_bits(a, b)


def test_backward_noop_and_untouched_columns():
    case = W.inplace_case("bwd_noop", 84, (2, 3, 2, 32), 8, 24, torch.float16, torch.float32)
    assert _same_bits(oracle.inplace_partial_rotary_mul(case.x, case.cos, case.sin, 8, 8, backward=True), case.x)
    dx = oracle.inplace_partial_rotary_mul(case.x, case.cos, case.sin, 8, 24, backward=True)
    assert _same_bits(dx[..., :8], case.x[..., :8]) and _same_bits(dx[..., 24:], case.x[..., 24:])


# ----------------------------------------------------------------------------
# cache-indexed operator: V2 interleaved splice (cacheMode 1)
# ----------------------------------------------------------------------------

def test_interleaved_cache_mode_hand_cases():
    g = _load("mrope_interleaved_cache_mode_hand_case.json")
    R = g["rotary_dim"]
    half = R // 2
    cache = torch.zeros(5, R)
    for r in range(5):
        cache[r, :half] = torch.arange(half) + 100 * r
    q = torch.ones(1, R)
    pos = torch.tensor(g["positions"], dtype=torch.int64)
    for key, spec in g["cases"].items():
        sec = [int(v) for v in key.split(",")]
        qo, ko, _ = oracle.rope_with_sin_cos_cache(pos, q, q.clone(), cache, R, True, sec, cache_mode=1)
        # positions rows hold 1, 2, 3: row k of the splice reads cache row k + 1
        want = [100 * (r + 1) + i for i, r in enumerate(spec["rows"])] * 2
        assert qo.reshape(-1).tolist() == want and ko.reshape(-1).tolist() == want, key


def test_interleaved_cache_mode_equal_rows_is_rope():
    c = W.cache_case("t", 27, 31, 2, 2, 128, 128, 600, torch.bfloat16, False)
    pos3 = c.positions[None, :].expand(3, -1).contiguous()
    a = oracle.rope_with_sin_cos_cache(c.positions, c.query, c.key, c.cache, 128, False)
    b = oracle.rope_with_sin_cos_cache(pos3, c.query, c.key, c.cache, 128, False, [24, 20, 20], cache_mode=1)
    assert _same_bits(a[0], b[0]) and _same_bits(a[1], b[1])


@pytest.mark.parametrize("section", [[24, 20, 20], [16, 24, 24], [11, 11, 10]])
def test_interleaved_cache_mode_matches_complex_form(section):
    R = 2 * sum(section)
    c = W.cache_case("t", 28, 23, 2, 1, R, R, 400, torch.float32, True, mrope_section=section)
    qo, ko, sk = oracle.rope_with_sin_cos_cache(c.positions, c.query, c.key, c.cache, R, True, section,
                                                cache_mode=1)
    half = R // 2
    owner = np.zeros(half, dtype=np.int64)  # row of each cos index, written out from the rule
    for i in range(half):
        if i < 3 * section[1] and i % 3 == 1:
            owner[i] = 1
        elif i < 3 * section[1] and i % 3 == 2:
            owner[i] = 2
    tab = c.cache.double().numpy()
    rows = c.positions.numpy()[owner, :].T
    idx = np.arange(half)[None, :]
    cos, sin = tab[rows, idx], tab[rows, half + idx]
    for got, x in ((qo, c.query), (ko, c.key)):
        h = x.double().numpy().reshape(23, -1, R)
        z = (h[..., :half] + 1j * h[..., half:]) * (cos + 1j * sin)[:, None, :]
        ref = np.concatenate([z.real, z.imag], axis=-1).reshape(23, -1)
        assert _ulp_dist(got, oracle.round_to(ref, torch.float32)).max() <= 1


# ----------------------------------------------------------------------------
# fused QKV split + RMSNorm + RoPE + paged cache write
# ----------------------------------------------------------------------------

def test_qkv_hand_case():
    g = _load("qkv_rmsnorm_rope_cache_hand_case.json")
    f = torch.float32
    cache = torch.zeros(g["cache_rows"], 2)
    for p in range(g["cache_rows"]):
        cache[p, 0], cache[p, 1] = p / 8, 0.25
    q_out = torch.full((3, 2), 99.0)
    k_cache = torch.full((g["num_blocks"], 1, g["block_size"], 2), 99.0)
    v_cache = torch.full_like(k_cache, 99.0)
    qo, kc, vc, bp, bs = oracle.qkv_rmsnorm_rope_cache(
        torch.tensor(g["qkv"], dtype=f), 1, 1, 1, torch.tensor(g["q_gamma"], dtype=f),
        torch.tensor(g["k_gamma"], dtype=f), 0.0, cache, torch.tensor(g["seq_lens"]),
        torch.tensor(g["query_start_loc"]), torch.tensor(g["slot_mapping"]), q_out, k_cache, v_cache)
    assert bp == 0 and bs == 0
    assert qo.tolist() == g["q_out"]
    want_k = torch.full_like(k_cache, 99.0)
    want_v = torch.full_like(v_cache, 99.0)
    for w in g["k_cache_writes"]:
        want_k[w["block"], 0, w["offset"]] = torch.tensor(w["value"])
    for w in g["v_cache_writes"]:
        want_v[w["block"], 0, w["offset"]] = torch.tensor(w["value"])
    assert torch.equal(kc, want_k) and torch.equal(vc, want_v)


def _qkv_reference(case):
    """Independent float64 composition: torch's rms_norm (a library routine),
    the textbook complex-number rotation, a scatter by slot; positions from
    the page's formula.  Returns (q_out, k_cache, v_cache) before rounding."""
    T, D = case.tokens, case.head_size
    x = case.qkv.double().reshape(T, -1, D)
    nq, nk = case.nq, case.nk
    q = torch.nn.functional.rms_norm(x[:, :nq], (D,), case.q_gamma.double(), case.eps)
    k = torch.nn.functional.rms_norm(x[:, nq:nq + nk], (D,), case.k_gamma.double(), case.eps)
    v = x[:, nq + nk:]
    pos = torch.cat([torch.arange(case.query_start_loc[b + 1] - case.query_start_loc[b]) + case.seq_lens[b]
                     - (case.query_start_loc[b + 1] - case.query_start_loc[b]) for b in range(len(case.seq_lens))])
    tab = case.cache.double()[pos]
    w = (tab[:, :D // 2] + 1j * tab[:, D // 2:])[:, None, :]

    def rot(y):
        z = (y[..., :D // 2] + 1j * y[..., D // 2:]).numpy() * w.numpy()
        return np.concatenate([z.real, z.imag], axis=-1)

    qo = rot(q).reshape(T, -1)
    kc = case.k_cache.double().numpy().copy()
    vc = case.v_cache.double().numpy().copy()
    kr, vr = rot(k), v.numpy()
    bs = case.k_cache.shape[2]
    for t in range(T):
        s = int(case.slot_mapping[t])
        if s < 0:
            continue
        kc[s // bs, :, s % bs] = kr[t]
        vc[s // bs, :, s % bs] = vr[t]
    return qo, kc, vc


@pytest.mark.parametrize("dt", DTYPES)
def test_qkv_matches_independent_composition(dt):
    case = W.qkv_case("t", 31, [5, 1, 3, 1], [2, 9, 0, 20], 3, 2, 2, 32, 4, dt, pad_every=4)
    qo, kc, vc, bp, bs = oracle.qkv_rmsnorm_rope_cache(
        case.qkv, case.nq, case.nk, case.nv, case.q_gamma, case.k_gamma, case.eps, case.cache, case.seq_lens,
        case.query_start_loc, case.slot_mapping, case.q_out, case.k_cache, case.v_cache)
    assert bp == 0 and bs == 0
    rq, rk, rv = _qkv_reference(case)
    # one rounding on each side of a float64 computation: within one ulp
    assert _ulp_dist(qo, oracle.round_to(rq, dt)).max() <= 1
    assert _ulp_dist(kc, oracle.round_to(rk, dt)).max() <= 1
    assert _same_bits(vc, oracle.round_to(rv, dt))


def test_qkv_identity_rotation_gives_unit_rms_heads():
    case = W.qkv_case("t", 32, [6], [0], 2, 1, 1, 64, 8, torch.float32)
    case.cache = torch.cat([torch.ones(case.cache.shape[0], 32), torch.zeros(case.cache.shape[0], 32)], dim=1)
    case.q_gamma = torch.ones(64)
    qo, _, _, _, _ = oracle.qkv_rmsnorm_rope_cache(
        case.qkv, 2, 1, 1, case.q_gamma, case.k_gamma, 0.0, case.cache, case.seq_lens, case.query_start_loc,
        case.slot_mapping, case.q_out, case.k_cache, case.v_cache)
    ms = qo.double().reshape(6, 2, 64).pow(2).mean(-1)
    assert torch.allclose(ms, torch.ones_like(ms), rtol=0, atol=1e-6)


def test_qkv_bad_position_and_slot_are_skipped():
    case = W.qkv_case("t", 33, [2, 2], [3, 3], 1, 1, 1, 32, 4, torch.bfloat16)
    case.cache = case.cache[:5].contiguous()  # positions 3, 4 valid; batch 1 also 3, 4
    case.seq_lens = torch.tensor([5, 6])      # batch 1 positions 4, 5: 5 is out of range
    case.slot_mapping = case.slot_mapping.clone()
    case.slot_mapping[0] = case.k_cache.shape[0] * case.k_cache.shape[2]  # past the pool
    qo, kc, vc, bp, bs = oracle.qkv_rmsnorm_rope_cache(
        case.qkv, 1, 1, 1, case.q_gamma, case.k_gamma, case.eps, case.cache, case.seq_lens, case.query_start_loc,
        case.slot_mapping, case.q_out, case.k_cache, case.v_cache)
    assert bp == 1 and bs == 1
    assert _same_bits(qo[3], case.q_out[3])  # bad position: q row unwritten
    assert not _same_bits(qo[0], case.q_out[0])  # bad slot: q still computed


def test_qkv_oracle_rejects_malformed_query_start_loc():
    """Batch b's tokens are [qsl[b], qsl[b+1]) ([QKV] §计算公式): a decreasing
    queryStartLoc, or one outside [0, T], is refused rather than read past."""
    c = W.qkv_case("bad_qsl", 3, [3, 2], [0, 4], 2, 1, 1, 64, 4, torch.float16)
    for bad in ([0, 4, 2], [0, 2, 6], [-1, 2, 5]):
        with pytest.raises(ValueError):
            oracle.qkv_rmsnorm_rope_cache(c.qkv, 2, 1, 1, c.q_gamma, c.k_gamma, c.eps, c.cache, c.seq_lens,
                                          torch.tensor(bad), c.slot_mapping, c.q_out, c.k_cache, c.v_cache)


def test_every_golden_fixture_cites_its_source():
    """Stored expected values come from the pages: each fixture names the page and
    section it was worked from, and how."""
    folder = os.path.join(os.path.dirname(__file__), "golden")
    names = sorted(f for f in os.listdir(folder) if f.endswith(".json"))
    assert names
    for name in names:
        with open(os.path.join(folder, name)) as f:
            g = json.load(f)
        assert isinstance(g.get("source"), str) and len(g["source"]) > 20, name
