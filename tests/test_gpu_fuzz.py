"""Seeded random parity sweep: shapes, dtypes, slices, cos/sin layouts, modes
and directions of the in-place operator; head sizes, rotary dims, styles,
mrope sections and splices of the cache operator, with V2 row views and
separate outputs; head counts, head sizes,
batch compositions, block sizes and padding of the fused QKV operator; each
case checked against the oracle with the tolerances of the parity tests.  The
cases are drawn from a fixed seed per case, so a failure names a reproducible
case."""
import numpy as np
import pytest
import torch

import oracle
import transformer_rope_positional_gb300 as R
import workloads as W
from parity import assert_matches

pytestmark = pytest.mark.gpu

COMBOS = [(torch.float32, torch.float32), (torch.float16, torch.float16), (torch.bfloat16, torch.bfloat16),
          (torch.float16, torch.float32), (torch.bfloat16, torch.float32)]
LAYOUTS = ["1S1L", "BS1L", "B11L", "111L", "BSNL", "B1NL", "1SNL"]


def _cs_shape(layout, B, S, N, L):
    return tuple(dict(B=B, S=S, N=N, L=L)[ch] if ch != "1" else 1 for ch in layout)


@pytest.mark.parametrize("i", range(100))
def test_inplace_random_case(rope_gpu, i):
    rng = np.random.default_rng(7000 + i)
    xdt, cdt = COMBOS[rng.integers(len(COMBOS))]
    B, S, N = int(rng.integers(1, 4)), int(rng.integers(1, 60)), int(rng.integers(1, 7))
    D = 2 * int(rng.integers(1, 129))  # even, up to 256
    if rng.random() < 0.1:
        start, end = 0, 0
        L = D
    else:
        start = int(rng.integers(0, D - 1))
        L = 2 * int(rng.integers(1, (D - start) // 2 + 1))
        end = start + L
    layout = LAYOUTS[rng.integers(len(LAYOUTS))]
    mode = int(rng.integers(0, 2))
    backward = bool(rng.integers(0, 2))
    kind = "randn" if "N" in layout else "rotary"
    case = W.inplace_case("fuzz%d" % i, 7000 + i, (B, S, N, D), start, end, xdt, cdt,
                          cs_shape=_cs_shape(layout, B, S, N, L), cs_kind=kind)
    x = case.x.cuda()
    fn = R.rope_inplace_partial_backward if backward else R.rope_inplace_partial
    fn(x, case.cos.cuda(), case.sin.cuda(), mode, [start, end])
    torch.cuda.synchronize()
    ref = oracle.inplace_partial_rotary_mul(case.x, case.cos, case.sin, start, end, rotary_mode=mode,
                                            backward=backward)
    assert_matches(x.cpu(), ref, "case %d: %s %s x%s slice [%d,%d) layout %s mode %d %s" % (
        i, xdt, cdt, (B, S, N, D), start, end, layout, mode, "bwd" if backward else "fwd"))


@pytest.mark.parametrize("i", range(100))
def test_cache_random_case(rope_gpu, i):
    rng = np.random.default_rng(8000 + i)
    dt = [torch.float32, torch.float16, torch.bfloat16][rng.integers(3)]
    mult = 16 if dt == torch.float32 else 32
    hs = mult * int(rng.integers(1, 256 // mult + 1))
    r = mult * int(rng.integers(1, hs // mult + 1))
    T, hq, hk = int(rng.integers(1, 300)), int(rng.integers(1, 7)), int(rng.integers(1, 5))
    neox = bool(rng.integers(0, 2))
    section, cache_mode = None, 0
    if rng.random() < 0.5:  # mrope: 3 or 4 sections summing to R/2, the first non-zero
        m = int(rng.integers(3, 5))
        cuts = np.sort(rng.integers(0, r // 2 + 1, m - 1))
        section = np.diff(np.concatenate([[0], cuts, [r // 2]])).astype(int).tolist()
        if section[0] == 0:
            section[0], section[-1] = section[-1], 0
        if section[0] == 0:
            section = None
        elif m == 3 and rng.random() < 0.5:
            cache_mode = 1  # V2 interleaved splice (three sections)
    case = W.cache_case("fuzz%d" % i, 8000 + i, T, hq, hk, hs, r, int(rng.integers(1, 3000)), dt, neox,
                        mrope_section=section)
    q, k = case.query.cuda(), case.key.cuda()
    R.rope_with_sin_cos_cache(case.positions.cuda(), q, k, case.cache.cuda(), hs, r, neox, section,
                              cache_mode=cache_mode)
    torch.cuda.synchronize()
    qo, ko, skipped = oracle.rope_with_sin_cos_cache(case.positions, case.query, case.key, case.cache, hs, neox,
                                                     section, cache_mode=cache_mode)
    assert skipped == 0
    what = "case %d: %s T=%d hq=%d hk=%d hs=%d R=%d %s section %s mode %d" % (
        i, dt, T, hq, hk, hs, r, "neox" if neox else "gptj", section, cache_mode)
    assert_matches(q.cpu(), qo, what + " query")
    assert_matches(k.cpu(), ko, what + " key")
    assert R.get_device_error() == 0


@pytest.mark.parametrize("i", range(50))
def test_fused_qkv_random_case(rope_gpu, i):
    from test_gpu_qkv import _check, _run_gpu, _run_oracle
    rng = np.random.default_rng(9000 + i)
    dt = [torch.float32, torch.float16, torch.bfloat16][rng.integers(3)]
    mult, top = (16, 256) if dt == torch.float32 else (32, 512)
    D = mult * int(rng.integers(1, top // mult + 1))
    nq, nk, nv = int(rng.integers(0, 9)), int(rng.integers(0, 5)), int(rng.integers(0, 5))
    if nq + nk + nv == 0:
        nq = 1
    B = int(rng.integers(1, 12))
    qlens = [int(v) for v in rng.integers(0, 40, B)]
    if sum(qlens) == 0:
        qlens[0] = 1
    ctx = [int(v) for v in rng.integers(0, 300, B)]
    bs = int(rng.choice([1, 4, 16, 32]))
    pad = int(rng.choice([0, 0, 3, 7]))
    case = W.qkv_case("fuzz_qkv%d" % i, 9000 + i, qlens, ctx, nq, nk, nv, D, bs, dt, pad_every=pad)
    bp, bslot = _check(case, _run_gpu(case), _run_oracle(case))
    assert bp == 0 and bslot == 0 and R.get_device_error() == 0


@pytest.mark.parametrize("i", range(50))
def test_cache_v2_random_case(rope_gpu, i):
    """V2: query and key as row views of a wider buffer (extra columns between
    and after them), optionally written to separate whole-row outputs."""
    rng = np.random.default_rng(9500 + i)
    dt = [torch.float32, torch.float16, torch.bfloat16][rng.integers(3)]
    mult = 16 if dt == torch.float32 else 32
    hs = mult * int(rng.integers(1, 256 // mult + 1))
    r = mult * int(rng.integers(1, hs // mult + 1))
    T, hq, hk = int(rng.integers(1, 200)), int(rng.integers(1, 6)), int(rng.integers(1, 4))
    neox = bool(rng.integers(0, 2))
    section = None
    if rng.random() < 0.4 and r >= 8:
        a = int(rng.integers(1, r // 2 - 1)) if r // 2 > 2 else 1
        b = int(rng.integers(0, r // 2 - a + 1))
        section = [a, b, r // 2 - a - b]
    case = W.cache_case("fuzz_v2_%d" % i, 9500 + i, T, hq, hk, hs, r, int(rng.integers(1, 2000)), dt, neox,
                        mrope_section=section)
    wq, wk = hq * hs, hk * hs
    gap = hs * int(rng.integers(0, 3))  # extra heads between q and k and after k
    buf = torch.zeros(T, wq + gap + wk + gap, dtype=dt, device="cuda")
    buf[:, :wq].copy_(case.query.cuda())
    buf[:, wq + gap:wq + gap + wk].copy_(case.key.cuda())
    q, k = buf[:, :wq], buf[:, wq + gap:wq + gap + wk]
    out = bool(rng.integers(0, 2))
    qo = torch.full((T, wq), 9.0, dtype=dt, device="cuda") if out else None
    ko = torch.full((T, wk), 9.0, dtype=dt, device="cuda") if out else None
    R.rope_with_sin_cos_cache(case.positions.cuda(), q, k, case.cache.cuda(), hs, r, neox, section,
                              query_out=qo, key_out=ko)
    torch.cuda.synchronize()
    ref_q, ref_k, skipped = oracle.rope_with_sin_cos_cache(case.positions, case.query, case.key, case.cache, hs,
                                                           neox, section)
    assert skipped == 0
    what = "case %d: %s T=%d hs=%d R=%d %s section %s gap %d out %s" % (
        i, dt, T, hs, r, "neox" if neox else "gptj", section, gap, out)
    got_q, got_k = (qo, ko) if out else (q, k)
    assert_matches(got_q.cpu(), ref_q, what + " query")
    assert_matches(got_k.cpu(), ref_k, what + " key")
    if out:  # inputs untouched
        assert torch.equal(q.cpu(), case.query) and torch.equal(k.cpu(), case.key)
    assert R.get_device_error() == 0
