"""Parity of the cache-indexed kernel (rope and mrope, NeoX and GPT-J) against
the oracle, with the tolerances of ``parity.py``."""
import json
import os

import pytest
import torch

import transformer_rope_positional_gb300 as R
import workloads as W
from gpu_runs import gpu_cache, oracle_cache
from parity import assert_matches, same_bits

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
DTYPES = [torch.float32, torch.float16, torch.bfloat16]


def _check(case, positions=None):
    qg, kg = gpu_cache(case, positions)
    qo, ko, skipped = oracle_cache(case, positions)
    assert skipped == 0
    assert_matches(qg, qo, case.name + " query")
    assert_matches(kg, ko, case.name + " key")
    assert R.get_device_error() == 0
    return qg, kg


def test_worked_example_from_the_page(rope_gpu):
    with open(os.path.join(GOLDEN, "rope_cache_worked_example_bf16.json")) as f:
        g = json.load(f)
    dt = torch.bfloat16
    q = torch.full(g["query_shape"], g["fill"], dtype=dt, device="cuda")
    k = torch.full(g["key_shape"], g["fill"], dtype=dt, device="cuda")
    cache = torch.full(g["cache_shape"], g["fill"], dtype=dt, device="cuda")
    pos = torch.tensor(g["positions"], dtype=torch.int64, device="cuda")
    R.rope_with_sin_cos_cache(pos, q, k, cache, g["head_size"], is_neox=g["is_neox"])
    torch.cuda.synchronize()
    want = [float(v) for v in g["expected_row"]]
    for t in (q, k):
        for row in t.cpu():
            assert row.float().tolist() == want


def _sizes(dt):
    mult = 16 if dt == torch.float32 else 32
    out = []
    for hs in (32, 64, 96, 128):
        if hs % mult:
            continue
        for r in (16, 32, 48, 64, 96, 128):
            if r % mult == 0 and r <= hs:
                out.append((hs, r))
    return out


SWEEP = [(dt, hs, r) for dt in DTYPES for hs, r in _sizes(dt)]


@pytest.mark.parametrize("dt,hs,r", SWEEP, ids=[f"{str(d)[6:]}_h{h}_r{r}" for d, h, r in SWEEP])
@pytest.mark.parametrize("neox", [True, False], ids=["neox", "gptj"])
@pytest.mark.parametrize("tokens", [1, 3, 257])
def test_head_size_rotary_dim_sweep(rope_gpu, dt, hs, r, neox, tokens):
    case = W.cache_case(f"sweep_{hs}_{r}", 61, tokens, 3, 2, hs, r, 513, dt, neox)
    _check(case)


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("neox", [True, False], ids=["neox", "gptj"])
def test_pass_through_columns_bit_exact(rope_gpu, dt, neox):
    hs, r = (128, 64) if dt != torch.float32 else (64, 16)
    case = W.cache_case("pass", 62, 33, 2, 2, hs, r, 100, dt, neox)
    bits = {4: torch.int32, 2: torch.int16}[case.query.element_size()]
    nan_base = 0x7FC00001 if dt == torch.float32 else 0x7E01
    for t in (case.query, case.key):
        v = t.view(bits).view(t.shape[0], -1, hs)
        v[..., r:] = (torch.arange(hs - r) + nan_base).to(bits)
    qg, kg = _check(case)
    for got, x in ((qg, case.query), (kg, case.key)):
        assert same_bits(got.view(33, -1, hs)[..., r:], x.view(33, -1, hs)[..., r:])


def test_neox_bf16_workload_reduced(rope_gpu):
    _check(W.cache_neox_bf16(1000))


def test_gptj_f16_partial_workload_reduced(rope_gpu):
    _check(W.cache_gptj_f16_partial(num_seqs=2, seq_len=512))


def test_mrope_workload_reduced(rope_gpu):
    full = W.mrope_neox_bf16()
    keep = torch.cat([torch.arange(0, 700), torch.arange(8192, 8192 + 1300)])
    case = W.cache_case("mrope_reduced", 4, len(keep), 28, 4, 128, 128, 40960, torch.bfloat16, True,
                        base=1e6, positions=full.positions[:, keep].contiguous(), mrope_section=[16, 24, 24])
    _check(case)


SECTIONS = [[16, 24, 24], [8, 12, 12], [24, 20, 20], [11, 11, 10], [16, 16, 16, 16], [0, 0, 0]]


@pytest.mark.parametrize("section", SECTIONS, ids=["_".join(map(str, s)) for s in SECTIONS])
@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("neox", [True, False], ids=["neox", "gptj"])
def test_mrope_sections(rope_gpu, section, dt, neox):
    R_ = 2 * sum(section) if section[0] > 0 else 64
    hs = R_ if R_ % (16 if dt == torch.float32 else 32) == 0 else 128
    if R_ % (16 if dt == torch.float32 else 32):
        pytest.skip("rotary dim %d is not a 64-byte multiple for %s" % (R_, dt))
    case = W.cache_case("mrope", 63, 77, 3, 2, hs, R_, 300, dt, neox, mrope_section=section)
    if section[0] == 0:  # first element 0: rope mode, positions 1-D
        case.positions = case.positions[0].contiguous()
    _check(case)


def test_mrope_equal_rows_is_rope_bit_exact(rope_gpu):
    case = W.cache_neox_bf16(300)
    qa, ka = gpu_cache(case)
    pos3 = case.positions[None, :].expand(3, -1).contiguous()
    case.mrope_section = [16, 24, 24]
    qb, kb = gpu_cache(case, pos3)
    assert same_bits(qa, qb) and same_bits(ka, kb)


@pytest.mark.parametrize("neox", [True, False], ids=["neox", "gptj"])
def test_out_of_range_positions_leave_tokens_untouched(rope_gpu, neox):
    case = W.cache_case("oob", 64, 9, 2, 1, 64, 64, 50, torch.bfloat16, neox)
    pos = case.positions.clone()
    pos[2] = 50
    pos[7] = -3
    assert R.get_device_error() == 0
    qg, kg = gpu_cache(case, pos)
    assert R.get_device_error() == R.ROPE_DEVICE_POSITION_OUT_OF_RANGE
    assert R.get_device_error() == 0  # read-and-clear
    qo, ko, skipped = oracle_cache(case, pos)
    assert skipped == 2
    for t in (2, 7):
        assert same_bits(qg[t], case.query[t]) and same_bits(kg[t], case.key[t])
    assert_matches(qg, qo, "oob query")
    assert_matches(kg, ko, "oob key")


def test_out_of_range_mrope_row(rope_gpu):
    case = W.cache_case("oob_mrope", 65, 5, 1, 1, 64, 64, 40, torch.float16, True, mrope_section=[8, 12, 12])
    pos = case.positions.clone()
    pos[2, 3] = 40
    qg, kg = gpu_cache(case, pos)
    assert R.get_device_error() == R.ROPE_DEVICE_POSITION_OUT_OF_RANGE
    qo, ko, skipped = oracle_cache(case, pos)
    assert skipped == 1
    assert same_bits(qg[3], case.query[3])
    assert_matches(qg, qo, "oob mrope")


@pytest.mark.parametrize("dt", DTYPES)
def test_special_values(rope_gpu, dt):
    case = W.cache_case("special", 66, 40, 2, 2, 64, 64, 80, dt, True)
    q = case.query.float()
    q.view(-1)[0::13] = float("inf")
    q.view(-1)[4::19] = float("nan")
    q.view(-1)[6::23] = float("-inf")
    case.query = q.to(dt)
    c = case.cache.float()
    c[5, 3] = float("nan")
    c[7, 40] = float("inf")
    case.cache = c.to(dt)
    _check(case)


def test_many_tokens_one_small_head(rope_gpu):
    # 2^17 + 1 tokens, the largest count of the page's test ranges
    case = W.cache_case("many_tokens", 67, 131073, 1, 1, 32, 32, 4096, torch.float16, True)
    _check(case)


def test_decode_many_heads(rope_gpu):
    for neox in (True, False):
        case = W.cache_case("decode", 68, 1, 64, 8, 128, 64, 2048, torch.bfloat16, neox)
        _check(case)


def test_rejected_arguments_raise(rope_gpu):
    case = W.cache_case("bad", 69, 4, 1, 1, 64, 64, 10, torch.bfloat16, True)
    with pytest.raises(R.RopeError) as e:
        R.rope_with_sin_cos_cache(case.positions.cuda(), case.query.cuda(), case.key.cuda(), case.cache.cuda(),
                                  48)
    assert e.value.status == R.ROPE_ERR_PARAM_INVALID


@pytest.mark.parametrize("neox,section", [(True, None), (False, None), (True, [16, 24, 24])])
def test_repeated_calls_are_bit_identical(rope_gpu, neox, section):
    """Results do not depend on the run: the same call on fresh copies of the
    inputs gives the same bits (no atomics or order-dependent sums on the path)."""
    case = W.cache_case("det", 140, 3000, 8, 2, 128, 128, 5000, torch.bfloat16, neox, mrope_section=section)
    pos, cache = case.positions.cuda(), case.cache.cuda()
    outs = []
    for _ in range(2):
        q, k = case.query.cuda(), case.key.cuda()
        R.rope_with_sin_cos_cache(pos, q, k, cache, 128, 128, neox, section)
        torch.cuda.synchronize()
        outs.append((q.cpu(), k.cpu()))
    assert same_bits(outs[0][0], outs[1][0]) and same_bits(outs[0][1], outs[1][1])
