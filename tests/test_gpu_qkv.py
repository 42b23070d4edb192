"""Parity of the fused QKV split + RMSNorm + RoPE + paged cache write.

Tolerance, element by element: each q/k output is o = y_lo*cos - y_hi*sin (or
y_hi*cos + y_lo*sin) of the RMS-normalised values y = x / rms * gamma, which
the kernel forms in binary32, so its error is bounded relative to the terms
|y_lo*cos| + |y_hi*sin| (resp. |y_hi*cos| + |y_lo*sin|), not to o itself:
    float32:          |got - ref| <= 2e-6 * terms
    float16/bfloat16: |got - ref| <= 1 ulp(ref) + 2e-6 * terms
with the terms computed here in float64 from the exact inputs (for the bound
only).  V is copied and must be bit-exact, as must every cache entry the call
does not own and every q_out row it does not write.  The largest error seen per
dtype (|got - ref| / terms, and ulps) is printed at the end of the module."""
import collections

import numpy as np
import pytest
import torch

import oracle
import transformer_rope_positional_gb300 as R
import workloads as W
from guard import Guards
from parity import FP32_REL_TOL, compare_terms, same_bits

pytestmark = pytest.mark.gpu

DTYPES = [torch.float32, torch.float16, torch.bfloat16]
REL = FP32_REL_TOL  # 2e-6 of the terms
_WORST = collections.defaultdict(lambda: {"max_err_over_bound": 0.0, "max_err_over_terms": 0.0, "max_ulp": 0,
                                          "elements": 0})


@pytest.fixture(scope="module", autouse=True)
def _report_worst():
    yield
    for dt, w in sorted(_WORST.items()):
        print("\nfused QKV parity %s: max |got-ref|/bound %.3g, max |got-ref|/terms %.3g, max %d ulp, %d elements"
              % (dt, w["max_err_over_bound"], w["max_err_over_terms"], w["max_ulp"], w["elements"]))


def _run_gpu(case):
    """The op on guarded device copies of the case's tensors (guard bands
    checked after the call); returns q_out, k_cache, v_cache."""
    g = Guards()
    d = g.put
    qo, kc, vc = d(case.q_out, "q_out"), d(case.k_cache, "k_cache"), d(case.v_cache, "v_cache")
    R.qkv_rmsnorm_rope_cache(d(case.qkv, "qkv"), case.nq, case.nk, case.nv, d(case.q_gamma, "q_gamma"),
                             d(case.k_gamma, "k_gamma"), case.eps, d(case.cache, "cache"), d(case.seq_lens, "seq_lens"),
                             d(case.query_start_loc, "query_start_loc"), d(case.slot_mapping, "slot_mapping"), qo, kc,
                             vc)
    g.check()
    return qo.cpu(), kc.cpu(), vc.cpu()


def _run_oracle(case):
    return oracle.qkv_rmsnorm_rope_cache(case.qkv, case.nq, case.nk, case.nv, case.q_gamma, case.k_gamma,
                                         case.eps, case.cache, case.seq_lens, case.query_start_loc,
                                         case.slot_mapping, case.q_out, case.k_cache, case.v_cache)


def _positions(case):
    """Position of every token (the page's seqLens / queryStartLoc rule) and
    whether it falls inside the cos/sin table."""
    qsl = case.query_start_loc.numpy()
    B = case.seq_lens.numel()
    t = np.arange(case.tokens)
    b = np.searchsorted(qsl[:B], t, side="right") - 1
    pos = case.seq_lens.numpy()[b] - (qsl[b + 1] - qsl[b]) + (t - qsl[b])
    return pos, (pos >= 0) & (pos < case.cache.shape[0])


def _terms(case, heads, gamma):
    """|y_lo*cos| + |y_hi*sin| | |y_hi*cos| + |y_lo*sin| per output element of
    the given head range, [T, heads, D], in float64."""
    D, half = case.head_size, case.head_size // 2
    x = case.qkv.double().reshape(case.tokens, -1, D)[:, heads]
    y = x / (x.pow(2).mean(-1, keepdim=True) + case.eps).sqrt() * gamma.double()
    pos, ok = _positions(case)
    cs = case.cache.double()[torch.from_numpy(np.where(ok, pos, 0))][:, None, :]
    c, s = cs[..., :half], cs[..., half:]
    lo = (y[..., :half] * c).abs() + (y[..., half:] * s).abs()
    hi = (y[..., half:] * c).abs() + (y[..., :half] * s).abs()
    return torch.cat([lo, hi], -1).numpy()


def _assert_terms(got, ref, terms, owned, what):
    """Owned elements within the term-relative bound, the others bit-exact."""
    owned = np.broadcast_to(owned, ref.shape)
    idx = torch.from_numpy(np.array(owned))
    assert same_bits(got[~idx], ref[~idx]), "%s: entries the call does not own changed" % what
    res = compare_terms(got[idx], ref[idx], np.broadcast_to(terms, ref.shape)[owned], REL)
    w = _WORST[str(ref.dtype).replace("torch.", "")]
    w["max_err_over_bound"] = max(w["max_err_over_bound"], res["max_err_over_bound"])
    w["max_err_over_terms"] = max(w["max_err_over_terms"], res["max_err_over_terms"])
    w["max_ulp"] = max(w["max_ulp"], res["max_ulp"])
    w["elements"] += res["n"]
    assert res["ok"], "%s: %s" % (what, res)


def _check(case, got, ref):
    qg, kg, vg = got
    qr, kr, vr, bp, bs = ref
    nq, nk, D, T = case.nq, case.nk, case.head_size, case.tokens
    _, pos_ok = _positions(case)
    tq = _terms(case, slice(0, nq), case.q_gamma)
    _assert_terms(qg.view(T, nq, D), qr.view(T, nq, D), tq, pos_ok[:, None, None], "q_out")
    # k: cache entries owned by a token (valid position and slot) within the bound
    tk = _terms(case, slice(nq, nq + nk), case.k_gamma)
    terms = np.zeros(kr.shape)
    owned = np.zeros(kr.shape[:3] + (1,), dtype=bool)
    bsz = case.k_cache.shape[2]
    for t in range(T):
        s = int(case.slot_mapping[t])
        if pos_ok[t] and 0 <= s < kr.shape[0] * bsz:
            terms[s // bsz, :, s % bsz] = tk[t]
            owned[s // bsz, :, s % bsz] = True
    _assert_terms(kg, kr, terms, owned, "k_cache")
    assert same_bits(vg, vr)
    return bp, bs


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("D", [64, 96, 128, 256])
def test_head_sizes_and_dtypes(rope_gpu, dt, D):
    case = W.qkv_case("qkv", 131, [37, 1, 1, 64, 3], [0, 100, 5, 30, 2000], 4, 2, 2, D, 16, dt, pad_every=7)
    bp, bs = _check(case, _run_gpu(case), _run_oracle(case))
    assert bp == 0 and bs == 0 and R.get_device_error() == 0


@pytest.mark.parametrize("heads", [(8, 1, 1), (1, 1, 0), (0, 2, 2), (5, 3, 1)])
def test_head_counts(rope_gpu, heads):
    nq, nk, nv = heads
    case = W.qkv_case("heads", 132, [17, 1, 9], [4, 50, 0], nq, nk, nv, 128, 8, torch.bfloat16)
    _check(case, _run_gpu(case), _run_oracle(case))


def test_mixed_prefill_decode_workload(rope_gpu):
    case = W.qkv_rmsnorm_rope_bf16()
    bp, bs = _check(case, _run_gpu(case), _run_oracle(case))
    assert bp == 0 and bs == 0 and R.get_device_error() == 0


def test_bad_position_and_slot(rope_gpu):
    case = W.qkv_case("bad", 133, [3, 2], [2, 4], 2, 1, 1, 64, 4, torch.float16)
    case.cache = case.cache[:6].contiguous()        # batch 1 positions 4, 5 valid; 3 valid
    case.seq_lens = torch.tensor([5, 7])            # batch 1 positions 5, 6: 6 is out of range
    case.slot_mapping = case.slot_mapping.clone()
    case.slot_mapping[1] = case.k_cache.shape[0] * case.k_cache.shape[2] + 3
    got = _run_gpu(case)
    assert R.get_device_error() == (R.ROPE_DEVICE_POSITION_OUT_OF_RANGE | R.ROPE_DEVICE_SLOT_OUT_OF_RANGE)
    ref = _run_oracle(case)
    bp, bs = _check(case, got, ref)
    assert bp == 1 and bs == 1
    assert same_bits(got[0][4], case.q_out[4])      # token with the bad position: q row unwritten


def test_padding_slots_write_nothing(rope_gpu):
    case = W.qkv_case("pad", 134, [8], [8], 2, 1, 1, 128, 4, torch.bfloat16, pad_every=1)
    qg, kg, vg = _run_gpu(case)
    assert same_bits(kg, case.k_cache) and same_bits(vg, case.v_cache)
    _check(case, (qg, kg, vg), _run_oracle(case))


def test_empty_sequences(rope_gpu):
    """Sequences with no new tokens (queryStartLoc repeats a value) sit between
    non-empty ones; the batch search must skip them."""
    case = W.qkv_case("empty", 135, [5, 0, 0, 3, 0, 7, 0], [0, 4, 0, 10, 2, 30, 9], 4, 2, 2, 128, 8,
                      torch.bfloat16)
    bp, bs = _check(case, _run_gpu(case), _run_oracle(case))
    assert bp == 0 and bs == 0 and R.get_device_error() == 0


@pytest.mark.parametrize("num_seqs", [2047, 2048, 2500])
def test_many_sequences(rope_gpu, num_seqs):
    """Up to 2047 sequences the batch tables sit in shared memory; from 2048 on
    the kernel searches queryStartLoc and seqLens in global memory."""
    rng = np.random.default_rng(num_seqs)
    query_lens = [1] * num_seqs
    for b in rng.choice(num_seqs, 8, replace=False):
        query_lens[int(b)] = int(rng.integers(2, 40))
    query_lens[int(rng.integers(num_seqs))] = 0
    context_lens = [int(v) for v in rng.integers(0, 300, num_seqs)]
    case = W.qkv_case("many", 136, query_lens, context_lens, 4, 2, 1, 64, 16, torch.float16, pad_every=11)
    bp, bs = _check(case, _run_gpu(case), _run_oracle(case))
    assert bp == 0 and bs == 0 and R.get_device_error() == 0


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("block_size", [3, 5, 12, 24])
def test_block_sizes_that_are_not_powers_of_two(rope_gpu, dt, block_size):
    """A slot splits into (block, offset) by a shift when the block size is a
    power of two and by a division otherwise: the division path."""
    case = W.qkv_case("bs%d" % block_size, 137, [29, 1, 6, 1], [3, 77, 40, 0], 4, 2, 2, 128, block_size, dt,
                      pad_every=5)
    bp, bs = _check(case, _run_gpu(case), _run_oracle(case))
    assert bp == 0 and bs == 0 and R.get_device_error() == 0


def test_repeated_calls_are_bit_identical(rope_gpu):
    """The norm's reduction has a fixed order: two runs of the same call give the same bits."""
    case = W.qkv_case("det", 141, [300, 1, 1, 57], [10, 90, 4, 0], 8, 2, 2, 128, 16, torch.bfloat16)
    runs = [_run_gpu(case) for _ in range(2)]
    for a, b in zip(runs[0], runs[1]):
        assert same_bits(a, b)
