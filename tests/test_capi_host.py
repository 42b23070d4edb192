"""Host-side checks of the C ABI: the library loads, exports every declared
symbol, and rejects bad arguments before touching the GPU.

Nothing here launches a kernel: every call either fails validation or is a
no-op that returns before any CUDA call, so the file runs on a machine without
a GPU.  Fake device pointers are never dereferenced.
"""
import ctypes
import os
import re

import pytest
import torch

from transformer_rope_positional_gb300 import _capi as C
from transformer_rope_positional_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rope_gb300.h")
FAKE = 0x10000  # a non-NULL, 64 KiB-aligned address that is never dereferenced


@pytest.fixture(scope="module")
def lib():
    B.build()
    return C.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rope_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(names) == set(C.EXPORTED)
    for n in names:
        assert hasattr(lib, n), n


def test_abi_version_and_status_strings(lib):
    assert lib.rope_abi_version() == 4
    for st in (C.ROPE_OK, C.ROPE_ERR_PARAM_NULLPTR, C.ROPE_ERR_PARAM_INVALID, C.ROPE_ERR_CUDA, 12345):
        s = C.status_string(st)
        assert isinstance(s, str) and s
    assert "NULLPTR" in C.status_string(161001) and "INVALID" in C.status_string(161002)


def _d(dtype, shape, ptr=FAKE):
    return C.describe(ptr, dtype, shape)


def _inplace(lib, x, c, s, mode=1, start=0, end=0):
    return lib.rope_inplace_partial(ctypes.byref(x) if x else None, ctypes.byref(c) if c else None,
                                    ctypes.byref(s) if s else None, mode, start, end, None)


X = (2, 3, 4, 64)
CS = (1, 3, 1, 64)


@pytest.mark.parametrize("which", [0, 1, 2])
def test_inplace_null_descriptors(lib, which):
    args = [_d(C.F32, X), _d(C.F32, CS), _d(C.F32, CS)]
    args[which] = None
    assert _inplace(lib, *args) == C.ROPE_ERR_PARAM_NULLPTR


def test_inplace_null_data_pointer(lib):
    # shapes are valid, so the missing data is what is reported
    assert _inplace(lib, _d(C.F32, X, 0), _d(C.F32, CS), _d(C.F32, CS)) == C.ROPE_ERR_PARAM_NULLPTR


@pytest.mark.parametrize("xdt,cdt,sdt,ok", [
    (C.F32, C.F16, C.F16, False),    # f32 x needs f32 cos/sin
    (C.F16, C.BF16, C.BF16, False),  # half x with the other half type
    (C.F16, C.F32, C.F16, False),    # cos and sin differ
    (C.I64, C.I64, C.I64, False),
    (C.BF16, C.F32, C.F32, True),    # mixed precision is allowed
])
def test_inplace_dtype_rules(lib, xdt, cdt, sdt, ok):
    st = _inplace(lib, _d(xdt, X), _d(cdt, CS), _d(sdt, CS), start=8, end=8)
    assert st == (C.ROPE_OK if ok else C.ROPE_ERR_PARAM_INVALID)


@pytest.mark.parametrize("mode", [2, 3, -1, 4])
def test_inplace_modes_without_a_formula_rejected(lib, mode):
    # 0 (half) and 1 (interleave) are accepted; QUARTER (2), DEEPSEEK_INTERLEAVE (3)
    # and anything else have no formula on the page
    assert _inplace(lib, _d(C.F32, X), _d(C.F32, CS), _d(C.F32, CS), mode=mode) == C.ROPE_ERR_PARAM_INVALID


def _backward(lib, x, c, s, mode=1, start=0, end=0):
    return lib.rope_inplace_partial_backward(ctypes.byref(x) if x else None, ctypes.byref(c) if c else None,
                                             ctypes.byref(s) if s else None, mode, start, end, None)


def test_backward_shares_the_forward_checks(lib):
    assert _backward(lib, None, _d(C.F32, CS), _d(C.F32, CS)) == C.ROPE_ERR_PARAM_NULLPTR
    assert _backward(lib, _d(C.F32, X), _d(C.F16, CS), _d(C.F16, CS)) == C.ROPE_ERR_PARAM_INVALID
    assert _backward(lib, _d(C.F32, X), _d(C.F32, CS), _d(C.F32, CS), mode=2) == C.ROPE_ERR_PARAM_INVALID
    assert _backward(lib, _d(C.F32, X), _d(C.F32, (1, 3, 1, 8)), _d(C.F32, (1, 3, 1, 8)), start=0,
                     end=16) == C.ROPE_ERR_PARAM_INVALID
    before = lib.rope_launch_count()
    assert _backward(lib, _d(C.F32, X), _d(C.F32, CS), _d(C.F32, CS), start=8, end=8) == C.ROPE_OK
    assert lib.rope_launch_count() == before


@pytest.mark.parametrize("xs,cs,start,end", [
    ((2, 3, 64), (1, 3, 1, 64), 0, 0),          # x not 4-D
    ((2, 3, 4, 1026), (1, 3, 1, 1026), 0, 0),   # D > 1024
    ((2, 3, 4, 63), (1, 3, 1, 63), 0, 0),       # D odd
    (X, (1, 3, 1, 8), -2, 6),                   # start < 0
    (X, (1, 3, 1, 8), 60, 68),                  # end > D
    (X, (1, 3, 1, 8), 10, 4),                   # start > end
    (X, (1, 3, 1, 7), 3, 10),                   # odd slice length
    (X, (1, 3, 1, 16), 0, 8),                   # cos last dim != slice length
    (X, (3, 3, 1, 64), 0, 0),                   # cos B neither 1 nor B
    (X, (1, 2, 1, 64), 0, 0),                   # cos S neither 1 nor S
    (X, (1, 3, 2, 64), 0, 0),                   # cos N neither 1 nor N
])
def test_inplace_shape_rules(lib, xs, cs, start, end):
    st = _inplace(lib, _d(C.F32, xs), _d(C.F32, cs), _d(C.F32, cs), start=start, end=end)
    assert st == C.ROPE_ERR_PARAM_INVALID


def test_inplace_cos_sin_shapes_must_match(lib):
    st = _inplace(lib, _d(C.F32, X), _d(C.F32, CS), _d(C.F32, (1, 3, 4, 64)))
    assert st == C.ROPE_ERR_PARAM_INVALID


def test_inplace_noop_enqueues_nothing(lib):
    before = lib.rope_launch_count()
    # start == end (not [0,0]) is a no-op, checked before the cos width
    assert _inplace(lib, _d(C.F32, X), _d(C.F32, (1, 3, 1, 5)), _d(C.F32, (1, 3, 1, 5)), start=8,
                    end=8) == C.ROPE_OK
    # an empty x is a no-op too
    assert _inplace(lib, _d(C.F32, (0, 3, 4, 64)), _d(C.F32, (1, 3, 1, 64)), _d(C.F32, (1, 3, 1, 64)),
                    start=0, end=0) == C.ROPE_OK
    assert lib.rope_launch_count() == before


def _cache(lib, pos, q, k, c, head_size=64, R=None, neox=1, section=None):
    R = (c.shape[1] if c is not None else 64) if R is None else R
    sec = None
    n = 0
    if section is not None:
        n = len(section)
        sec = (ctypes.c_int64 * max(1, n))(*section)
    return lib.rope_with_sin_cos_cache(*(ctypes.byref(t) if t is not None else None for t in (pos, q, k, c)),
                                       head_size, R, neox, sec, n, None)


T = 7


def good(dt=C.BF16, R=64, hs=64):
    return (_d(C.I64, (T,)), _d(dt, (T, 4 * hs)), _d(dt, (T, 2 * hs)), _d(dt, (100, R)))


@pytest.mark.parametrize("which", [0, 1, 2, 3])
def test_cache_null_descriptors(lib, which):
    args = list(good())
    args[which] = None
    assert _cache(lib, *args) == C.ROPE_ERR_PARAM_NULLPTR


def test_cache_null_data(lib):
    p, q, k, c = good()
    q = _d(C.BF16, (T, 256), 0)
    assert _cache(lib, p, q, k, c) == C.ROPE_ERR_PARAM_NULLPTR


def _bad(lib, **kw):
    p, q, k, c = good()
    args = dict(pos=p, q=q, k=k, c=c, head_size=64, R=None, neox=1, section=None)
    args.update(kw)
    return _cache(lib, args["pos"], args["q"], args["k"], args["c"], args["head_size"], args["R"],
                  args["neox"], args["section"])


@pytest.mark.parametrize("case", [
    dict(pos=_d(C.F32, (T,))),                                  # positions not int64
    dict(k=_d(C.F16, (T, 128))),                                # key dtype differs
    dict(c=_d(C.F16, (100, 64))),                               # cache dtype differs
    dict(q=_d(C.BF16, (T, 4, 64))),                             # query not 2-D
    dict(q=_d(C.BF16, (0, 256)), k=_d(C.BF16, (0, 128)), pos=_d(C.I64, (0,))),  # no tokens
    dict(k=_d(C.BF16, (T + 1, 128))),                           # token counts differ
    dict(head_size=48),                                         # not a multiple of 32 for bf16
    dict(head_size=96),                                         # does not divide the row widths
    dict(R=32),                                                 # rotary_dim != cache width
    dict(c=_d(C.BF16, (100, 48)), R=48),                        # R not a multiple of 32
    dict(c=_d(C.BF16, (100, 128)), R=128),                      # R > head_size
    dict(pos=_d(C.I64, (T + 1,))),                              # positions length
    dict(section=[16, 16]),                                     # section count not 3 or 4
    dict(section=[16, 8, 4], pos=_d(C.I64, (3, T))),            # 2 * sum != R
    dict(section=[16, -8, 24], pos=_d(C.I64, (3, T))),          # negative element
    dict(section=[8, 12, 12]),                                  # mrope with 1-D positions
    dict(section=[8, 12, 12], pos=_d(C.I64, (4, T))),           # rows != section count
])
def test_cache_rejections(lib, case):
    assert _bad(lib, **case) == C.ROPE_ERR_PARAM_INVALID


def test_cache_fp32_sizes_follow_16_element_rule(lib):
    p, _, _, _ = good()
    q = _d(C.F32, (T, 4 * 48))
    k = _d(C.F32, (T, 2 * 48))
    c = _d(C.F32, (100, 40))
    # 48 is a multiple of 16 (allowed for fp32) but 40 is not
    assert _cache(lib, p, q, k, c, head_size=48) == C.ROPE_ERR_PARAM_INVALID


def test_cache_misaligned_pointers_rejected(lib):
    p, q, k, c = good()
    q = _d(C.BF16, (T, 256), FAKE + 2)
    assert _cache(lib, p, q, k, c) == C.ROPE_ERR_PARAM_INVALID


def test_device_error_needs_an_out_pointer(lib):
    assert lib.rope_get_device_error(None, None) == C.ROPE_ERR_PARAM_NULLPTR


def test_python_binding_refuses_cpu_tensors():
    B.build()
    x = torch.zeros(1, 2, 2, 8)
    c = torch.ones(1, 2, 1, 8)
    with pytest.raises(ValueError):
        C.rope_inplace_partial(x, c, c)


def _v2(lib, pos, q, k, c, head_size=64, R=None, neox=1, section=None, mode=0, qs=0, ks=0, qo=None, ko=None):
    R = (c.shape[1] if c is not None else 64) if R is None else R
    sec, n = None, 0
    if section is not None:
        n = len(section)
        sec = (ctypes.c_int64 * max(1, n))(*section)
    ref = lambda t: ctypes.byref(t) if t is not None else None  # noqa: E731
    return lib.rope_with_sin_cos_cache_v2(ref(pos), ref(q), ref(k), ref(c), head_size, R, neox, sec, n, mode,
                                          qs, ks, ref(qo), ref(ko), None)


@pytest.mark.parametrize("case,status", [
    (dict(mode=2), C.ROPE_ERR_PARAM_INVALID),                                   # unknown cache mode
    (dict(mode=1), C.ROPE_ERR_PARAM_INVALID),                                   # interleaved splice needs mrope
    (dict(mode=1, section=[8, 8, 8, 8], pos=_d(C.I64, (4, T))), C.ROPE_ERR_PARAM_INVALID),  # and 3 sections
    (dict(qs=200), C.ROPE_ERR_PARAM_INVALID),                                   # stride below the row width
    (dict(qs=260), C.ROPE_ERR_PARAM_INVALID),                                   # stride not a 16-byte multiple
    (dict(qo=_d(C.BF16, (T, 256), FAKE * 8)), C.ROPE_ERR_PARAM_NULLPTR),        # key_out missing
    (dict(qo=_d(C.BF16, (T, 128), FAKE * 8), ko=_d(C.BF16, (T, 128), FAKE * 9)), C.ROPE_ERR_PARAM_INVALID),
    (dict(qo=_d(C.F16, (T, 256), FAKE * 8), ko=_d(C.BF16, (T, 128), FAKE * 9)), C.ROPE_ERR_PARAM_INVALID),
    (dict(qo=_d(C.BF16, (T, 256), FAKE + 64), ko=_d(C.BF16, (T, 128), FAKE * 9)), C.ROPE_ERR_PARAM_INVALID),
])
def test_cache_v2_rejections(lib, case, status):
    p, q, k, c = good()
    args = dict(pos=p, q=q, k=k, c=c)
    args.update(case)
    pos, q, k, c = args.pop("pos"), args.pop("q"), args.pop("k"), args.pop("c")
    assert _v2(lib, pos, q, k, c, **args) == status


def _qkv(lib, **over):
    T, nq, nk, nv, D, NB, BS, B = 6, 2, 1, 1, 64, 3, 4, 2
    t = dict(qkv=_d(C.BF16, (T, (nq + nk + nv) * D)), qg=_d(C.BF16, (D,)), kg=_d(C.BF16, (D,)),
             cache=_d(C.BF16, (50, D)), sl=_d(C.I64, (B,)), qsl=_d(C.I64, (B + 1,)), slots=_d(C.I64, (T,)),
             qo=_d(C.BF16, (T, nq * D)), kc=_d(C.BF16, (NB, nk, BS, D)), vc=_d(C.BF16, (NB, nv, BS, D)),
             nq=nq, nk=nk, nv=nv, eps=1e-6)
    t.update(over)
    ref = lambda x: ctypes.byref(x) if x is not None else None  # noqa: E731
    return lib.rope_qkv_rmsnorm_rope_cache(ref(t["qkv"]), t["nq"], t["nk"], t["nv"], ref(t["qg"]), ref(t["kg"]),
                                           t["eps"], ref(t["cache"]), ref(t["sl"]), ref(t["qsl"]), ref(t["slots"]),
                                           ref(t["qo"]), ref(t["kc"]), ref(t["vc"]), None)


@pytest.mark.parametrize("over,status", [
    (dict(qkv=None), C.ROPE_ERR_PARAM_NULLPTR),
    (dict(vc=None), C.ROPE_ERR_PARAM_NULLPTR),
    (dict(qg=_d(C.F16, (64,))), C.ROPE_ERR_PARAM_INVALID),          # gamma dtype
    (dict(sl=_d(C.F32, (2,))), C.ROPE_ERR_PARAM_INVALID),           # seq_lens not int64
    (dict(nq=3), C.ROPE_ERR_PARAM_INVALID),                         # heads do not divide the width
    (dict(qkv=_d(C.BF16, (6, 4 * 48)), qg=_d(C.BF16, (48,)), kg=_d(C.BF16, (48,))), C.ROPE_ERR_PARAM_INVALID),
    (dict(qkv=_d(C.BF16, (6, 4 * 1024)), qg=_d(C.BF16, (1024,)), kg=_d(C.BF16, (1024,))), C.ROPE_ERR_PARAM_INVALID),
    (dict(cache=_d(C.BF16, (50, 32))), C.ROPE_ERR_PARAM_INVALID),   # cache width != D
    (dict(qsl=_d(C.I64, (2,))), C.ROPE_ERR_PARAM_INVALID),          # query_start_loc length != B + 1
    (dict(slots=_d(C.I64, (5,))), C.ROPE_ERR_PARAM_INVALID),        # one slot per token
    (dict(sl=_d(C.I64, ((1 << 30) + 1,)), qsl=_d(C.I64, ((1 << 30) + 2,))), C.ROPE_ERR_PARAM_INVALID),  # > 2^30 seqs
    (dict(kc=_d(C.BF16, (1, 1, (1 << 30) + 1, 64)), vc=_d(C.BF16, (1, 1, (1 << 30) + 1, 64))),
     C.ROPE_ERR_PARAM_INVALID),  # block size past 2^30
    (dict(qo=_d(C.BF16, (6, 64))), C.ROPE_ERR_PARAM_INVALID),       # q_out width
    (dict(vc=_d(C.BF16, (3, 1, 8, 64))), C.ROPE_ERR_PARAM_INVALID),  # block sizes differ
    (dict(eps=-1.0), C.ROPE_ERR_PARAM_INVALID),
    (dict(eps=float("nan")), C.ROPE_ERR_PARAM_INVALID),
    (dict(qkv=_d(C.BF16, (6, 256), FAKE + 8)), C.ROPE_ERR_PARAM_INVALID),  # misaligned
])
def test_qkv_rejections(lib, over, status):
    assert _qkv(lib, **over) == status


def test_overlapping_row_views_are_refused_before_the_library():
    """A row view whose stride is below its width (one row expanded to many:
    stride 0) would make the operator read and write every row through the
    same memory; the binding refuses it before building a descriptor."""
    one = torch.randn(1, 256)
    with pytest.raises(ValueError, match="rows overlap"):
        C.rows_desc(one.expand(16, 256))
    with pytest.raises(ValueError, match="rows overlap"):
        C.rows_desc(torch.randn(16, 300).as_strided((16, 256), (128, 1)))
    # a single row is fine whatever its stride; it reports its width
    with pytest.raises(ValueError, match="CUDA"):
        C.rows_desc(one.expand(1, 256))
    with pytest.raises(ValueError, match="overlap"):
        C.rope_with_sin_cos_cache(torch.zeros(16, dtype=torch.int64), one.expand(16, 256), torch.randn(16, 256),
                                  torch.randn(8, 128), 128)


class _OnDevice:
    def __init__(self, index):
        self.index = index

    def get_device(self):
        return self.index


def test_tensors_on_several_devices_are_refused():
    assert C._one_device(_OnDevice(1), None, _OnDevice(1)) == 1
    with pytest.raises(ValueError, match="different devices"):
        C._one_device(_OnDevice(0), _OnDevice(1))
    with pytest.raises(ValueError, match="different devices"):
        C._one_device(torch.empty(1), _OnDevice(0))


def test_shapes_whose_element_count_overflows_are_refused(lib):
    """Element counts are taken with overflow checks: a shape whose product
    wraps int64 (or passes INT64_MAX / 8) is refused, not launched with a
    wrapped count."""
    big = 1 << 40
    assert _inplace(lib, _d(C.F32, (big, big, 2, 64)), _d(C.F32, (1, 1, 1, 64)), _d(C.F32, (1, 1, 1, 64))) \
        == C.ROPE_ERR_PARAM_INVALID
    assert _inplace(lib, _d(C.F32, (1 << 30, 1 << 30, 2, 64)), _d(C.F32, (1, 1, 1, 64)),
                    _d(C.F32, (1, 1, 1, 64))) == C.ROPE_ERR_PARAM_INVALID  # 2^67 elements
    p, q, k, c = good()
    assert _cache(lib, _d(C.I64, (1 << 33,)), _d(C.BF16, (1 << 33, 1 << 33)), _d(C.BF16, (1 << 33, 128)), c) \
        == C.ROPE_ERR_PARAM_INVALID
    # a row stride whose extent (T - 1) * stride + width wraps
    assert _v2(lib, p, q, k, c, qs=1 << 62) == C.ROPE_ERR_PARAM_INVALID
    assert _v2(lib, p, q, k, c, ks=(1 << 62) + 8) == C.ROPE_ERR_PARAM_INVALID
    # slots = blocks * block size wraps although the caches hold no heads
    assert _qkv(lib, nq=4, nk=0, nv=0, qkv=_d(C.BF16, (6, 4 * 64)), qo=_d(C.BF16, (6, 4 * 64)),
                kc=_d(C.BF16, (big, 0, 1 << 30, 64)), vc=_d(C.BF16, (big, 0, 1 << 30, 64))) \
        == C.ROPE_ERR_PARAM_INVALID


# ---------------------------------------------------------------------------
# Aliasing: a tensor the call rewrites must not share memory with one it reads
# (the result would depend on the order in which threads run).  Only
# rejections are tested here: an accepted call would launch.
# ---------------------------------------------------------------------------
MB = 1 << 20  # distinct tensors sit MB apart


@pytest.mark.parametrize("cos_at,sin_at", [(FAKE + 256, FAKE + MB), (FAKE + MB, FAKE + 1024), (FAKE, FAKE)])
def test_inplace_x_sharing_memory_with_cos_or_sin_is_rejected(lib, cos_at, sin_at):
    x = _d(C.F32, X, FAKE)  # 6 KB
    assert _inplace(lib, x, _d(C.F32, CS, cos_at), _d(C.F32, CS, sin_at)) == C.ROPE_ERR_PARAM_INVALID


@pytest.mark.parametrize("q_at,k_at,p_at,c_at", [
    (FAKE, FAKE, FAKE + 4 * MB, FAKE + 8 * MB),             # query and key the same buffer
    (FAKE, FAKE + 512, FAKE + 4 * MB, FAKE + 8 * MB),       # key starts inside query
    (FAKE, FAKE + 2 * MB, FAKE + 1024, FAKE + 8 * MB),      # positions inside query
    (FAKE, FAKE + 2 * MB, FAKE + 4 * MB, FAKE + 2 * MB + 64),  # the cache inside key
])
def test_cache_rewritten_rows_sharing_memory_are_rejected(lib, q_at, k_at, p_at, c_at):
    _, q, k, c = good()
    pos = _d(C.I64, (T,), p_at)
    q, k, c = _d(q.dtype, tuple(q.shape[:2]), q_at), _d(k.dtype, tuple(k.shape[:2]), k_at), \
        _d(c.dtype, tuple(c.shape[:2]), c_at)
    assert _cache(lib, pos, q, k, c) == C.ROPE_ERR_PARAM_INVALID


def test_cache_row_views_whose_columns_collide_are_rejected(lib):
    # q and k as row views of one [T, 3 * 256] buffer: k's columns [128, 384)
    # cross q's [0, 256); the disjoint layout ([256, 384)) is what fused QKV
    # buffers use and is exercised on the GPU
    W = 3 * 256
    q = _d(C.BF16, (T, 256), FAKE)
    k = _d(C.BF16, (T, 128), FAKE + 128 * 2)
    assert _v2(lib, _d(C.I64, (T,), FAKE + 4 * MB), q, k, _d(C.BF16, (100, 64), FAKE + 8 * MB), qs=W,
               ks=W) == C.ROPE_ERR_PARAM_INVALID


@pytest.mark.parametrize("over", [
    dict(qo=_d(C.BF16, (6, 2 * 64), 1 * MB + 1024)),      # q_out inside qkv
    dict(vc=_d(C.BF16, (3, 1, 4, 64), 12 * MB)),          # v_cache is k_cache
    dict(kc=_d(C.BF16, (3, 1, 4, 64), 10 * MB + 512)),    # k_cache over q_out
    dict(slots=_d(C.I64, (6,), 12 * MB + 8)),             # slot_mapping inside k_cache
], ids=["q_out_in_qkv", "v_cache_is_k_cache", "k_cache_over_q_out", "slots_in_k_cache"])
def test_qkv_outputs_sharing_memory_are_rejected(lib, over):
    D = 64
    t = dict(qkv=_d(C.BF16, (6, 4 * D), 1 * MB), qg=_d(C.BF16, (D,), 2 * MB), kg=_d(C.BF16, (D,), 3 * MB),
             cache=_d(C.BF16, (50, D), 4 * MB), sl=_d(C.I64, (2,), 5 * MB), qsl=_d(C.I64, (3,), 6 * MB),
             slots=_d(C.I64, (6,), 7 * MB), qo=_d(C.BF16, (6, 2 * D), 10 * MB),
             kc=_d(C.BF16, (3, 1, 4, D), 12 * MB), vc=_d(C.BF16, (3, 1, 4, D), 13 * MB))
    t.update(over)
    assert _qkv(lib, **t) == C.ROPE_ERR_PARAM_INVALID
