"""Parity of the in-place partial interleave kernel against the oracle.

Every case runs the CUDA library through the C ABI and the oracle on the same
seeded inputs, then applies the tolerances of ``parity.py``: float32 within
2e-6 relative, float16/bfloat16 within one ulp, untouched columns bit-exact.
"""
import pytest
import torch

import oracle
import transformer_rope_positional_gb300 as R
import workloads as W
from gpu_runs import gpu_inplace, oracle_inplace
from parity import assert_matches, same_bits

pytestmark = pytest.mark.gpu

COMBOS = [(torch.float32, torch.float32), (torch.float16, torch.float16), (torch.bfloat16, torch.bfloat16),
          (torch.float16, torch.float32), (torch.bfloat16, torch.float32)]
COMBO_IDS = ["f32", "f16", "bf16", "f16x_f32cs", "bf16x_f32cs"]


def _check(case):
    got = gpu_inplace(case)
    ref = oracle_inplace(case)
    return assert_matches(got, ref, case.name)


@pytest.mark.parametrize("variant", ["slice", "full"])
def test_small_f32_workload(rope_gpu, variant):
    _check(W.inplace_f32_small(variant))


def test_small_f32_noop_is_bit_exact_and_launches_nothing(rope_gpu):
    case = W.inplace_f32_small("noop")
    before = R.launch_count()
    got = gpu_inplace(case)
    assert R.launch_count() == before
    assert same_bits(got, case.x)


def test_mixed_bf16_workload_reduced(rope_gpu):
    # the [4,4096,32,128] workload with S cut to 96 and B to 2: same layout and slice
    case = W.inplace_case("bf16_mixed_reduced", 1, (2, 96, 32, 128), 64, 128, torch.bfloat16, torch.float32)
    _check(case)


LAYOUTS = {
    "1S1L": lambda B, S, N, L: (1, S, 1, L),
    "BS1L": lambda B, S, N, L: (B, S, 1, L),
    "B11L": lambda B, S, N, L: (B, 1, 1, L),
    "111L": lambda B, S, N, L: (1, 1, 1, L),
    "BSNL": lambda B, S, N, L: (B, S, N, L),
    "B1NL": lambda B, S, N, L: (B, 1, N, L),
    "1SNL": lambda B, S, N, L: (1, S, N, L),
}
SLICES = [(0, 0), (32, 96), (8, 40), (2, 34), (3, 35), (94, 96)]


@pytest.mark.parametrize("combo", COMBOS, ids=COMBO_IDS)
@pytest.mark.parametrize("layout", list(LAYOUTS))
@pytest.mark.parametrize("sl", SLICES, ids=[f"{a}_{b}" for a, b in SLICES])
def test_dtypes_layouts_slices(rope_gpu, combo, layout, sl):
    B, S, N, D = 3, 37, 5, 96
    start, end = sl
    L = D if (start, end) == (0, 0) else end - start
    kind = "randn" if layout in ("BSNL", "B1NL") else "rotary"
    case = W.inplace_case(f"{layout}_{start}_{end}", 31, (B, S, N, D), start, end, combo[0], combo[1],
                          cs_shape=LAYOUTS[layout](B, S, N, L), cs_kind=kind)
    _check(case)


@pytest.mark.parametrize("combo", COMBOS, ids=COMBO_IDS)
def test_columns_outside_slice_are_bit_exact(rope_gpu, combo):
    case = W.inplace_case("sentinels", 41, (2, 9, 3, 64), 16, 48, combo[0], combo[1])
    x = case.x.clone()
    bits = {4: torch.int32, 2: torch.int16}[x.element_size()]
    nan_base = 0x7FC00001 if x.element_size() == 4 else 0x7E01
    fill = torch.arange(64, dtype=torch.int64) + nan_base
    xv = x.view(bits)
    xv[..., :16] = fill[:16].to(bits)
    xv[..., 48:] = fill[48:].to(bits)
    case.x = x
    got = gpu_inplace(case)
    assert same_bits(got[..., :16], x[..., :16]) and same_bits(got[..., 48:], x[..., 48:])
    assert_matches(got, oracle_inplace(case), "sentinels")


def test_page_example_shapes_b11d(rope_gpu):
    # x {96,1,1,512}, cos/sin {96,1,1,64}, slice {448,512}, all float32
    case = W.inplace_case("b11d_example", 51, (96, 1, 1, 512), 448, 512, torch.float32, torch.float32,
                          cs_shape=(96, 1, 1, 64))
    _check(case)


def test_python_example_randn_cos_sin_fp16(rope_gpu):
    # B=2, S=32, N=8, D=128, slice [0, 64), fp16 x and randn cos/sin of shape [B, S, 1, 64]
    case = W.inplace_case("py_example", 52, (2, 32, 8, 128), 0, 64, torch.float16, torch.float16,
                          cs_shape=(2, 32, 1, 64), cs_kind="randn")
    _check(case)


@pytest.mark.parametrize("combo", COMBOS, ids=COMBO_IDS)
def test_special_values(rope_gpu, combo):
    case = W.inplace_case("special", 53, (2, 4, 3, 32), 0, 32, combo[0], combo[1])
    x = case.x.clone().float()
    flat = x.view(-1)
    flat[0::17] = float("inf")
    flat[5::23] = float("-inf")
    flat[9::29] = float("nan")
    tiny = 1e-40 if combo[0] == torch.float32 else 1e-7
    flat[3::31] = tiny
    flat[7::37] = 6e4 if combo[0] == torch.float16 else 1e30
    case.x = x.to(combo[0])
    _check(case)


@pytest.mark.parametrize("combo", COMBOS, ids=COMBO_IDS)
@pytest.mark.parametrize("shape", [(1, 1, 1, 64), (1, 1, 3, 128), (1, 2, 40, 64), (5, 1, 1, 1024)])
def test_decode_and_edge_shapes(rope_gpu, combo, shape):
    D = shape[3]
    case = W.inplace_case("edge", 54, shape, 0, 0, combo[0], combo[1])
    _check(case)
    case2 = W.inplace_case("edge_tail", 55, shape, D - 2, D, combo[0], combo[1])
    _check(case2)


@pytest.mark.parametrize("combo", COMBOS, ids=COMBO_IDS)
def test_misaligned_base_pointer(rope_gpu, combo):
    case = W.inplace_case("misaligned", 56, (2, 6, 4, 64), 0, 32, combo[0], combo[1])
    n = case.x.numel()
    buf = torch.empty(n + 1, dtype=case.x.dtype, device="cuda")
    x = buf[1:].view(case.x.shape)
    x.copy_(case.x.cuda())
    R.rope_inplace_partial(x, case.cos.cuda(), case.sin.cuda(), 1, [0, 32])
    torch.cuda.synchronize()
    assert_matches(x.cpu(), oracle_inplace(case), "misaligned")


def test_empty_x_launches_nothing(rope_gpu):
    x = torch.empty(0, 4, 2, 64, device="cuda")
    c = torch.ones(1, 4, 1, 64, device="cuda")
    before = R.launch_count()
    R.rope_inplace_partial(x, c, c)
    assert R.launch_count() == before


def test_rejected_arguments_raise(rope_gpu):
    x = torch.zeros(1, 2, 2, 64, device="cuda")
    c = torch.ones(1, 2, 1, 64, device="cuda")
    with pytest.raises(R.RopeError) as e:
        R.rope_inplace_partial(x, c, c, rotary_mode=2)
    assert e.value.status == R.ROPE_ERR_PARAM_INVALID
    with pytest.raises(R.RopeError):
        R.rope_inplace_partial(x, c, c, partial_slice=[0, 32])  # cos width != slice


def test_runs_on_a_side_stream(rope_gpu):
    case = W.inplace_case("stream", 57, (2, 16, 4, 64), 0, 64, torch.bfloat16, torch.float32)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        got = gpu_inplace(case, stream=s)
    assert_matches(got, oracle_inplace(case), "side stream")


def test_repeated_application_is_deterministic(rope_gpu):
    case = W.inplace_case("determinism", 58, (2, 33, 7, 128), 0, 128, torch.bfloat16, torch.float32)
    a = gpu_inplace(case)
    b = gpu_inplace(case)
    assert same_bits(a, b)
    # oracle applied twice equals the kernel applied twice (each step within tolerance)
    twice = oracle.inplace_partial_rotary_mul(oracle_inplace(case), case.cos, case.sin, 0, 128)
    x = case.x.cuda()
    for _ in range(2):
        R.rope_inplace_partial(x, case.cos.cuda(), case.sin.cuda())
    torch.cuda.synchronize()
    from parity import ulp_distance
    assert ulp_distance(x.cpu(), twice).max() <= 2
