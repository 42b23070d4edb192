"""Parity of the in-place kernels in half mode (rotary_mode 0) and of the
backward in both modes, against the oracle; plus the autograd entry point."""
import pytest
import torch

import oracle
import transformer_rope_positional_gb300 as R
import workloads as W
from parity import assert_matches, same_bits

pytestmark = pytest.mark.gpu

COMBOS = [(torch.float32, torch.float32), (torch.float16, torch.float16), (torch.bfloat16, torch.bfloat16),
          (torch.float16, torch.float32), (torch.bfloat16, torch.float32)]
COMBO_IDS = ["f32", "f16", "bf16", "f16x_f32cs", "bf16x_f32cs"]
LAYOUTS = {
    "1S1L": lambda B, S, N, L: (1, S, 1, L),
    "BS1L": lambda B, S, N, L: (B, S, 1, L),
    "BSNL": lambda B, S, N, L: (B, S, N, L),
    "111L": lambda B, S, N, L: (1, 1, 1, L),
}
SLICES = [(0, 0), (32, 96), (8, 40), (2, 34), (3, 35), (94, 96)]
RUNS = [("half", False), ("half", True), ("interleave", True)]


def _gpu(case, mode, backward):
    x = case.x.cuda()
    fn = R.rope_inplace_partial_backward if backward else R.rope_inplace_partial
    fn(x, case.cos.cuda(), case.sin.cuda(), mode, [case.start, case.end])
    torch.cuda.synchronize()
    return x.cpu()


def _oracle(case, mode, backward):
    return oracle.inplace_partial_rotary_mul(case.x, case.cos, case.sin, case.start, case.end,
                                             rotary_mode=R._capi.MODES[mode], backward=backward)


@pytest.mark.parametrize("run", RUNS, ids=["half_fwd", "half_bwd", "interleave_bwd"])
@pytest.mark.parametrize("combo", COMBOS, ids=COMBO_IDS)
@pytest.mark.parametrize("layout", list(LAYOUTS))
@pytest.mark.parametrize("sl", SLICES, ids=[f"{a}_{b}" for a, b in SLICES])
def test_modes_and_directions(rope_gpu, run, combo, layout, sl):
    mode, backward = run
    B, S, N, D = 3, 29, 5, 96
    start, end = sl
    L = D if (start, end) == (0, 0) else end - start
    case = W.inplace_case("modes", 101, (B, S, N, D), start, end, combo[0], combo[1],
                          cs_shape=LAYOUTS[layout](B, S, N, L), cs_kind="randn")
    assert_matches(_gpu(case, mode, backward), _oracle(case, mode, backward), f"{mode} bwd={backward}")


@pytest.mark.parametrize("run", RUNS, ids=["half_fwd", "half_bwd", "interleave_bwd"])
def test_mixed_bf16_layout_reduced(rope_gpu, run):
    mode, backward = run
    case = W.inplace_case("bf16_mixed_reduced", 1, (2, 80, 32, 128), 64, 128, torch.bfloat16, torch.float32)
    assert_matches(_gpu(case, mode, backward), _oracle(case, mode, backward), "reduced")


@pytest.mark.parametrize("run", RUNS, ids=["half_fwd", "half_bwd", "interleave_bwd"])
def test_untouched_columns_and_noop(rope_gpu, run):
    mode, backward = run
    case = W.inplace_case("sentinel", 102, (2, 7, 3, 64), 16, 48, torch.bfloat16, torch.float32)
    x = case.x.clone()
    xv = x.view(torch.int16)
    xv[..., :16] = (torch.arange(16) + 0x7E01).to(torch.int16)
    xv[..., 48:] = (torch.arange(16) + 0x7E21).to(torch.int16)
    case.x = x
    got = _gpu(case, mode, backward)
    assert same_bits(got[..., :16], x[..., :16]) and same_bits(got[..., 48:], x[..., 48:])
    before = R.launch_count()
    case.start, case.end = 8, 8
    assert same_bits(_gpu(case, mode, backward), x)
    assert R.launch_count() == before


def test_backward_then_forward_is_identity_for_a_rotation(rope_gpu):
    """With true rotations the backward is the inverse rotation: forward then
    backward returns x within two roundings."""
    case = W.inplace_case("inverse", 103, (2, 33, 4, 64), 0, 0, torch.float32, torch.float32)
    x = case.x.cuda()
    R.rope_inplace_partial(x, case.cos.cuda(), case.sin.cuda())
    R.rope_inplace_partial_backward(x, case.cos.cuda(), case.sin.cuda())
    torch.cuda.synchronize()
    assert torch.allclose(x.cpu(), case.x, rtol=4e-7, atol=1e-6)


@pytest.mark.parametrize("mode", ["interleave", "half"])
@pytest.mark.parametrize("dt", [torch.float32, torch.float16, torch.bfloat16])
def test_autograd_entry_point(rope_gpu, mode, dt):
    """The page's training-mode usage: y = x * 1.0; rotate y in place; backward."""
    B, S, N, D = 2, 32, 8, 128
    x0 = W.normal(104, (B, S, N, D), dt)
    r1 = W.normal(105, (B, S, 1, 64), dt)
    r2 = W.normal(106, (B, S, 1, 64), dt)
    w = W.normal(107, (B, S, N, D), dt)
    x = x0.cuda().requires_grad_(True)
    y = x * 1.0
    R.inplace_partial_rotary_mul(y, r1.cuda(), r2.cuda(), rotary_mode=mode, partial_slice=[0, 64])
    (y * w.cuda()).sum().backward()
    code = R._capi.MODES[mode]
    assert_matches(y.detach().cpu(), oracle.inplace_partial_rotary_mul(x0, r1, r2, 0, 64, rotary_mode=code),
                   "forward")
    assert_matches(x.grad.cpu(), oracle.inplace_partial_rotary_mul(w, r1, r2, 0, 64, rotary_mode=code,
                                                                   backward=True), "x.grad")


def test_autograd_without_grad_is_plain_call(rope_gpu):
    case = W.inplace_case("nograd", 108, (1, 4, 2, 32), 0, 0, torch.float16, torch.float16)
    x = case.x.cuda()
    assert R.inplace_partial_rotary_mul(x, case.cos.cuda(), case.sin.cuda()) is None
    torch.cuda.synchronize()
    assert_matches(x.cpu(), oracle.inplace_partial_rotary_mul(case.x, case.cos, case.sin, 0, 0), "nograd")
