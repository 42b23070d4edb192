"""Operators on tensors of more than 2^31 elements: every offset past the
32-bit range must be formed in 64-bit arithmetic.

The large inputs are tiled on the device from a small seeded block (token s
holds block row s % rows), so the oracle checks sampled rows from the block,
among them the rows on both sides of element 2^31."""
import pytest
import torch

import oracle
import transformer_rope_positional_gb300 as R
import workloads as W
from parity import assert_close_scaled, assert_matches, same_bits

pytestmark = pytest.mark.gpu


def test_inplace_past_2_31_elements(rope_gpu):
    B, S, N, D = 4, 16385, 32, 1024  # 2^31 + 2^17 bf16 elements (4.3 GB)
    start, end = 512, 1024
    rows = 64
    blk = W.inplace_case("large_inplace", 141, (1, rows, N, D), start, end, torch.bfloat16, torch.float32,
                         cs_shape=(1, S, 1, end - start))
    dev = torch.device("cuda")
    tile = torch.arange(S, device=dev) % rows
    x = blk.x.to(dev)[0][tile].unsqueeze(0).expand(B, S, N, D).contiguous()
    assert x.numel() > 2 ** 31
    R.rope_inplace_partial(x, blk.cos.to(dev), blk.sin.to(dev), 1, [start, end])
    torch.cuda.synchronize()
    # element 2^31 lies in token (b=3, s=16381): (3 * S + 16381) * N * D == 2^31
    assert (3 * S + 16381) * N * D == 2 ** 31
    for b, s in [(0, 0), (0, 1), (1, 8000), (2, 12345), (3, 16380), (3, 16381), (3, 16382), (3, S - 1)]:
        src = blk.x[:, s % rows:s % rows + 1]
        ref = oracle.inplace_partial_rotary_mul(src, blk.cos[:, s:s + 1], blk.sin[:, s:s + 1], start, end)
        got = x[b, s].cpu().unsqueeze(0).unsqueeze(0)
        assert_matches(got, ref, "token (%d, %d)" % (b, s))
        assert same_bits(got[..., :start], src[..., :start])


def test_cache_op_past_2_31_elements(rope_gpu):
    T, hq, hk, hs = (1 << 21) + 64, 8, 1, 128  # query: 2^31 + 2^13 bf16 elements (4.3 GB)
    rows, max_seq = 128, 4096
    blk = W.cache_case("large_cache", 142, rows, hq, hk, hs, hs, max_seq, torch.bfloat16, True)
    positions = W.uniform_int(W.stream_seed(142, 5), T, 0, max_seq)
    dev = torch.device("cuda")
    tile = torch.arange(T, device=dev) % rows
    q = blk.query.to(dev)[tile]
    k = blk.key.to(dev)[tile]
    assert q.numel() > 2 ** 31
    R.rope_with_sin_cos_cache(positions.to(dev), q, k, blk.cache.to(dev), hs, hs, True, None)
    torch.cuda.synchronize()
    assert R.get_device_error() == 0
    # query row t starts at element t * hq * hs; row 2^21 starts at 2^31
    sample = torch.tensor([0, 1, 77, (1 << 20) + 5, (1 << 21) - 1, 1 << 21, (1 << 21) + 1, T - 1])
    qo, ko, skipped = oracle.rope_with_sin_cos_cache(positions[sample], blk.query[sample % rows],
                                                     blk.key[sample % rows], blk.cache, hs, True)
    assert skipped == 0
    assert_matches(q[sample.to(dev)].cpu(), qo, "query rows")
    assert_matches(k[sample.to(dev)].cpu(), ko, "key rows")


def test_fused_qkv_past_2_31_elements(rope_gpu):
    """One sequence of T new tokens (positions 0..T-1) whose qkv buffer holds
    more than 2^31 elements; token t goes to cache slot t."""
    nq, nk, nv, D, BS = 32, 8, 8, 128, 16
    W_ = (nq + nk + nv) * D
    T = (1 << 31) // W_ + 64  # qkv: 2^31 + 2^18 bf16 elements (4.3 GB)
    rows = 96
    blk = W.qkv_case("large_qkv_block", 143, [rows], [0], nq, nk, nv, D, BS, torch.bfloat16)
    cache = W.cos_sin_cache(T, D, 10000.0, torch.bfloat16)
    dev = torch.device("cuda")
    tile = torch.arange(T, device=dev) % rows
    qkv = blk.qkv.to(dev)[tile]
    assert qkv.numel() > 2 ** 31
    NB = (T + BS - 1) // BS
    q_out = torch.full((T, nq * D), 3.0, dtype=torch.bfloat16, device=dev)
    k_cache = torch.full((NB, nk, BS, D), 5.0, dtype=torch.bfloat16, device=dev)
    v_cache = torch.full((NB, nv, BS, D), 7.0, dtype=torch.bfloat16, device=dev)
    seq_lens = torch.tensor([T], dtype=torch.int64)
    qsl = torch.tensor([0, T], dtype=torch.int64)
    slots = torch.arange(T, dtype=torch.int64)
    R.qkv_rmsnorm_rope_cache(qkv, nq, nk, nv, blk.q_gamma.to(dev), blk.k_gamma.to(dev), blk.eps, cache.to(dev),
                             seq_lens.to(dev), qsl.to(dev), slots.to(dev), q_out, k_cache, v_cache)
    torch.cuda.synchronize()
    assert R.get_device_error() == 0
    boundary = (1 << 31) // W_  # the token whose qkv row holds element 2^31
    for t in [0, 1, 1000, boundary - 1, boundary, boundary + 1, T - 1]:
        one = W.qkv_case("large_qkv_token", 143, [1], [0], nq, nk, nv, D, BS, torch.bfloat16)
        one.qkv = blk.qkv[t % rows:t % rows + 1].clone()
        ref_q, ref_k, ref_v, bp, bs = oracle.qkv_rmsnorm_rope_cache(
            one.qkv, nq, nk, nv, blk.q_gamma, blk.k_gamma, blk.eps, cache, torch.tensor([t + 1]),
            torch.tensor([0, 1]), torch.tensor([0]), one.q_out, one.k_cache, one.v_cache)
        assert bp == 0 and bs == 0
        x = one.qkv.double().reshape(1, -1, D)
        y = x / (x.pow(2).mean(-1, keepdim=True) + blk.eps).sqrt()
        scale_q = (2 * (y[:, :nq] * blk.q_gamma.double()).abs().amax(-1, keepdim=True)).numpy()
        scale_k = (2 * (y[:, nq:nq + nk] * blk.k_gamma.double()).abs().amax(-1, keepdim=True)).numpy()
        assert_close_scaled(q_out[t].cpu().view(1, nq, D), ref_q.view(1, nq, D), scale_q, 8e-6, "q token %d" % t)
        assert_close_scaled(k_cache[t // BS, :, t % BS].cpu().view(1, nk, D), ref_k[0, :, 0].view(1, nk, D),
                            scale_k, 8e-6, "k token %d" % t)
        assert same_bits(v_cache[t // BS, :, t % BS].cpu(), ref_v[0, :, 0])
