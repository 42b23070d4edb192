"""Calls whose rewritten tensors share memory with tensors they read are
refused on the host, before any launch, and leave every tensor as it was;
q and k as disjoint column ranges of one fused buffer are still accepted
(their parity is checked in test_gpu_cache_v2.py and test_gpu_guard_bands.py)."""
import pytest
import torch

import transformer_rope_positional_gb300 as R
import workloads as W
from parity import same_bits

pytestmark = pytest.mark.gpu


def _refused(call, *tensors):
    before = [t.clone() for t in tensors]
    torch.cuda.synchronize()
    n0 = R.launch_count()
    with pytest.raises(R.RopeError) as e:
        call()
    torch.cuda.synchronize()
    assert e.value.status == R.ROPE_ERR_PARAM_INVALID
    assert R.launch_count() == n0
    for t, b in zip(tensors, before):
        assert same_bits(t.cpu(), b.cpu())


def test_query_that_is_the_key(rope_gpu):
    case = W.cache_case("alias_qk", 130, 16, 2, 2, 64, 64, 100, torch.bfloat16, True)
    q = case.query.cuda()
    pos, cache = case.positions.cuda(), case.cache.cuda()
    _refused(lambda: R.rope_with_sin_cos_cache(pos, q, q, cache, 64), q)


def test_key_columns_crossing_the_query_columns(rope_gpu):
    case = W.cache_case("alias_cols", 131, 16, 2, 1, 64, 64, 100, torch.bfloat16, True)
    buf = torch.randn(16, 3 * 64, dtype=torch.bfloat16, device="cuda")
    q, k = buf[:, :128], buf[:, 64:128]  # k is the second q head
    pos, cache = case.positions.cuda(), case.cache.cuda()
    _refused(lambda: R.rope_with_sin_cos_cache(pos, q, k, cache, 64), buf)


def test_positions_inside_the_rewritten_rows(rope_gpu):
    case = W.cache_case("alias_pos", 132, 16, 2, 2, 64, 64, 100, torch.float32, True)
    q, k, cache = case.query.cuda(), case.key.cuda(), case.cache.cuda()
    pos = q.view(-1).view(torch.int64)[:16]  # 16 int64 values over q's first row
    _refused(lambda: R.rope_with_sin_cos_cache(pos, q, k, cache, 64), q, k)


def test_inplace_x_overlapping_cos(rope_gpu):
    case = W.inplace_case("alias_x", 133, (1, 4, 2, 64), 0, 64, torch.float32, torch.float32)
    x = case.x.cuda()
    cos = x.view(-1)[:4 * 64].view(1, 4, 1, 64)  # x's first 256 elements
    sin = case.sin.cuda()
    _refused(lambda: R.rope_inplace_partial(x, cos, sin, 1, [0, 64]), x, sin)


def test_fused_op_output_overlapping_its_input(rope_gpu):
    qc = W.qkv_case("alias_qkv", 134, [3, 2], [4, 9], 2, 1, 1, 64, 4, torch.bfloat16)
    t = [v.cuda() for v in (qc.qkv, qc.q_gamma, qc.k_gamma, qc.cache, qc.seq_lens, qc.query_start_loc,
                            qc.slot_mapping, qc.q_out, qc.k_cache, qc.v_cache)]
    q_out = t[0].view(-1)[:t[7].numel()].view(t[7].shape)  # q_out over the start of qkv itself
    assert q_out.shape == t[7].shape
    _refused(lambda: R.qkv_rmsnorm_rope_cache(t[0], qc.nq, qc.nk, qc.nv, t[1], t[2], qc.eps, t[3], t[4], t[5], t[6],
                                              q_out, t[8], t[9]), t[0], t[8], t[9])
    # and the same call with separate tensors is accepted
    R.qkv_rmsnorm_rope_cache(t[0], qc.nq, qc.nk, qc.nv, t[1], t[2], qc.eps, *t[3:])
    torch.cuda.synchronize()
    assert R.get_device_error() == 0


@pytest.mark.parametrize("neox", [True, False])
def test_key_columns_before_query_columns_are_accepted(rope_gpu, neox):
    """q and k as disjoint column ranges of one buffer, k first (a negative
    offset for the overlap check): accepted, and rotated as the oracle says."""
    import oracle
    from parity import assert_matches

    case = W.cache_case("k_first", 135, 24, 2, 1, 64, 64, 100, torch.bfloat16, neox)
    buf = torch.zeros(24, 4 * 64, dtype=torch.bfloat16, device="cuda")
    k, q = buf[:, :64], buf[:, 128:256]  # columns [64, 128) stay untouched
    k.copy_(case.key.cuda())
    q.copy_(case.query.cuda())
    R.rope_with_sin_cos_cache(case.positions.cuda(), q, k, case.cache.cuda(), 64, 64, neox)
    torch.cuda.synchronize()
    qr, kr, _ = oracle.rope_with_sin_cos_cache(case.positions, case.query, case.key, case.cache, 64, neox)
    assert_matches(q.cpu(), qr, "query")
    assert_matches(k.cpu(), kr, "key")
    assert not buf[:, 64:128].any()
