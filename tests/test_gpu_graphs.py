"""The operators inside a captured CUDA graph: launches with programmatic
stream serialization are recorded as graph nodes and replay with the same
results as direct calls."""
import pytest
import torch

import oracle
import transformer_rope_positional_gb300 as R
import workloads as W
from parity import assert_matches

pytestmark = pytest.mark.gpu


def test_graph_capture_and_replay(rope_gpu):
    ic = W.inplace_case("graph_inplace", 141, (2, 64, 8, 128), 64, 128, torch.bfloat16, torch.float32)
    cc = W.cache_case("graph_cache", 142, 500, 8, 2, 128, 128, 1000, torch.bfloat16, True)
    mc = W.cache_case("graph_mrope", 143, 300, 4, 2, 128, 128, 700, torch.bfloat16, False,
                      mrope_section=[16, 24, 24])
    x, cs, sn = ic.x.cuda(), ic.cos.cuda(), ic.sin.cuda()
    ins = [(c.positions.cuda(), c.query.cuda(), c.key.cuda(), c.cache.cuda()) for c in (cc, mc)]
    x0 = x.clone()
    qk0 = [(q.clone(), k.clone()) for _, q, k, _ in ins]
    R.load()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            R.rope_inplace_partial(x, cs, sn, 1, [64, 128])
            for (p, q, k, cache), c in zip(ins, (cc, mc)):
                R.rope_with_sin_cos_cache(p, q, k, cache, c.head_size, c.rotary_dim, c.is_neox, c.mrope_section)
    torch.cuda.synchronize()
    # capture records work without running it: restore the inputs, then replay twice
    for reps in (1, 2):
        x.copy_(x0)
        for (_, q, k, _), (q0, k0) in zip(ins, qk0):
            q.copy_(q0)
            k.copy_(k0)
        for _ in range(reps):
            graph.replay()
        torch.cuda.synchronize()
        xr, qr = ic.x, [(c.query, c.key) for c in (cc, mc)]
        for _ in range(reps):
            xr = oracle.inplace_partial_rotary_mul(xr, ic.cos, ic.sin, 64, 128)
            qr = [oracle.rope_with_sin_cos_cache(c.positions, q_, k_, c.cache, c.head_size, c.is_neox,
                                                 c.mrope_section)[:2] for c, (q_, k_) in zip((cc, mc), qr)]
        tol_ok = reps == 1  # after two applications each side has rounded twice
        if tol_ok:
            assert_matches(x.cpu(), xr, "graph inplace")
            for (_, q, k, _), (qo, ko) in zip(ins, qr):
                assert_matches(q.cpu(), qo, "graph query")
                assert_matches(k.cpu(), ko, "graph key")
        else:
            from parity import ulp_distance
            assert ulp_distance(x.cpu(), xr).max() <= 2
            for (_, q, k, _), (qo, ko) in zip(ins, qr):
                assert ulp_distance(q.cpu(), qo).max() <= 2 and ulp_distance(k.cpu(), ko).max() <= 2
    assert R.get_device_error() == 0


def test_graph_fused_qkv(rope_gpu):
    """The fused op (dynamic shared memory for its batch tables) captured and
    replayed: outputs as the oracle's."""
    from test_gpu_qkv import _check, _run_oracle
    case = W.qkv_case("graph_qkv", 144, [37, 1, 1, 64, 3], [0, 100, 5, 30, 200], 4, 2, 2, 128, 16,
                      torch.bfloat16, pad_every=7)
    d = lambda t: t.cuda()  # noqa: E731
    ins = [d(t) for t in (case.qkv, case.q_gamma, case.k_gamma, case.cache, case.seq_lens, case.query_start_loc,
                          case.slot_mapping)]
    qo, kc, vc = d(case.q_out), d(case.k_cache), d(case.v_cache)
    qo0, kc0, vc0 = qo.clone(), kc.clone(), vc.clone()
    R.load()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            R.qkv_rmsnorm_rope_cache(ins[0], case.nq, case.nk, case.nv, ins[1], ins[2], case.eps, ins[3], ins[4],
                                     ins[5], ins[6], qo, kc, vc)
    torch.cuda.synchronize()
    for t, t0 in ((qo, qo0), (kc, kc0), (vc, vc0)):
        t.copy_(t0)
    for _ in range(2):  # the op does not read its outputs: replaying twice gives the same result
        graph.replay()
    torch.cuda.synchronize()
    _check(case, (qo.cpu(), kc.cpu(), vc.cpu()), _run_oracle(case))
    assert R.get_device_error() == 0
