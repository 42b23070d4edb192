"""Operators called from several host threads at once, each on its own CUDA
stream (the C calls release the GIL): the host-side caches (occupancy, device
error word address) are shared, and every result must still be the oracle's."""
import threading

import pytest
import torch

import oracle
import transformer_rope_positional_gb300 as R
import workloads as W
from parity import assert_matches

pytestmark = pytest.mark.gpu


def test_concurrent_threads_and_streams(rope_gpu):
    R.load()
    ic = W.inplace_case("thr_inplace", 151, (2, 96, 8, 128), 64, 128, torch.bfloat16, torch.float32)
    nc = W.cache_case("thr_neox", 152, 700, 8, 2, 128, 128, 2048, torch.bfloat16, True)
    gc = W.cache_case("thr_gptj", 153, 500, 4, 4, 256, 64, 4096, torch.float16, False)
    mc = W.cache_case("thr_mrope", 154, 600, 4, 2, 128, 128, 1024, torch.bfloat16, True, mrope_section=[16, 24, 24])
    ref_x = oracle.inplace_partial_rotary_mul(ic.x, ic.cos, ic.sin, 64, 128)
    refs = {c.name: oracle.rope_with_sin_cos_cache(c.positions, c.query, c.key, c.cache, c.head_size, c.is_neox,
                                                   c.mrope_section)[:2] for c in (nc, gc, mc)}
    errors = []
    reps = 25

    def run_inplace():
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            cs, sn = ic.cos.cuda(), ic.sin.cuda()
            for _ in range(reps):
                x = ic.x.cuda()
                R.rope_inplace_partial(x, cs, sn, 1, [64, 128])
                s.synchronize()
                assert_matches(x.cpu(), ref_x, "thread inplace")

    def run_cache(c):
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            p, cache = c.positions.cuda(), c.cache.cuda()
            for _ in range(reps):
                q, k = c.query.cuda(), c.key.cuda()
                R.rope_with_sin_cos_cache(p, q, k, cache, c.head_size, c.rotary_dim, c.is_neox, c.mrope_section)
                s.synchronize()
                assert_matches(q.cpu(), refs[c.name][0], "thread %s query" % c.name)
                assert_matches(k.cpu(), refs[c.name][1], "thread %s key" % c.name)

    def guarded(fn, *a):
        try:
            fn(*a)
        except BaseException as e:  # reported to the main thread
            errors.append(e)

    threads = [threading.Thread(target=guarded, args=(run_inplace,))]
    threads += [threading.Thread(target=guarded, args=(run_cache, c)) for c in (nc, gc, mc)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors[0]
    torch.cuda.synchronize()
    assert R.get_device_error() == 0
