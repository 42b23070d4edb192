"""RoPE oracle -- TEST INFRASTRUCTURE ONLY.

Python marshalling around ``rope_oracle.c``, the plain binary64 CPU statement
of the two operators.  Only ``tests/``, the package smoke check and the
benchmark's CPU-baseline / reference legs may import this module; the product
path (``transformer_rope_positional_gb300``) never does, and shares no code
with it.

All functions take CPU tensors in their storage dtype and return new CPU
tensors; the inputs are never modified.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence, Tuple

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rope_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "librope_oracle.so")
_lib = None

F32, F16, BF16 = 0, 1, 2
_CODE = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}
_BITS = {torch.float32: torch.int32, torch.float16: torch.int16, torch.bfloat16: torch.int16}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    if _LIB_PATH != os.path.join(_OUT_DIR, "librope_oracle.so"):
        return _LIB_PATH
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    os.makedirs(_OUT_DIR, exist_ok=True)
    tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    "-fno-fast-math", _SRC, "-o", tmp, "-lm"], check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _get_lib():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.oracle_decode.argtypes = [ctypes.c_uint32, ctypes.c_int]
        lib.oracle_decode.restype = ctypes.c_double
        lib.oracle_encode.argtypes = [ctypes.c_double, ctypes.c_int]
        lib.oracle_encode.restype = ctypes.c_uint32
        lib.oracle_inplace_partial_rope.argtypes = [
            ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_int]
        lib.oracle_inplace_partial_rope.restype = ctypes.c_int
        lib.oracle_rope_with_sin_cos_cache.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
            ctypes.c_int64, ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int]
        lib.oracle_rope_with_sin_cos_cache.restype = ctypes.c_int64
        lib.oracle_qkv_rmsnorm_rope_cache.argtypes = [
            ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_double, ctypes.c_void_p, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_qkv_rmsnorm_rope_cache.restype = ctypes.c_int64
        _lib = lib
    return _lib


def use_library(path: Optional[str]) -> None:
    """Load the oracle from another build of ``rope_oracle.c`` (``None``: the
    default one).  Used only by the tests that plant mistakes in a copy of the
    oracle to show that the pins catch them."""
    global _lib, _LIB_PATH
    _lib = None
    _LIB_PATH = path or os.path.join(_OUT_DIR, "librope_oracle.so")


def build_copy(src_text: str, out_path: str) -> str:
    """Compile ``src_text`` (a variant of ``rope_oracle.c``) to ``out_path``."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    "-fno-fast-math", src, "-o", out_path, "-lm"], check=True, capture_output=True)
    return out_path


def _cpu(t: torch.Tensor) -> torch.Tensor:
    return t.detach().to("cpu").contiguous()


def decode(bits: int, dtype: torch.dtype) -> float:
    """Exact value of one ``dtype`` bit pattern."""
    return _get_lib().oracle_decode(bits & 0xFFFFFFFF, _CODE[dtype])


def encode(value: float, dtype: torch.dtype) -> int:
    """Bits of ``value`` rounded to nearest-even in ``dtype``."""
    return _get_lib().oracle_encode(float(value), _CODE[dtype])


def round_to(values: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    """Round float64 ``values`` once to ``dtype`` (returns a CPU tensor)."""
    flat = np.asarray(values, dtype=np.float64).reshape(-1)
    lib = _get_lib()
    code = _CODE[dtype]
    bits = np.fromiter((lib.oracle_encode(float(v), code) for v in flat), dtype=np.uint32,
                       count=flat.size)
    if dtype == torch.float32:
        out = torch.from_numpy(bits.view(np.int32).copy()).view(torch.float32)
    else:
        out = torch.from_numpy(bits.astype(np.uint16).view(np.int16).copy()).view(dtype)
    return out.reshape(np.shape(values))


def inplace_partial_rotary_mul(x: torch.Tensor, cos: torch.Tensor, sin: torch.Tensor,
                               start: int, end: int, rotary_mode: int = 1,
                               backward: bool = False) -> torch.Tensor:
    """Oracle of the in-place partial operator (mode 1 interleave, 0 half).

    Forward returns the new x; ``backward=True`` treats ``x`` as dL/dy and
    returns dL/dx."""
    out = _cpu(x).clone()
    c, s = _cpu(cos), _cpu(sin)
    assert out.dim() == 4 and c.dim() == 4 and tuple(c.shape) == tuple(s.shape)
    assert c.dtype == s.dtype and rotary_mode in (0, 1)
    xs = (ctypes.c_int64 * 4)(*out.shape)
    cs = (ctypes.c_int64 * 4)(*c.shape)
    rc = _get_lib().oracle_inplace_partial_rope(
        out.data_ptr(), _CODE[out.dtype], ctypes.addressof(xs), c.data_ptr(), s.data_ptr(),
        _CODE[c.dtype], ctypes.addressof(cs), int(start), int(end), int(rotary_mode), 1 if backward else 0)
    if rc != 0:
        raise MemoryError("oracle allocation failed")
    return out


def rope_with_sin_cos_cache(positions: torch.Tensor, query: torch.Tensor, key: torch.Tensor,
                            cache: torch.Tensor, head_size: int, is_neox: bool = True,
                            mrope_section: Optional[Sequence[int]] = None, cache_mode: int = 0
                            ) -> Tuple[torch.Tensor, torch.Tensor, int]:
    """Oracle of the cache-indexed operator.

    Returns ``(query_out, key_out, skipped)`` where ``skipped`` counts tokens
    left untouched because a position fell outside ``[0, cache.shape[0])``.
    """
    q, k, c = _cpu(query).clone(), _cpu(key).clone(), _cpu(cache)
    pos = _cpu(positions).to(torch.int64)
    assert q.dtype == k.dtype == c.dtype
    sec = None
    sec_len = 0
    sec_ptr = None
    if mrope_section is not None:
        sec = (ctypes.c_int64 * len(mrope_section))(*[int(v) for v in mrope_section])
        sec_len = len(mrope_section)
        sec_ptr = ctypes.addressof(sec)
    T = q.shape[0]
    skipped = _get_lib().oracle_rope_with_sin_cos_cache(
        pos.data_ptr(), sec_ptr, sec_len, q.data_ptr(), q.shape[1], k.data_ptr(), k.shape[1], T,
        c.data_ptr(), c.shape[0], c.shape[1], _CODE[c.dtype], int(head_size), 1 if is_neox else 0,
        int(cache_mode))
    if skipped < 0:
        raise ValueError("oracle rejected the inputs (allocation or mrope section sum)")
    return q, k, int(skipped)


def qkv_rmsnorm_rope_cache(qkv: torch.Tensor, num_q_heads: int, num_k_heads: int, num_v_heads: int,
                           q_gamma: torch.Tensor, k_gamma: torch.Tensor, eps: float, cache: torch.Tensor,
                           seq_lens: torch.Tensor, query_start_loc: torch.Tensor, slot_mapping: torch.Tensor,
                           q_out: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor):
    """Oracle of the fused QKV split + RMSNorm + RoPE + paged cache write.

    ``q_out``, ``k_cache`` and ``v_cache`` give the initial contents (entries the
    operator does not write keep them).  Returns ``(q_out, k_cache, v_cache,
    bad_positions, bad_slots)`` as new CPU tensors."""
    x = _cpu(qkv)
    qo, kc, vc = _cpu(q_out).clone(), _cpu(k_cache).clone(), _cpu(v_cache).clone()
    qg, kg, c = _cpu(q_gamma), _cpu(k_gamma), _cpu(cache)
    sl, qs, sm = (_cpu(t).to(torch.int64) for t in (seq_lens, query_start_loc, slot_mapping))
    assert x.dtype == qg.dtype == kg.dtype == c.dtype == qo.dtype == kc.dtype == vc.dtype
    T = x.shape[0]
    D = x.shape[1] // (num_q_heads + num_k_heads + num_v_heads)
    r = _get_lib().oracle_qkv_rmsnorm_rope_cache(
        x.data_ptr(), _CODE[x.dtype], T, num_q_heads, num_k_heads, num_v_heads, D, qg.data_ptr(), kg.data_ptr(),
        float(eps), c.data_ptr(), c.shape[0], sl.data_ptr(), qs.data_ptr(), sl.shape[0], sm.data_ptr(),
        kc.shape[2], kc.shape[0], qo.data_ptr(), kc.data_ptr(), vc.data_ptr())
    if r == -2:
        raise ValueError("query_start_loc must be non-decreasing within [0, T]")
    if r < 0:
        raise MemoryError("oracle allocation failed")
    return qo, kc, vc, int(r & 0xFFFFFFFF), int(r >> 32)


def exact_values(t: torch.Tensor) -> np.ndarray:
    """float64 copy of a float32/float16/bfloat16 CPU tensor (exact widening)."""
    return _cpu(t).to(torch.float64).numpy()
