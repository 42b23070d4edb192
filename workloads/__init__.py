"""Seeded synthetic inputs for the RoPE workloads.

Shared by the parity tests, the benchmark and the oracle checks.  Nothing here
rotates anything: this module only draws random numbers (``gen.c``) and builds
the cos/sin inputs that the operators take as data.  Every tensor comes back on
the CPU in its storage dtype; callers move it to the device themselves.

Stream seeds: tensor ``k`` of a workload with seed ``s`` uses the SplitMix64
stream ``s * 16 + k``, so that adding a tensor never shifts the others.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field
from typing import Optional, Sequence

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libworkloads_gen.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``gen.c`` with gcc into ``_build/`` (OpenMP if available)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    os.makedirs(_OUT_DIR, exist_ok=True)
    tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _get_lib():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.wl_normal_f32.argtypes = [ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p]
        lib.wl_uniform_f64.argtypes = [ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p]
        lib.wl_uniform_int.argtypes = [ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64,
                                       ctypes.c_int64, ctypes.c_void_p]
        _lib = lib
    return _lib


def stream_seed(seed: int, tensor_id: int) -> int:
    return (seed * 16 + tensor_id) & 0xFFFFFFFFFFFFFFFF


def normal(seed: int, shape: Sequence[int], dtype: torch.dtype) -> torch.Tensor:
    """~N(0,1) draws (float32 Box-Muller values rounded once to ``dtype``)."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = torch.empty(n, dtype=torch.float32)
    if n:
        _get_lib().wl_normal_f32(seed, n, out.data_ptr())
    out = out.reshape(tuple(shape))
    return out if dtype == torch.float32 else out.to(dtype)


def uniform(seed: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    if n:
        _get_lib().wl_uniform_f64(seed, n, out.ctypes.data)
    return out


def uniform_int(seed: int, n: int, lo: int, hi: int) -> torch.Tensor:
    """``n`` int64 values uniform in ``[lo, hi)``."""
    out = torch.empty(n, dtype=torch.int64)
    if n:
        _get_lib().wl_uniform_int(seed, n, lo, hi, out.data_ptr())
    return out


# --------------------------------------------------------------------------
# cos/sin inputs.  Both operators take cos/sin as data; these builders give the
# usual rotary tables the workloads are defined with.
# --------------------------------------------------------------------------

def interleaved_cos_sin(positions: np.ndarray, length: int, base: float):
    """Per-element cos/sin rows for the in-place interleave operator.

    Element ``j`` of a row at position ``pos`` holds cos/sin of
    ``pos * base ** (-2 * (j // 2) / length)``: the two members of a pair share
    one angle.  Returns float64 arrays of shape ``[len(positions), length]``.
    """
    j = np.arange(length)
    theta = np.power(float(base), -2.0 * (j // 2) / float(length))
    ang = np.asarray(positions, dtype=np.float64)[:, None] * theta[None, :]
    return np.cos(ang), np.sin(ang)


def cos_sin_cache(max_seq: int, rotary_dim: int, base: float, dtype: torch.dtype) -> torch.Tensor:
    """``[max_seq, rotary_dim]`` table: row p = cos(p*theta_i) (i < R/2) then sin(p*theta_i)."""
    half = rotary_dim // 2
    i = np.arange(half)
    theta = np.power(float(base), -2.0 * i / float(rotary_dim))
    ang = np.arange(max_seq, dtype=np.float64)[:, None] * theta[None, :]
    table = np.concatenate([np.cos(ang), np.sin(ang)], axis=1)
    return torch.from_numpy(table).to(torch.float32).to(dtype).contiguous()


def _to(arr: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(arr)).to(torch.float32).to(dtype).contiguous()


# --------------------------------------------------------------------------
# Workload descriptions
# --------------------------------------------------------------------------

@dataclass
class InplaceCase:
    """Inputs of the in-place partial interleave operator (BSND x)."""
    name: str
    x: torch.Tensor
    cos: torch.Tensor
    sin: torch.Tensor
    start: int
    end: int
    rotary_mode: int = 1

    @property
    def tokens(self) -> int:
        return int(self.x.shape[0] * self.x.shape[1])


@dataclass
class CacheCase:
    """Inputs of the cache-indexed operator (rope or mrope)."""
    name: str
    positions: torch.Tensor
    query: torch.Tensor
    key: torch.Tensor
    cache: torch.Tensor
    head_size: int
    rotary_dim: int
    is_neox: bool
    mrope_section: Optional[Sequence[int]] = None
    meta: dict = field(default_factory=dict)

    @property
    def tokens(self) -> int:
        return int(self.query.shape[0])


def inplace_case(name: str, seed: int, shape: Sequence[int], start: int, end: int,
                 x_dtype: torch.dtype, cs_dtype: torch.dtype, cs_shape: Optional[Sequence[int]] = None,
                 base: float = 10000.0, cs_kind: str = "rotary") -> InplaceCase:
    """x ~ N(0,1) of ``shape``; cos/sin of ``cs_shape`` (default [1,S,1,L]).

    ``cs_kind='rotary'``: cos/sin row r (flat index over the first three dims
    of ``cs_shape``) is the rotation of position r, i.e. position s for the
    [1,S,1,L] layout.  ``cs_kind='randn'``: cos/sin are free N(0,1) tensors.
    """
    B, S, N, D = shape
    s0, e0 = (0, D) if (start == 0 and end == 0) else (start, end)
    L = e0 - s0
    if cs_shape is None:
        cs_shape = (1, S, 1, L)
    x = normal(stream_seed(seed, 0), shape, x_dtype)
    rows = int(np.prod(cs_shape[:3]))
    if cs_kind == "randn":
        cos = normal(stream_seed(seed, 1), cs_shape, cs_dtype)
        sin = normal(stream_seed(seed, 2), cs_shape, cs_dtype)
    else:
        pos = np.arange(rows, dtype=np.float64)
        c, s = interleaved_cos_sin(pos, cs_shape[3], base)
        cos = _to(c.reshape(cs_shape), cs_dtype)
        sin = _to(s.reshape(cs_shape), cs_dtype)
    return InplaceCase(name, x, cos, sin, start, end)


def cache_case(name: str, seed: int, num_tokens: int, q_heads: int, k_heads: int, head_size: int,
               rotary_dim: int, max_seq: int, dtype: torch.dtype, is_neox: bool, base: float = 10000.0,
               positions: Optional[torch.Tensor] = None,
               mrope_section: Optional[Sequence[int]] = None) -> CacheCase:
    """q/k ~ N(0,1); positions uniform in [0, max_seq) unless given."""
    q = normal(stream_seed(seed, 0), (num_tokens, q_heads * head_size), dtype)
    k = normal(stream_seed(seed, 1), (num_tokens, k_heads * head_size), dtype)
    if positions is None:
        rows = len(mrope_section) if mrope_section else 1
        p = uniform_int(stream_seed(seed, 2), rows * num_tokens, 0, max_seq)
        positions = p.reshape(rows, num_tokens) if mrope_section else p
    cache = cos_sin_cache(max_seq, rotary_dim, base, dtype)
    return CacheCase(name, positions.contiguous(), q, k, cache, head_size, rotary_dim, is_neox,
                     list(mrope_section) if mrope_section else None)


# --------------------------------------------------------------------------
# The five named workloads
# --------------------------------------------------------------------------

def inplace_f32_small(variant: str = "slice") -> InplaceCase:
    """x f32 [1,16,2,64] seed 0; slice [16,48) (or [0,0] whole-D, or [8,8] no-op)."""
    if variant == "slice":
        return inplace_case("inplace_f32_1x16x2x64_slice16_48", 0, (1, 16, 2, 64), 16, 48,
                            torch.float32, torch.float32)
    if variant == "full":
        return inplace_case("inplace_f32_1x16x2x64_slice0_0", 0, (1, 16, 2, 64), 0, 0,
                            torch.float32, torch.float32)
    if variant == "noop":
        c = inplace_case("inplace_f32_1x16x2x64_slice8_8", 0, (1, 16, 2, 64), 16, 48,
                         torch.float32, torch.float32)
        c.start, c.end = 8, 8
        return c
    raise ValueError(variant)


def inplace_bf16_mixed(batch: int = 4) -> InplaceCase:
    """x bf16 [4,4096,32,128] seed 1, slice [64,128), cos/sin f32 [1,4096,1,64] base 1e4."""
    return inplace_case("inplace_bf16x_f32cs_%dx4096x32x128_slice64_128" % batch, 1,
                        (batch, 4096, 32, 128), 64, 128, torch.bfloat16, torch.float32)


def cache_neox_bf16(num_tokens: int = 16384) -> CacheCase:
    """16384 tokens, q 32x128 / k 8x128 bf16, R=128, cache [32768,128], NeoX, seed 2."""
    return cache_case("rope_neox_bf16_%dtok_32q8k_h128" % num_tokens, 2, num_tokens, 32, 8, 128, 128,
                      32768, torch.bfloat16, True)


def cache_gptj_f16_partial(num_seqs: int = 8, seq_len: int = 1024) -> CacheCase:
    """8 seqs x 1024 consecutive positions from offsets < 60000; q/k 16x256 f16; R=64; GPT-J; seed 3."""
    offs = uniform_int(stream_seed(3, 2), num_seqs, 0, 60000)
    pos = (offs[:, None] + torch.arange(seq_len, dtype=torch.int64)[None, :]).reshape(-1)
    return cache_case("rope_gptj_f16_%dtok_16q16k_h256_r64" % (num_seqs * seq_len), 3,
                      num_seqs * seq_len, 16, 16, 256, 64, 65536, torch.float16, False, positions=pos)


def mrope_positions(text_tokens: int = 8192, grid=(6, 64, 64)) -> torch.Tensor:
    """[3, T] positions: text tokens have t=h=w=i; image tokens sit on a t/h/w grid
    (t-major, then h, then w) with every axis offset by the text length."""
    t_, h_, w_ = grid
    txt = torch.arange(text_tokens, dtype=torch.int64)
    tt, hh, ww = torch.meshgrid(torch.arange(t_), torch.arange(h_), torch.arange(w_), indexing="ij")
    img = torch.stack([tt.reshape(-1), hh.reshape(-1), ww.reshape(-1)]).to(torch.int64) + text_tokens
    return torch.cat([txt.expand(3, -1), img], dim=1).contiguous()


def mrope_neox_bf16() -> CacheCase:
    """positions [3,32768] (8192 text + 6x64x64 image), section [16,24,24], q 28x128 / k 4x128 bf16,
    cache [40960,128] base 1e6, NeoX, seed 4."""
    pos = mrope_positions()
    return cache_case("mrope_neox_bf16_32768tok_28q4k_h128_s16_24_24", 4, pos.shape[1], 28, 4, 128, 128,
                      40960, torch.bfloat16, True, base=1e6, positions=pos, mrope_section=[16, 24, 24])


# --------------------------------------------------------------------------
# Fused QKV split + RMSNorm + RoPE + paged KV-cache write
# --------------------------------------------------------------------------

@dataclass
class QkvCase:
    """Inputs of the fused QKV operator; q_out/k_cache/v_cache hold the initial
    contents (sentinel values that unwritten entries keep)."""
    name: str
    qkv: torch.Tensor
    nq: int
    nk: int
    nv: int
    q_gamma: torch.Tensor
    k_gamma: torch.Tensor
    eps: float
    cache: torch.Tensor
    seq_lens: torch.Tensor
    query_start_loc: torch.Tensor
    slot_mapping: torch.Tensor
    q_out: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor

    @property
    def tokens(self) -> int:
        return int(self.qkv.shape[0])

    @property
    def head_size(self) -> int:
        return int(self.qkv.shape[1]) // (self.nq + self.nk + self.nv)


def qkv_case(name: str, seed: int, query_lens: Sequence[int], context_lens: Sequence[int], nq: int, nk: int,
             nv: int, head_size: int, block_size: int, dtype: torch.dtype, base: float = 10000.0,
             eps: float = 1e-6, pad_every: int = 0) -> QkvCase:
    """Batches with ``query_lens[b]`` new tokens on top of ``context_lens[b]``
    cached ones (seqLens = context + query).  Paged cache as in paged-attention
    serving: every sequence owns ceil(seqLen / block_size) blocks drawn from a
    shuffled pool, and the token at position p goes to slot
    block_table[p // block_size] * block_size + p % block_size.  With
    ``pad_every`` > 0 every pad_every-th token gets slot -1 (padding)."""
    T = int(sum(query_lens))
    seq_lens = torch.tensor([c + q for c, q in zip(context_lens, query_lens)], dtype=torch.int64)
    qsl = torch.tensor([0] + list(np.cumsum(query_lens)), dtype=torch.int64)
    W = (nq + nk + nv) * head_size
    qkv = normal(stream_seed(seed, 0), (T, W), dtype)
    g = normal(stream_seed(seed, 1), (2, head_size), torch.float32)
    q_gamma = (1.0 + 0.25 * g[0]).to(dtype)
    k_gamma = (1.0 + 0.25 * g[1]).to(dtype)
    max_seq = int(seq_lens.max()) + 1
    cache = cos_sin_cache(max_seq, head_size, base, dtype)
    blocks_per_seq = [(int(n) + block_size - 1) // block_size for n in seq_lens]
    num_blocks = sum(blocks_per_seq) + 1
    pool = np.argsort(uniform(stream_seed(seed, 2), num_blocks), kind="stable")
    slots = torch.empty(T, dtype=torch.int64)
    first = 0
    for b, (q_len, c_len) in enumerate(zip(query_lens, context_lens)):
        table = pool[sum(blocks_per_seq[:b]):sum(blocks_per_seq[:b + 1])]
        p = np.arange(c_len, c_len + q_len)
        slots[first:first + q_len] = torch.from_numpy(table[p // block_size] * block_size + p % block_size)
        first += q_len
    if pad_every:
        slots[::pad_every] = -1
    q_out = torch.full((T, nq * head_size), 3.0, dtype=dtype)
    k_cache = torch.full((num_blocks, nk, block_size, head_size), 5.0, dtype=dtype)
    v_cache = torch.full((num_blocks, nv, block_size, head_size), 7.0, dtype=dtype)
    return QkvCase(name, qkv, nq, nk, nv, q_gamma, k_gamma, eps, cache, seq_lens, qsl, slots, q_out, k_cache,
                   v_cache)


def qkv_rmsnorm_rope_bf16() -> QkvCase:
    """Mixed prefill/decode batch of 8192 new tokens: 4 prefill chunks of 1984
    tokens after 4096 cached ones, then 256 decode requests with 16..1023 cached
    tokens; 32 q, 8 k, 8 v heads of 128; bf16; 16-token KV blocks; seed 5."""
    ctx_dec = uniform_int(stream_seed(5, 3), 256, 16, 1024).tolist()
    query_lens = [1984] * 4 + [1] * 256
    context_lens = [4096] * 4 + ctx_dec
    return qkv_case("qkv_rmsnorm_rope_bf16_8192tok_32q8k8v_h128", 5, query_lens, context_lens, 32, 8, 8, 128,
                    16, torch.bfloat16)
