"""ctypes binding of ``librope_gb300.so`` (see ``include/rope_gb300.h``).

Argument marshalling only: every step of both operators runs in the CUDA
library.  The library must have been built (``python -m
transformer_rope_positional_gb300.build``); there is no fallback, and calling
an operator without it raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# ROPE_GB300_DEBUG_BOUNDS=1 selects the bounds-checking debug build (see build.py)
DEBUG_BOUNDS = os.environ.get("ROPE_GB300_DEBUG_BOUNDS", "0") not in ("", "0")
LIB_PATH = os.path.join(_HERE, "lib", "librope_gb300_debug.so" if DEBUG_BOUNDS else "librope_gb300.so")

F32, F16, BF16, I64 = 0, 1, 2, 3
DTYPE_CODE = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16, torch.int64: I64}

ROPE_OK = 0
ROPE_ERR_PARAM_NULLPTR = 161001
ROPE_ERR_PARAM_INVALID = 161002
ROPE_ERR_CUDA = 561000
ROPE_DEVICE_POSITION_OUT_OF_RANGE = 1
ROPE_DEVICE_SLOT_OUT_OF_RANGE = 2
ROPE_DEVICE_INDEX_OUT_OF_BOUNDS = 4

EXPORTED = ("rope_inplace_partial", "rope_inplace_partial_backward", "rope_with_sin_cos_cache",
            "rope_with_sin_cos_cache_v2", "rope_qkv_rmsnorm_rope_cache", "rope_get_device_error",
            "rope_status_string", "rope_launch_count", "rope_abi_version")


class RopeTensor(ctypes.Structure):
    """Mirror of ``rope_tensor_t``."""
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4)]


class RopeError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__("%s failed with status %d (%s)" % (what, status, status_string(status)))
        self.status = status


_lib = None


def load() -> ctypes.CDLL:
    """Load the shared library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("%s is not built; run `python -m transformer_rope_positional_gb300.build%s`"
                           % (LIB_PATH, " --debug" if DEBUG_BOUNDS else ""))
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER(RopeTensor)
    lib.rope_inplace_partial.argtypes = [P, P, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_void_p]
    lib.rope_inplace_partial.restype = ctypes.c_int
    lib.rope_inplace_partial_backward.argtypes = lib.rope_inplace_partial.argtypes
    lib.rope_inplace_partial_backward.restype = ctypes.c_int
    lib.rope_with_sin_cos_cache.argtypes = [P, P, P, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                            ctypes.POINTER(ctypes.c_int64), ctypes.c_int64, ctypes.c_void_p]
    lib.rope_with_sin_cos_cache.restype = ctypes.c_int
    lib.rope_with_sin_cos_cache_v2.argtypes = [P, P, P, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                               ctypes.POINTER(ctypes.c_int64), ctypes.c_int64, ctypes.c_int32,
                                               ctypes.c_int64, ctypes.c_int64, P, P, ctypes.c_void_p]
    lib.rope_with_sin_cos_cache_v2.restype = ctypes.c_int
    lib.rope_qkv_rmsnorm_rope_cache.argtypes = [P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, P, P,
                                                ctypes.c_float, P, P, P, P, P, P, P, ctypes.c_void_p]
    lib.rope_qkv_rmsnorm_rope_cache.restype = ctypes.c_int
    lib.rope_get_device_error.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)]
    lib.rope_get_device_error.restype = ctypes.c_int
    lib.rope_status_string.argtypes = [ctypes.c_int]
    lib.rope_status_string.restype = ctypes.c_char_p
    lib.rope_launch_count.argtypes = []
    lib.rope_launch_count.restype = ctypes.c_uint64
    lib.rope_abi_version.argtypes = []
    lib.rope_abi_version.restype = ctypes.c_int
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().rope_status_string(int(status)).decode()


_Shape4 = ctypes.c_int64 * 4


def describe(data_ptr: int, dtype_code: int, shape: Sequence[int]) -> RopeTensor:
    """A ``rope_tensor_t`` from a raw device pointer (no checks here)."""
    return RopeTensor(data_ptr or None, dtype_code, len(shape), _Shape4(*shape))


def tensor_desc(t: torch.Tensor) -> RopeTensor:
    """Describe a contiguous CUDA tensor."""
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor, got one on %s" % t.device)
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    if t.dtype not in DTYPE_CODE:
        raise ValueError("unsupported dtype %s" % t.dtype)
    return describe(t.data_ptr(), DTYPE_CODE[t.dtype], tuple(t.shape))


def rows_desc(t: torch.Tensor):
    """Describe a 2-D CUDA tensor whose rows may be strided (unit column
    stride); returns (descriptor, row stride in elements).

    Rows must not overlap: a view whose row stride is below its row width
    (e.g. ``expand`` of one row, stride 0) is refused, since the operator
    writes every row.  A tensor of at most one row gets its width as stride."""
    if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1):
        raise ValueError("expected a 2-D tensor with contiguous rows")
    width = int(t.shape[1])
    stride = int(t.stride(0)) if t.shape[0] > 1 else width
    if stride < width:
        raise ValueError("rows overlap: row stride %d is below the row width %d" % (stride, width))
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor, got one on %s" % t.device)
    if t.dtype not in DTYPE_CODE:
        raise ValueError("unsupported dtype %s" % t.dtype)
    return describe(t.data_ptr(), DTYPE_CODE[t.dtype], tuple(t.shape)), stride


def _one_device(*tensors) -> int:
    """Index of the CUDA device that holds every given tensor (None entries
    skipped); raises if they are spread over several devices."""
    dev = None
    for t in tensors:
        if t is None:
            continue
        d = t.get_device()
        if dev is None:
            dev = d
        elif d != dev:
            raise ValueError("tensors on different devices (cuda:%d and cuda:%d)" % (dev, d))
    return dev


# the current device without the public call's lazy-initialisation check (CUDA
# is initialised once CUDA tensors exist); the public call is the fallback
_current_device = getattr(torch._C, "_cuda_getDevice", None) or torch.cuda.current_device


def _on_device(dev: int, fn, args):
    """Call fn(*args) with device ``dev`` current (the library launches on the
    current device and sizes its grid from it)."""
    if dev is None or dev < 0 or _current_device() == dev:
        return fn(*args)
    with torch.cuda.device(dev):
        return fn(*args)


# the current stream's raw handle without building a Stream object (about 10x
# cheaper per call); the public call is the fallback
_raw_current_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_handle(t: torch.Tensor, stream) -> int:
    if stream is None:
        if _raw_current_stream is not None:
            return _raw_current_stream(t.get_device())
        return torch.cuda.current_stream(t.device).cuda_stream
    if hasattr(stream, "device") and stream.device.index != t.get_device():
        raise ValueError("stream of %s for tensors on cuda:%d" % (stream.device, t.get_device()))
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


MODES = {"interleave": 1, "half": 0, 1: 1, 0: 0}


def _mode(rotary_mode) -> int:
    if rotary_mode not in MODES:
        raise RopeError(ROPE_ERR_PARAM_INVALID, "rotary_mode %r" % (rotary_mode,))
    return MODES[rotary_mode]


def _slice(partial_slice):
    if partial_slice is None:
        return 0, 0
    if len(partial_slice) != 2:
        raise RopeError(ROPE_ERR_PARAM_INVALID, "partial_slice must have two elements")
    return int(partial_slice[0]), int(partial_slice[1])


def _inplace_args(x, cos, sin, rotary_mode, partial_slice, stream, backward):
    """(C function, its arguments, objects to keep alive, name) of one call."""
    lib = load()
    start, end = _slice(partial_slice)
    _one_device(x, cos, sin)
    dx, dc, ds = tensor_desc(x), tensor_desc(cos), tensor_desc(sin)
    args = (ctypes.byref(dx), ctypes.byref(dc), ctypes.byref(ds), _mode(rotary_mode), start, end,
            _stream_handle(x, stream))
    if backward:
        return lib.rope_inplace_partial_backward, args, (x, cos, sin, dx, dc, ds), "rope_inplace_partial_backward"
    return lib.rope_inplace_partial, args, (x, cos, sin, dx, dc, ds), "rope_inplace_partial"


def _run(fn, args, keep, what) -> None:
    st = _on_device(keep[0].get_device(), fn, args)
    if st != ROPE_OK:
        raise RopeError(st, what)


def rope_inplace_partial(x: torch.Tensor, cos: torch.Tensor, sin: torch.Tensor, rotary_mode=1,
                         partial_slice: Optional[Sequence[int]] = None, stream=None) -> None:
    """In-place partial RoPE of ``x`` [B, S, N, D] over ``partial_slice``.

    ``rotary_mode``: 1 / "interleave" or 0 / "half".  ``partial_slice=None``
    means ``[0, 0]``, the whole D axis.  Returns None; x is rewritten on
    ``stream`` (default: the current stream of x's device).
    """
    _run(*_inplace_args(x, cos, sin, rotary_mode, partial_slice, stream, False))


def rope_inplace_partial_backward(grad: torch.Tensor, cos: torch.Tensor, sin: torch.Tensor, rotary_mode=1,
                                  partial_slice: Optional[Sequence[int]] = None, stream=None) -> None:
    """Backward of :func:`rope_inplace_partial`: turns dL/dy in ``grad`` into
    dL/dx in place."""
    _run(*_inplace_args(grad, cos, sin, rotary_mode, partial_slice, stream, True))


def rope_with_sin_cos_cache(positions: torch.Tensor, query: torch.Tensor, key: torch.Tensor,
                            cos_sin_cache: torch.Tensor, head_size: int, rotary_dim: Optional[int] = None,
                            is_neox: bool = True, mrope_section: Optional[Sequence[int]] = None,
                            stream=None, *, cache_mode: int = 0, query_out: Optional[torch.Tensor] = None,
                            key_out: Optional[torch.Tensor] = None) -> None:
    """Cache-indexed RoPE of ``query`` and ``key`` (rope or mrope mode).

    In place unless ``query_out``/``key_out`` are given.  ``query``/``key`` may
    be strided row views (e.g. slices of a fused QKV tensor); ``cache_mode=1``
    selects the interleaved mrope splice.  Contiguous in-place calls with
    ``cache_mode=0`` use the V1 entry point, everything else the V2 one."""
    _run(*_cache_args(positions, query, key, cos_sin_cache, head_size, rotary_dim, is_neox, mrope_section, stream,
                      cache_mode, query_out, key_out))


def _cache_args(positions, query, key, cos_sin_cache, head_size, rotary_dim, is_neox, mrope_section, stream,
                cache_mode, query_out, key_out):
    """(C function, its arguments, objects to keep alive, name) of one
    cache-operator call: the V1 entry point for a contiguous in-place call with
    cache_mode 0, else V2."""
    lib = load()
    R = int(cos_sin_cache.shape[1]) if rotary_dim is None else int(rotary_dim)
    _one_device(query, key, positions, cos_sin_cache, query_out, key_out)
    dq, qs = rows_desc(query)
    dk, ks = rows_desc(key)
    dp, dc = tensor_desc(positions), tensor_desc(cos_sin_cache)
    sec = None
    n_sec = 0
    if mrope_section is not None:
        n_sec = len(mrope_section)
        sec = (ctypes.c_int64 * max(1, n_sec))(*[int(v) for v in mrope_section])
    handle = _stream_handle(query, stream)
    contiguous = qs == query.shape[1] and ks == key.shape[1]
    if cache_mode == 0 and query_out is None and key_out is None and contiguous:
        args = (ctypes.byref(dp), ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dc), int(head_size), R,
                1 if is_neox else 0, sec, n_sec, handle)
        return (lib.rope_with_sin_cos_cache, args, (positions, query, key, cos_sin_cache, dp, dq, dk, dc, sec),
                "rope_with_sin_cos_cache")
    dqo = tensor_desc(query_out) if query_out is not None else None
    dko = tensor_desc(key_out) if key_out is not None else None
    args = (ctypes.byref(dp), ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dc), int(head_size), R,
            1 if is_neox else 0, sec, n_sec, int(cache_mode), qs, ks,
            ctypes.byref(dqo) if dqo is not None else None, ctypes.byref(dko) if dko is not None else None, handle)
    return (lib.rope_with_sin_cos_cache_v2, args,
            (positions, query, key, cos_sin_cache, query_out, key_out, dp, dq, dk, dc, dqo, dko, sec),
            "rope_with_sin_cos_cache_v2")


def _qkv_args(qkv, num_q_heads, num_k_heads, num_v_heads, q_gamma, k_gamma, eps, cos_sin_cache, seq_lens,
              query_start_loc, slot_mapping, q_out, k_cache, v_cache, stream):
    tensors = (qkv, q_gamma, k_gamma, cos_sin_cache, seq_lens, query_start_loc, slot_mapping, q_out, k_cache,
               v_cache)
    _one_device(*tensors)
    descs = [tensor_desc(t) for t in tensors]
    r = [ctypes.byref(d) for d in descs]
    args = (r[0], int(num_q_heads), int(num_k_heads), int(num_v_heads), r[1], r[2], float(eps), r[3], r[4], r[5],
            r[6], r[7], r[8], r[9], _stream_handle(qkv, stream))
    return args, descs


def qkv_rmsnorm_rope_cache(qkv: torch.Tensor, num_q_heads: int, num_k_heads: int, num_v_heads: int,
                           q_gamma: torch.Tensor, k_gamma: torch.Tensor, eps: float, cos_sin_cache: torch.Tensor,
                           seq_lens: torch.Tensor, query_start_loc: torch.Tensor, slot_mapping: torch.Tensor,
                           q_out: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, stream=None) -> None:
    """Fused QKV split + RMSNorm + RoPE + paged KV-cache write (see the C header)."""
    lib = load()
    args, _ = _qkv_args(qkv, num_q_heads, num_k_heads, num_v_heads, q_gamma, k_gamma, eps, cos_sin_cache,
                        seq_lens, query_start_loc, slot_mapping, q_out, k_cache, v_cache, stream)
    _run(lib.rope_qkv_rmsnorm_rope_cache, args, (qkv,), "rope_qkv_rmsnorm_rope_cache")


def prepare_qkv_rmsnorm_rope_cache(qkv: torch.Tensor, num_q_heads: int, num_k_heads: int, num_v_heads: int,
                                   q_gamma: torch.Tensor, k_gamma: torch.Tensor, eps: float,
                                   cos_sin_cache: torch.Tensor, seq_lens: torch.Tensor,
                                   query_start_loc: torch.Tensor, slot_mapping: torch.Tensor, q_out: torch.Tensor,
                                   k_cache: torch.Tensor, v_cache: torch.Tensor, stream=None) -> "PreparedCall":
    """:func:`qkv_rmsnorm_rope_cache` with its arguments marshalled once."""
    lib = load()
    tensors = (qkv, q_gamma, k_gamma, cos_sin_cache, seq_lens, query_start_loc, slot_mapping, q_out, k_cache,
               v_cache)
    args, descs = _qkv_args(qkv, num_q_heads, num_k_heads, num_v_heads, q_gamma, k_gamma, eps, cos_sin_cache,
                            seq_lens, query_start_loc, slot_mapping, q_out, k_cache, v_cache, stream)
    return PreparedCall(lib.rope_qkv_rmsnorm_rope_cache, args, (tensors, descs), "rope_qkv_rmsnorm_rope_cache")


def get_device_error(stream=None, device=None) -> int:
    """Synchronise ``stream`` and read-and-clear the error word of its device
    (``device``, else the stream's device, else the current device)."""
    lib = load()
    if device is None and stream is not None and hasattr(stream, "device"):
        device = stream.device
    dev = device if isinstance(device, int) else torch.device(device).index if device is not None else None
    if dev is None:
        dev = torch.cuda.current_device()
    with torch.cuda.device(dev):
        if stream is None:
            stream = torch.cuda.current_stream(dev)
        handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        code = ctypes.c_int32(0)
        st = lib.rope_get_device_error(handle, ctypes.byref(code))
    if st != ROPE_OK:
        raise RopeError(st, "rope_get_device_error")
    return int(code.value)


def launch_count() -> int:
    return int(load().rope_launch_count())


class PreparedCall:
    """One operator call with its C arguments marshalled once.

    Calling it re-issues the same launch on the same tensors and the same
    stream (the one given, or the current one, when it was prepared), for
    loops that apply the operator many times; it keeps the tensors alive.
    """

    def __init__(self, fn, args, keep, what):
        self._fn = fn
        self._args = args
        self._keep = keep
        self._what = what
        first = keep[0]
        while isinstance(first, (tuple, list)):
            first = first[0]
        self._device = first.get_device()

    def __call__(self) -> None:
        st = _on_device(self._device, self._fn, self._args)
        if st != ROPE_OK:
            raise RopeError(st, self._what)


def prepare_inplace_partial(x: torch.Tensor, cos: torch.Tensor, sin: torch.Tensor, rotary_mode=1,
                            partial_slice: Optional[Sequence[int]] = None, stream=None,
                            backward: bool = False) -> PreparedCall:
    """:func:`rope_inplace_partial` (or its backward) with its arguments marshalled once."""
    return PreparedCall(*_inplace_args(x, cos, sin, rotary_mode, partial_slice, stream, backward))


def prepare_with_sin_cos_cache(positions: torch.Tensor, query: torch.Tensor, key: torch.Tensor,
                               cos_sin_cache: torch.Tensor, head_size: int, rotary_dim: Optional[int] = None,
                               is_neox: bool = True, mrope_section: Optional[Sequence[int]] = None,
                               stream=None, *, cache_mode: int = 0, query_out: Optional[torch.Tensor] = None,
                               key_out: Optional[torch.Tensor] = None) -> PreparedCall:
    """:func:`rope_with_sin_cos_cache` with its arguments marshalled once."""
    return PreparedCall(*_cache_args(positions, query, key, cos_sin_cache, head_size, rotary_dim, is_neox,
                                     mrope_section, stream, cache_mode, query_out, key_out))
