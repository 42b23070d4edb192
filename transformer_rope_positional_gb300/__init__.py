"""GB300-native rotary position embedding.

Two operators behind a C ABI (``include/rope_gb300.h``), implemented as
hand-written CUDA kernels for sm_103a:

* ``rope_inplace_partial`` -- in-place partial-slice interleave RoPE of a BSND
  tensor, with fp32 cos/sin allowed for fp16/bf16 x;
* ``rope_with_sin_cos_cache`` -- cos/sin-cache-indexed RoPE of query and key,
  rope or mrope mode, GPT-NeoX or GPT-J style, pass-through columns untouched.

PyTorch supplies device memory and streams only.
"""
from ._capi import (  # noqa: F401
    ROPE_DEVICE_POSITION_OUT_OF_RANGE,
    ROPE_ERR_CUDA,
    ROPE_ERR_PARAM_INVALID,
    ROPE_ERR_PARAM_NULLPTR,
    ROPE_OK,
    RopeError,
    get_device_error,
    launch_count,
    PreparedCall,
    load,
    prepare_inplace_partial,
    prepare_with_sin_cos_cache,
    rope_inplace_partial,
    rope_inplace_partial_backward,
    rope_with_sin_cos_cache,
    qkv_rmsnorm_rope_cache,
    prepare_qkv_rmsnorm_rope_cache,
    ROPE_DEVICE_SLOT_OUT_OF_RANGE,
    ROPE_DEVICE_INDEX_OUT_OF_BOUNDS,
    status_string,
)

from .autograd import inplace_partial_rotary_mul  # noqa: E402,F401

__all__ = [
    "inplace_partial_rotary_mul",
    "rope_inplace_partial",
    "rope_inplace_partial_backward",
    "rope_with_sin_cos_cache",
    "qkv_rmsnorm_rope_cache",
    "get_device_error",
    "launch_count",
    "status_string",
    "load",
    "RopeError",
]
