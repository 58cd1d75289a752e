"""GB300-native fused QK-prep for the MiniMax-H3 video VAE decoder and DiT
attention: per-head RMSNorm of Q and K, partial multi-axis RoPE, the permute
of the packed QKV projection to head-major Q/K/V, and an optional per-tensor
e4m3 cast (dynamic or static scales, valid-prefix mask).

The path is libh3qk.so (hand-written sm_103a CUDA behind the C-ABI in
include/h3qk.h); ``prepare`` is its thin Python binding, and
``prepare_sage`` writes the float32 Q / K and float16 V a sage attention
kernel reads, and ``prepare_host`` runs the path on host tensors with the
transfers overlapped.  The library also
carries the two adjacent streaming operations of the decoder block
(``silu_and_mul``, ``scaled_residual``).
"""
from .h3qk import (H3QKError, amax, cast, norm_rope_tensor, prepare,  # noqa: F401
                   prepare_dynamic_sharded, prepare_host, prepare_sage, scaled_residual, silu_and_mul)

__all__ = ["prepare", "prepare_host", "prepare_sage", "norm_rope_tensor", "amax", "cast", "prepare_dynamic_sharded",
           "silu_and_mul", "scaled_residual", "H3QKError"]
