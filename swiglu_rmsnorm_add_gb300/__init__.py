"""GB300-native fused per-token decoder path: RMSNorm, residual-add + RMSNorm,
RoPE (neox or interleaved) with paged KV-cache store, SwiGLU / ReGLU, UClip / DyHT,
the decode-attention read of the paged cache, and RMSNorm / GLU fused into the
projection they feed.

Every operator runs in the hand-written sm_103a CUDA kernels of ``libsra.so``
(C ABI in ``include/sra.h``). This module only marshals torch tensors into that
ABI: pointers, sizes, strides, dtype code and the current CUDA stream. There is
no CPU or PyTorch fallback: without the built library every call raises.
"""
from ._binding import (  # noqa: F401
    SRAError,
    add_rmsnorm,
    decode_attention_workspace,
    dyht,
    force_variant,
    glu,
    glu_linear,
    lib,
    linear_workspace,
    paged_decode_attention,
    paged_decode_attention_noalloc,
    pick_variant,
    reglu,
    rmsnorm,
    rmsnorm_linear,
    rope_kv_store,
    set_pdl,
    status_string,
    swiglu,
    uclip,
    variant_count,
    variant_name,
    wait_selftest,
    wait_timeouts,
)

__all__ = ["rmsnorm", "add_rmsnorm", "rope_kv_store", "swiglu", "reglu", "glu", "uclip", "dyht", "paged_decode_attention",
           "paged_decode_attention_noalloc", "decode_attention_workspace",
           "rmsnorm_linear", "glu_linear", "linear_workspace", "lib",
           "SRAError",
           "force_variant", "set_pdl", "variant_count", "variant_name", "pick_variant", "status_string",
           "wait_timeouts", "wait_selftest"]
