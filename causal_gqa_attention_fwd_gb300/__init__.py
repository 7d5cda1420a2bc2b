"""Causal grouped-query attention (forward and backward) for GB300 (sm_103a).

The public entry points mirror the C ABI of include/gqa_attn.h and take
PyTorch CUDA tensors (PyTorch supplies device memory and the stream):

    attn_fwd(q, k, v, causal=True, scale=None) -> (o, lse)
    attn_fwd_rope(q, k, v, rope_cos_sin, causal=True, scale=None) -> (o, lse), q and k rotated
    attn_varlen_fwd_rope(q, k, v, cu_seqlens, max_seqlen, rope_cos_sin, ...) -> (o, lse)
    attn_bwd(q, k, v, o, lse, dout, causal=True, scale=None) -> (dq, dk, dv)
    attn_bwd_rope(q, k, v, o, lse, dout, rope_cos_sin, ...) -> (dq, dk, dv), the backward of attn_fwd_rope
    attn_varlen_bwd_rope(q, k, v, o, lse, dout, cu_seqlens, max_seqlen, rope_cos_sin, ...) -> (dq, dk, dv)
    attn_varlen_fwd(q, k, v, cu_seqlens, max_seqlen, ...) -> (o, lse)
    attn_varlen_bwd(q, k, v, o, lse, dout, cu_seqlens, max_seqlen, ...) -> (dq, dk, dv)
    attn_decode_fwd(q, k_cache, v_cache, cache_lens, scale=None) -> (o, lse)
    attn_decode_paged_fwd(q, k_pages, v_pages, block_table, cache_lens, scale=None) -> (o, lse)
    attn_decode_fp8_fwd / attn_decode_paged_fp8_fwd: the same over E4M3 caches with per-tensor scales

All arithmetic runs in the library's hand-written sm_103a kernels; a call
raises if the library is not built.
"""
from ._binding import (  # noqa: F401
    LIB_PATH,
    AttnError,
    attn_bwd,
    attn_bwd_noalloc,
    attn_bwd_rope,
    attn_bwd_rope_workspace_size,
    attn_bwd_workspace_size,
    attn_decode_fp8_fwd,
    attn_decode_fwd,
    attn_decode_paged_fp8_fwd,
    attn_decode_paged_fwd,
    attn_decode_workspace_size,
    attn_fwd,
    attn_fwd_rope,
    attn_fwd_rope_workspace_size,
    attn_varlen_fwd_rope,
    attn_varlen_fwd_rope_workspace_size,
    attn_varlen_bwd,
    attn_varlen_bwd_rope,
    attn_varlen_bwd_rope_workspace_size,
    attn_varlen_bwd_workspace_size,
    attn_varlen_fwd,
    get_check_line,
    get_device_status,
    lib,
    profile_enable,
    profile_read,
    profile_reset,
    status_string,
)
