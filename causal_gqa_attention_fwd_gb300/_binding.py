"""ctypes binding of libgqa_attn.so (include/gqa_attn.h).

Argument marshalling only: shape/dtype checks, output allocation with torch
(device memory is PyTorch's), the current CUDA stream, and the C call.  Every
step of the attention runs in the library's CUDA kernels; there is no other
code path.  Importing this module does not load the library; the first call
does, and raises if the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libgqa_attn.so")
DEBUG_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libgqa_attn_debug.so")

STATUS = {
    0: "ATTN_OK", 1: "ATTN_ERR_NULL", 2: "ATTN_ERR_SHAPE", 3: "ATTN_ERR_HEADDIM", 4: "ATTN_ERR_ALIGN",
    5: "ATTN_ERR_SEQLENS", 6: "ATTN_ERR_WORKSPACE", 7: "ATTN_ERR_ARCH", 8: "ATTN_ERR_CUDA",
    9: "ATTN_ERR_TIMEOUT", 10: "ATTN_ERR_SCRATCH_LIMIT", 11: "ATTN_ERR_PAGES", 12: "ATTN_ERR_CHECK",
    13: "ATTN_ERR_RANGE",
}

# name -> (restype, argtypes)
_P, _I, _F, _Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "attn_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P]),
    "attn_fwd_rope_workspace_size": (_Z, [_I, _I, _I, _I, _I]),
    "attn_fwd_rope": (_I, [_P, _P, _P, _P, _P, _P, _Z, _I, _I, _I, _I, _I, _I, _F, _P, _I, _P]),
    "attn_varlen_fwd_rope_workspace_size": (_Z, [_I, _I, _I, _I]),
    "attn_varlen_fwd_rope": (_I, [_P] * 6 + [_I] * 7 + [_F, _P, _I, _P, _Z, _P]),
    "attn_bwd_workspace_size": (_Z, [_I, _I, _I, _I, _I]),
    "attn_bwd_rope_workspace_size": (_Z, [_I, _I, _I, _I, _I]),
    "attn_bwd_rope": (_I, [_P] * 10 + [_Z, _I, _I, _I, _I, _I, _I, _F, _P, _I, _P]),
    "attn_varlen_bwd_rope_workspace_size": (_Z, [_I, _I, _I, _I, _I]),
    "attn_varlen_bwd_rope": (_I, [_P] * 10 + [_Z, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _I, _P]),
    "attn_bwd": (_I, [_P] * 10 + [_Z, _I, _I, _I, _I, _I, _I, _F, _P]),
    "attn_varlen_fwd": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P]),
    "attn_varlen_bwd_workspace_size": (_Z, [_I, _I, _I, _I, _I]),
    "attn_varlen_bwd": (_I, [_P] * 10 + [_Z, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P]),
    "attn_status_string": (ctypes.c_char_p, [_I]),
    "attn_get_device_status": (_I, [_P, ctypes.POINTER(_I), _I]),
    "attn_get_check_line": (_I, [_P, ctypes.POINTER(_I), _I]),
    "attn_is_debug_build": (_I, []),
    "attn_bwd_noalloc": (_I, [_P] * 9 + [_I, _I, _I, _I, _I, _I, _F, _P]),
    "attn_bwd_noalloc_scratch_bytes": (_Z, []),
    "attn_selftest_wait_timeout": (_I, [_I, _P]),
    "attn_test_inject_timeout": (_I, [_I, _I]),
    "attn_profile_enable": (_I, [_I]),
    "attn_profile_reset": (_I, []),
    "attn_profile_read": (_I, [_I, ctypes.POINTER(_I), ctypes.POINTER(ctypes.c_double)]),
    "attn_decode_workspace_size": (_Z, [_I, _I, _I, _I, _I, _I]),
    "attn_decode_fwd": (_I, [_P] * 7 + [_Z, _I, _I, _I, _I, _I, _I, _F, _P, _I, _P]),
    "attn_decode_paged_fwd": (_I, [_P] * 8 + [_Z] + [_I] * 8 + [_F, _P, _I, _P]),
    "attn_decode_fp8_fwd": (_I, [_P, _P, _P, _F, _F] + [_P] * 4 + [_Z] + [_I] * 6 + [_F, _P, _I, _P]),
    "attn_decode_paged_fp8_fwd": (_I, [_P, _P, _P, _F, _F] + [_P] * 5 + [_Z] + [_I] * 8 + [_F, _P, _I, _P]),
}

PROFILE_KINDS = {"attn_fwd": 0, "bwd_pre": 1, "bwd_dkdv": 2, "decode": 4, "decode_merge": 5, "bwd_dq": 6}

_lib = None


class AttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)} ({status_string(code) if _lib else ''})")


def lib():
    """The loaded ctypes library (raises if it is not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with causal_gqa_attention_fwd_gb300.build.build() "
                "(nvcc, sm_103a). There is no fallback implementation.")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name, None)
            if fn is None:      # reported by the export test; calls raise AttributeError
                continue
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def status_string(code: int) -> str:
    return lib().attn_status_string(int(code)).decode()


def _check(code: int, where: str):
    if code != 0:
        raise AttnError(code, where)


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _need(t: torch.Tensor, name: str, dtype=torch.bfloat16):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _scale(scale, D):
    return float(scale) if scale is not None else 1.0 / float(D) ** 0.5


def get_check_line(clear: bool = True, stream=None) -> int:
    """Debug build: synchronise and return (and clear) the source line of the first failed bounds check."""
    out = ctypes.c_int(0)
    _check(lib().attn_get_check_line(_stream(stream), ctypes.byref(out), int(clear)), "attn_get_check_line")
    return out.value


def get_device_status(clear: bool = True, stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status word."""
    out = ctypes.c_int(0)
    _check(lib().attn_get_device_status(_stream(stream), ctypes.byref(out), int(clear)), "attn_get_device_status")
    return out.value


def profile_enable(on: bool = True):
    """Record CUDA events around every kernel launch (see attn_profile_read)."""
    _check(lib().attn_profile_enable(int(on)), "attn_profile_enable")


def profile_reset():
    _check(lib().attn_profile_reset(), "attn_profile_reset")


def profile_read() -> dict:
    """{kernel: (launches, total_ms)} since the last reset (synchronises)."""
    out = {}
    for name, kind in PROFILE_KINDS.items():
        n = ctypes.c_int(0)
        ms = ctypes.c_double(0.0)
        _check(lib().attn_profile_read(kind, ctypes.byref(n), ctypes.byref(ms)), "attn_profile_read")
        out[name] = (n.value, ms.value)
    return out


def attn_fwd(q, k, v, causal: bool = True, scale=None, o=None, lse=None, stream=None):
    """Dense forward.  q [B,Hq,T,D], k/v [B,Hkv,T,D] bf16 -> (o bf16, lse f32 [B,Hq,T])."""
    B, Hq, T, D = q.shape
    Hkv = k.shape[1]
    if k.shape != (B, Hkv, T, D) or v.shape != k.shape:
        raise ValueError("k, v must be [B, Hkv, T, D] matching q")
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, Hq, T), dtype=torch.float32, device=q.device) if lse is None else lse
    st = lib().attn_fwd(_need(q, "q"), _need(k, "k"), _need(v, "v"), _need(o, "o"),
                        _need(lse, "lse", torch.float32), B, Hq, Hkv, T, D, int(causal), _scale(scale, D),
                        _stream(stream))
    _check(st, "attn_fwd")
    return o, lse


def attn_fwd_rope_workspace_size(B, Hq, Hkv, T, D) -> int:
    return int(lib().attn_fwd_rope_workspace_size(B, Hq, Hkv, T, D))


def attn_fwd_rope(q, k, v, rope_cos_sin, causal: bool = True, scale=None, o=None, lse=None, workspace=None,
                  stream=None):
    """Dense forward with q and k rotated at positions 0..T-1 (rotary table rope_cos_sin float32
    [>= T, D] on the device, as attn_decode_fwd) -> (o bf16, lse f32 [B,Hq,T])."""
    B, Hq, T, D = q.shape
    Hkv = k.shape[1]
    if k.shape != (B, Hkv, T, D) or v.shape != k.shape:
        raise ValueError("k, v must be [B, Hkv, T, D] matching q")
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, Hq, T), dtype=torch.float32, device=q.device) if lse is None else lse
    if workspace is None:
        workspace = torch.empty(max(attn_fwd_rope_workspace_size(B, Hq, Hkv, T, D), 256), dtype=torch.uint8,
                                device=q.device)
    rope_ptr, rope_n = _rope(rope_cos_sin)
    st = lib().attn_fwd_rope(_need(q, "q"), _need(k, "k"), _need(v, "v"), _need(o, "o"),
                             _need(lse, "lse", torch.float32), _need(workspace, "workspace", torch.uint8),
                             workspace.numel(), B, Hq, Hkv, T, D, int(causal), _scale(scale, D), rope_ptr, rope_n,
                             _stream(stream))
    _check(st, "attn_fwd_rope")
    return o, lse


def attn_varlen_fwd_rope(q, k, v, cu_seqlens, max_seqlen, rope_cos_sin, causal: bool = True, scale=None, o=None,
                         lse=None, workspace=None, stream=None):
    """Packed variable-length forward with q and k rotated at their offsets in their sequences
    (positions 0..len-1; rotary table as attn_fwd_rope) -> (o, lse [Hq,total])."""
    total, Hq, D = q.shape
    Hkv = k.shape[1]
    if k.shape != (total, Hkv, D) or v.shape != k.shape:
        raise ValueError("k, v must be [total, Hkv, D] matching q")
    num_seqs = cu_seqlens.numel() - 1
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((Hq, total), dtype=torch.float32, device=q.device) if lse is None else lse
    if workspace is None:
        workspace = torch.empty(max(attn_varlen_fwd_rope_workspace_size(total, Hq, Hkv, D), 256),
                                dtype=torch.uint8, device=q.device)
    rope_ptr, rope_n = _rope(rope_cos_sin)
    st = lib().attn_varlen_fwd_rope(_need(q, "q"), _need(k, "k"), _need(v, "v"), _need(o, "o"),
                                    _need(lse, "lse", torch.float32), _need(cu_seqlens, "cu_seqlens", torch.int32),
                                    num_seqs, total, int(max_seqlen), Hq, Hkv, D, int(causal), _scale(scale, D),
                                    rope_ptr, rope_n, _need(workspace, "workspace", torch.uint8), workspace.numel(),
                                    _stream(stream))
    _check(st, "attn_varlen_fwd_rope")
    return o, lse


def attn_varlen_fwd_rope_workspace_size(total, Hq, Hkv, D) -> int:
    return int(lib().attn_varlen_fwd_rope_workspace_size(total, Hq, Hkv, D))


def attn_bwd_workspace_size(B, Hq, Hkv, T, D) -> int:
    return int(lib().attn_bwd_workspace_size(B, Hq, Hkv, T, D))


def attn_bwd_rope_workspace_size(B, Hq, Hkv, T, D) -> int:
    return int(lib().attn_bwd_rope_workspace_size(B, Hq, Hkv, T, D))


def attn_varlen_bwd_rope_workspace_size(num_seqs, total, Hq, Hkv, D) -> int:
    return int(lib().attn_varlen_bwd_rope_workspace_size(num_seqs, total, Hq, Hkv, D))


def attn_bwd(q, k, v, o, lse, dout, causal: bool = True, scale=None, dq=None, dk=None, dv=None,
             workspace=None, stream=None):
    """Dense backward -> (dq, dk, dv) bf16."""
    B, Hq, T, D = q.shape
    Hkv = k.shape[1]
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws_bytes = attn_bwd_workspace_size(B, Hq, Hkv, T, D)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
    st = lib().attn_bwd(_need(q, "q"), _need(k, "k"), _need(v, "v"), _need(o, "o"),
                        _need(lse, "lse", torch.float32), _need(dout, "dout"), _need(dq, "dq"), _need(dk, "dk"),
                        _need(dv, "dv"), _need(workspace, "workspace", torch.uint8), workspace.numel(),
                        B, Hq, Hkv, T, D, int(causal), _scale(scale, D), _stream(stream))
    _check(st, "attn_bwd")
    return dq, dk, dv


def attn_bwd_rope(q, k, v, o, lse, dout, rope_cos_sin, causal: bool = True, scale=None, dq=None, dk=None, dv=None,
                  workspace=None, stream=None):
    """Backward of attn_fwd_rope -> (dq, dk, dv) bf16, gradients with respect to the unrotated q, k, v
    (rotary table as attn_fwd_rope; o, lse from attn_fwd_rope)."""
    B, Hq, T, D = q.shape
    Hkv = k.shape[1]
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        workspace = torch.empty(max(attn_bwd_rope_workspace_size(B, Hq, Hkv, T, D), 256),
                                dtype=torch.uint8, device=q.device)
    rope_ptr, rope_n = _rope(rope_cos_sin)
    st = lib().attn_bwd_rope(_need(q, "q"), _need(k, "k"), _need(v, "v"), _need(o, "o"),
                             _need(lse, "lse", torch.float32), _need(dout, "dout"), _need(dq, "dq"), _need(dk, "dk"),
                             _need(dv, "dv"), _need(workspace, "workspace", torch.uint8), workspace.numel(),
                             B, Hq, Hkv, T, D, int(causal), _scale(scale, D), rope_ptr, rope_n, _stream(stream))
    _check(st, "attn_bwd_rope")
    return dq, dk, dv


def attn_varlen_bwd_rope(q, k, v, o, lse, dout, cu_seqlens, max_seqlen: int, rope_cos_sin, causal: bool = True,
                         scale=None, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Backward of attn_varlen_fwd_rope -> (dq, dk, dv)."""
    total, Hq, D = q.shape
    Hkv = k.shape[1]
    n = cu_seqlens.numel() - 1
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        workspace = torch.empty(max(attn_varlen_bwd_rope_workspace_size(n, total, Hq, Hkv, D), 256),
                                dtype=torch.uint8, device=q.device)
    rope_ptr, rope_n = _rope(rope_cos_sin)
    st = lib().attn_varlen_bwd_rope(_need(q, "q"), _need(k, "k"), _need(v, "v"), _need(o, "o"),
                                    _need(lse, "lse", torch.float32), _need(dout, "dout"), _need(dq, "dq"),
                                    _need(dk, "dk"), _need(dv, "dv"), _need(workspace, "workspace", torch.uint8),
                                    workspace.numel(), _need(cu_seqlens, "cu_seqlens", torch.int32), n, total,
                                    int(max_seqlen), Hq, Hkv, D, int(causal), _scale(scale, D), rope_ptr, rope_n,
                                    _stream(stream))
    _check(st, "attn_varlen_bwd_rope")
    return dq, dk, dv


def attn_bwd_noalloc(q, k, v, o, lse, dout, causal: bool = True, scale=None, dq=None, dk=None, dv=None,
                     stream=None):
    """Dense backward through attn_bwd_noalloc: no workspace and no allocation
    inside the library (it uses its built-in scratch array).  Outputs are
    allocated here unless passed in."""
    B, Hq, T, D = q.shape
    Hkv = k.shape[1]
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    st = lib().attn_bwd_noalloc(_need(q, "q"), _need(k, "k"), _need(v, "v"), _need(o, "o"),
                                _need(lse, "lse", torch.float32), _need(dout, "dout"), _need(dq, "dq"),
                                _need(dk, "dk"), _need(dv, "dv"), B, Hq, Hkv, T, D, int(causal), _scale(scale, D),
                                _stream(stream))
    _check(st, "attn_bwd_noalloc")
    return dq, dk, dv


def attn_varlen_fwd(q, k, v, cu_seqlens, max_seqlen: int, causal: bool = True, scale=None, o=None, lse=None,
                    stream=None):
    """Packed forward.  q [total,Hq,D], k/v [total,Hkv,D], cu_seqlens int32 (device) [N+1]
    -> (o [total,Hq,D], lse [Hq,total])."""
    total, Hq, D = q.shape
    Hkv = k.shape[1]
    n = cu_seqlens.numel() - 1
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((Hq, total), dtype=torch.float32, device=q.device) if lse is None else lse
    st = lib().attn_varlen_fwd(_need(q, "q"), _need(k, "k"), _need(v, "v"), _need(o, "o"),
                               _need(lse, "lse", torch.float32), _need(cu_seqlens, "cu_seqlens", torch.int32),
                               n, total, int(max_seqlen), Hq, Hkv, D, int(causal), _scale(scale, D),
                               _stream(stream))
    _check(st, "attn_varlen_fwd")
    return o, lse


def attn_varlen_bwd_workspace_size(num_seqs, total, Hq, Hkv, D) -> int:
    return int(lib().attn_varlen_bwd_workspace_size(num_seqs, total, Hq, Hkv, D))


def attn_varlen_bwd(q, k, v, o, lse, dout, cu_seqlens, max_seqlen: int, causal: bool = True, scale=None,
                    dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Packed backward -> (dq, dk, dv)."""
    total, Hq, D = q.shape
    Hkv = k.shape[1]
    n = cu_seqlens.numel() - 1
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws_bytes = attn_varlen_bwd_workspace_size(n, total, Hq, Hkv, D)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
    st = lib().attn_varlen_bwd(_need(q, "q"), _need(k, "k"), _need(v, "v"), _need(o, "o"),
                               _need(lse, "lse", torch.float32), _need(dout, "dout"), _need(dq, "dq"),
                               _need(dk, "dk"), _need(dv, "dv"), _need(workspace, "workspace", torch.uint8),
                               workspace.numel(), _need(cu_seqlens, "cu_seqlens", torch.int32), n, total,
                               int(max_seqlen), Hq, Hkv, D, int(causal), _scale(scale, D), _stream(stream))
    _check(st, "attn_varlen_bwd")
    return dq, dk, dv


def attn_decode_workspace_size(B, Hq, Hkv, Tq, S, D) -> int:
    return int(lib().attn_decode_workspace_size(B, Hq, Hkv, Tq, S, D))


def _rope(rope_cos_sin):
    if rope_cos_sin is None:
        return None, 0
    return _need(rope_cos_sin, "rope_cos_sin", torch.float32), int(rope_cos_sin.shape[0])


def attn_decode_fwd(q, k_cache, v_cache, cache_lens, scale=None, o=None, lse=None, workspace=None, stream=None,
                    rope_cos_sin=None):
    """Cached (decode) attention.  q [B,Hq,Tq,D]; k_cache, v_cache [B,Hkv,S,D] bf16; cache_lens int32
    (device) [B], keys held per row including the Tq new ones; query t of row b sees keys
    j <= cache_lens[b] - Tq + t -> (o [B,Hq,Tq,D] bf16, lse [B,Hq,Tq] f32).  rope_cos_sin: optional
    float32 (device) [positions, D] rotary table; the queries are rotated at their positions."""
    B, Hq, Tq, D = q.shape
    Hkv, S = k_cache.shape[1], k_cache.shape[2]
    if k_cache.shape != (B, Hkv, S, D) or v_cache.shape != k_cache.shape:
        raise ValueError("k_cache, v_cache must be [B, Hkv, S, D] matching q")
    if cache_lens.shape != (B,):
        raise ValueError("cache_lens must be [B]")
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, Hq, Tq), dtype=torch.float32, device=q.device) if lse is None else lse
    ws_bytes = attn_decode_workspace_size(B, Hq, Hkv, Tq, S, D)
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    ws_ptr = _need(workspace, "workspace", torch.uint8) if workspace is not None else None
    ws_len = workspace.numel() if workspace is not None else 0
    rope_ptr, rope_n = _rope(rope_cos_sin)
    st = lib().attn_decode_fwd(_need(q, "q"), _need(k_cache, "k_cache"), _need(v_cache, "v_cache"),
                               _need(cache_lens, "cache_lens", torch.int32), _need(o, "o"),
                               _need(lse, "lse", torch.float32), ws_ptr, ws_len, B, Hq, Hkv, Tq, S, D,
                               _scale(scale, D), rope_ptr, rope_n, _stream(stream))
    _check(st, "attn_decode_fwd")
    return o, lse


def attn_decode_paged_fwd(q, k_pages, v_pages, block_table, cache_lens, scale=None, o=None, lse=None, workspace=None,
                          stream=None, rope_cos_sin=None):
    """Cached attention over a paged KV cache.  q [B,Hq,Tq,D]; k_pages, v_pages [num_pages,Hkv,page_size,D]
    bf16; block_table int32 (device) [B, max_pages]; cache_lens int32 (device) [B]
    -> (o [B,Hq,Tq,D] bf16, lse [B,Hq,Tq] f32).  rope_cos_sin as attn_decode_fwd."""
    B, Hq, Tq, D = q.shape
    num_pages, Hkv, page_size = k_pages.shape[0], k_pages.shape[1], k_pages.shape[2]
    if k_pages.shape != (num_pages, Hkv, page_size, D) or v_pages.shape != k_pages.shape:
        raise ValueError("k_pages, v_pages must be [num_pages, Hkv, page_size, D] matching q")
    if block_table.dim() != 2 or block_table.shape[0] != B or cache_lens.shape != (B,):
        raise ValueError("block_table must be [B, max_pages], cache_lens [B]")
    max_pages = block_table.shape[1]
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, Hq, Tq), dtype=torch.float32, device=q.device) if lse is None else lse
    ws_bytes = attn_decode_workspace_size(B, Hq, Hkv, Tq, max_pages * page_size, D)
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    ws_ptr = _need(workspace, "workspace", torch.uint8) if workspace is not None else None
    ws_len = workspace.numel() if workspace is not None else 0
    st = lib().attn_decode_paged_fwd(_need(q, "q"), _need(k_pages, "k_pages"), _need(v_pages, "v_pages"),
                                     _need(block_table, "block_table", torch.int32),
                                     _need(cache_lens, "cache_lens", torch.int32), _need(o, "o"),
                                     _need(lse, "lse", torch.float32), ws_ptr, ws_len, B, Hq, Hkv, Tq, page_size,
                                     num_pages, max_pages, D, _scale(scale, D), *_rope(rope_cos_sin), _stream(stream))
    _check(st, "attn_decode_paged_fwd")
    return o, lse


def attn_decode_fp8_fwd(q, k8, v8, k_scale: float, v_scale: float, cache_lens, scale=None, o=None, lse=None,
                        workspace=None, stream=None, rope_cos_sin=None):
    """Cached attention over FP8 (E4M3) caches.  k8, v8 uint8 [B,Hkv,S,D] (E4M3 codes), K = e4m3(k8) * k_scale,
    V = e4m3(v8) * v_scale; everything else as attn_decode_fwd."""
    B, Hq, Tq, D = q.shape
    Hkv, S = k8.shape[1], k8.shape[2]
    if k8.shape != (B, Hkv, S, D) or v8.shape != k8.shape:
        raise ValueError("k8, v8 must be [B, Hkv, S, D] matching q")
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, Hq, Tq), dtype=torch.float32, device=q.device) if lse is None else lse
    ws_bytes = attn_decode_workspace_size(B, Hq, Hkv, Tq, S, D)
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    ws_ptr = _need(workspace, "workspace", torch.uint8) if workspace is not None else None
    ws_len = workspace.numel() if workspace is not None else 0
    st = lib().attn_decode_fp8_fwd(_need(q, "q"), _need(k8, "k8", torch.uint8), _need(v8, "v8", torch.uint8),
                                   float(k_scale), float(v_scale), _need(cache_lens, "cache_lens", torch.int32),
                                   _need(o, "o"), _need(lse, "lse", torch.float32), ws_ptr, ws_len, B, Hq, Hkv, Tq, S,
                                   D, _scale(scale, D), *_rope(rope_cos_sin), _stream(stream))
    _check(st, "attn_decode_fp8_fwd")
    return o, lse


def attn_decode_paged_fp8_fwd(q, k8_pages, v8_pages, k_scale: float, v_scale: float, block_table, cache_lens,
                              scale=None, o=None, lse=None, workspace=None, stream=None, rope_cos_sin=None):
    """Cached attention over paged FP8 (E4M3) caches: k8_pages, v8_pages uint8 [num_pages,Hkv,page_size,D];
    otherwise as attn_decode_paged_fwd and attn_decode_fp8_fwd."""
    B, Hq, Tq, D = q.shape
    num_pages, Hkv, page_size = k8_pages.shape[0], k8_pages.shape[1], k8_pages.shape[2]
    if k8_pages.shape != (num_pages, Hkv, page_size, D) or v8_pages.shape != k8_pages.shape:
        raise ValueError("k8_pages, v8_pages must be [num_pages, Hkv, page_size, D] matching q")
    max_pages = block_table.shape[1]
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, Hq, Tq), dtype=torch.float32, device=q.device) if lse is None else lse
    ws_bytes = attn_decode_workspace_size(B, Hq, Hkv, Tq, max_pages * page_size, D)
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    ws_ptr = _need(workspace, "workspace", torch.uint8) if workspace is not None else None
    ws_len = workspace.numel() if workspace is not None else 0
    st = lib().attn_decode_paged_fp8_fwd(_need(q, "q"), _need(k8_pages, "k8_pages", torch.uint8),
                                         _need(v8_pages, "v8_pages", torch.uint8), float(k_scale), float(v_scale),
                                         _need(block_table, "block_table", torch.int32),
                                         _need(cache_lens, "cache_lens", torch.int32), _need(o, "o"),
                                         _need(lse, "lse", torch.float32), ws_ptr, ws_len, B, Hq, Hkv, Tq, page_size,
                                         num_pages, max_pages, D, _scale(scale, D), *_rope(rope_cos_sin),
                                         _stream(stream))
    _check(st, "attn_decode_paged_fp8_fwd")
    return o, lse
