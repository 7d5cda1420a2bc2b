"""fp64 CPU oracle for causal grouped-query attention (forward and backward).

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the
benchmark's CPU-baseline leg use it; the product path never imports it.
It shares no code with the CUDA library (``gqa_oracle.c`` is plain C, built by
``build()`` with gcc and OpenMP).

Every function takes float64 numpy arrays (callers up-cast the exact bf16
inputs) and returns float64 arrays.  Layouts: dense Q/O/dO [B,Hq,T,D],
K/V [B,Hkv,T,D], LSE/Delta [B,Hq,T]; packed variable length Q [total,Hq,D],
K/V [total,Hkv,D], LSE/Delta [Hq,total].

What is computed is stated in the header of ``gqa_oracle.c`` with its sources
("Project Overview" of llm-from-scratch, section "Performance Layer: kernel/
and parallel/" and the llm/transformer.py component list; the microLLM-rocm
README, section "Why this project exists").  ``paged_decode_fwd`` reads a
paged KV cache (the RoseLLM README, section "Inference and serving": global
paged KV-cache management) by gathering each row's pages into a contiguous
cache, then runs ``decode_fwd``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gqa_oracle.c")
_LIB = os.path.join(_HERE, "libgqa_oracle.so")

_lib = None


def build(force: bool = False, extra_cflags=()) -> str:
    """Compile gqa_oracle.c into libgqa_oracle.so next to it (gcc, OpenMP)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", *extra_cflags, _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def build_variant(out_path: str, extra_cflags) -> str:
    """Compile a variant of the oracle (e.g. with a planted mistake) to ``out_path``."""
    cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", *extra_cflags, _SRC, "-o", out_path, "-lm"]
    subprocess.run(cmd, check=True)
    return out_path


_D = ctypes.POINTER(ctypes.c_double)
_I = ctypes.POINTER(ctypes.c_int)
_L = ctypes.c_long


def _bind(lib):
    lib.oracle_fwd.argtypes = [_D, _D, _D, _D, _D, _L, _L, _L, _L, _L, ctypes.c_int, ctypes.c_double]
    lib.oracle_bwd.argtypes = [_D] * 13 + [_L, _L, _L, _L, _L, ctypes.c_int, ctypes.c_double]
    lib.oracle_varlen_fwd.argtypes = [_D, _D, _D, _D, _D, _I, _L, _L, _L, _L, _L, ctypes.c_int, ctypes.c_double]
    lib.oracle_varlen_bwd.argtypes = [_D] * 13 + [_I, _L, _L, _L, _L, _L, ctypes.c_int, ctypes.c_double]
    lib.oracle_decode_fwd.argtypes = [_D, _D, _D, _I, _D, _D, _L, _L, _L, _L, _L, _L, ctypes.c_double]
    lib.oracle_set_threads.argtypes = [ctypes.c_int]
    for f in (lib.oracle_fwd, lib.oracle_bwd, lib.oracle_varlen_fwd, lib.oracle_varlen_bwd,
              lib.oracle_decode_fwd, lib.oracle_set_threads):
        f.restype = ctypes.c_int
    return lib


def load(path: str | None = None):
    """Load the oracle library (building it first if needed)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        build()
        _lib = _bind(ctypes.CDLL(_LIB))
    return _lib


def _p(a):
    return a.ctypes.data_as(_D)


def _c(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def set_threads(n: int = 0) -> int:
    """Set the OpenMP thread count (0 keeps it); returns the count in use."""
    return load().oracle_set_threads(int(n))


def fwd(q, k, v, causal: bool = True, scale: float | None = None, lib=None):
    """Dense forward.  Returns (O [B,Hq,T,D], LSE [B,Hq,T])."""
    lib = lib or load()
    q, k, v = _c(q), _c(k), _c(v)
    B, Hq, T, D = q.shape
    Hkv = k.shape[1]
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    o = np.zeros_like(q)
    lse = np.zeros((B, Hq, T))
    st = lib.oracle_fwd(_p(q), _p(k), _p(v), _p(o), _p(lse), B, Hq, Hkv, T, D, int(causal), scale)
    if st:
        raise ValueError(f"oracle_fwd status {st}")
    return o, lse


def _err_bufs(want, q, k):
    if not want:
        return None, None, None, ctypes.cast(None, _D), ctypes.cast(None, _D), ctypes.cast(None, _D)
    eq, ek, ev = np.zeros_like(q), np.zeros_like(k), np.zeros_like(k)
    return eq, ek, ev, _p(eq), _p(ek), _p(ev)


def bwd(q, k, v, dout, causal: bool = True, scale: float | None = None, lib=None, err_terms: bool = False):
    """Dense backward of L = sum(dO * O).

    Returns dict with dq, dk, dv and the forward's o, lse and the row term
    delta; with err_terms, also edq, edk, edv: the root-sum-square rounding-
    error scale of each output element (multiply by the unit roundoff) when
    P, dS and the stored O are bf16 operands."""
    lib = lib or load()
    q, k, v, dout = _c(q), _c(k), _c(v), _c(dout)
    B, Hq, T, D = q.shape
    Hkv = k.shape[1]
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    o = np.zeros_like(q)
    lse = np.zeros((B, Hq, T))
    delta = np.zeros((B, Hq, T))
    eq, ek, ev, peq, pek, pev = _err_bufs(err_terms, q, k)
    st = lib.oracle_bwd(_p(q), _p(k), _p(v), _p(dout), _p(dq), _p(dk), _p(dv), _p(o), _p(lse), _p(delta),
                        peq, pek, pev, B, Hq, Hkv, T, D, int(causal), scale)
    if st:
        raise ValueError(f"oracle_bwd status {st}")
    r = dict(dq=dq, dk=dk, dv=dv, o=o, lse=lse, delta=delta)
    if err_terms:
        r.update(edq=np.sqrt(eq), edk=np.sqrt(ek), edv=np.sqrt(ev))
    return r


def _cu(cu_seqlens):
    return np.ascontiguousarray(np.asarray(cu_seqlens), dtype=np.int32)


def varlen_fwd(q, k, v, cu_seqlens, causal: bool = True, scale: float | None = None, lib=None):
    """Packed variable-length forward.  Returns (O [total,Hq,D], LSE [Hq,total])."""
    lib = lib or load()
    q, k, v = _c(q), _c(k), _c(v)
    cu = _cu(cu_seqlens)
    total, Hq, D = q.shape
    Hkv = k.shape[1]
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    o = np.zeros_like(q)
    lse = np.zeros((Hq, total))
    st = lib.oracle_varlen_fwd(_p(q), _p(k), _p(v), _p(o), _p(lse), cu.ctypes.data_as(_I), len(cu) - 1,
                               total, Hq, Hkv, D, int(causal), scale)
    if st:
        raise ValueError(f"oracle_varlen_fwd status {st}")
    return o, lse


def varlen_bwd(q, k, v, dout, cu_seqlens, causal: bool = True, scale: float | None = None, lib=None,
               err_terms: bool = False):
    """Packed variable-length backward; returns the same dict as ``bwd``."""
    lib = lib or load()
    q, k, v, dout = _c(q), _c(k), _c(v), _c(dout)
    cu = _cu(cu_seqlens)
    total, Hq, D = q.shape
    Hkv = k.shape[1]
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    o = np.zeros_like(q)
    lse = np.zeros((Hq, total))
    delta = np.zeros((Hq, total))
    eq, ek, ev, peq, pek, pev = _err_bufs(err_terms, q, k)
    st = lib.oracle_varlen_bwd(_p(q), _p(k), _p(v), _p(dout), _p(dq), _p(dk), _p(dv), _p(o), _p(lse),
                               _p(delta), peq, pek, pev, cu.ctypes.data_as(_I), len(cu) - 1, total, Hq, Hkv,
                               D, int(causal), scale)
    if st:
        raise ValueError(f"oracle_varlen_bwd status {st}")
    r = dict(dq=dq, dk=dk, dv=dv, o=o, lse=lse, delta=delta)
    if err_terms:
        r.update(edq=np.sqrt(eq), edk=np.sqrt(ek), edv=np.sqrt(ev))
    return r


def rope_rotate(x, positions, cos_sin):
    """Rotary position embedding of vectors x [..., D] at integer positions
    [...] (the RoPE of MultiHeadAttentionWithRoPE, llm-from-scratch "Project
    Overview", and the positions-aware RoPE of the microLLM-rocm README):
    with c = cos_sin[p, :D/2], s = cos_sin[p, D/2:], feature i pairs with
    feature i + D/2:  x'_i = x_i c_i - x_{i+D/2} s_i,  x'_{i+D/2} = x_{i+D/2} c_i + x_i s_i."""
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    h = D // 2
    cs = np.asarray(cos_sin, dtype=np.float64)[np.asarray(positions)]
    c, s = cs[..., :h], cs[..., h:]
    lo, hi = x[..., :h], x[..., h:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


def rope_rotate_t(x, positions, cos_sin):
    """The transpose (= inverse) of ``rope_rotate`` at the same positions:
    x'_i = x_i c_i + x_{i+D/2} s_i,  x'_{i+D/2} = x_{i+D/2} c_i - x_i s_i.  It takes
    a gradient with respect to rotated vectors back to the unrotated ones."""
    x = np.asarray(x, dtype=np.float64)
    h = x.shape[-1] // 2
    cs = np.asarray(cos_sin, dtype=np.float64)[np.asarray(positions)]
    c, s = cs[..., :h], cs[..., h:]
    lo, hi = x[..., :h], x[..., h:]
    return np.concatenate([lo * c + hi * s, hi * c - lo * s], axis=-1)


def _rope_err_t(e, positions, cos_sin):
    """Root-sum-square rounding-error scales carried through rope_rotate_t."""
    e = np.asarray(e, dtype=np.float64)
    h = e.shape[-1] // 2
    cs = np.asarray(cos_sin, dtype=np.float64)[np.asarray(positions)]
    c2, s2 = cs[..., :h] ** 2, cs[..., h:] ** 2
    lo2, hi2 = e[..., :h] ** 2, e[..., h:] ** 2
    return np.sqrt(np.concatenate([lo2 * c2 + hi2 * s2, hi2 * c2 + lo2 * s2], axis=-1))


def _dense_positions(x):
    B, H, T = np.asarray(x).shape[:3]
    return np.broadcast_to(np.arange(T), (B, H, T))


def _varlen_positions(x, cu_seqlens):
    cu = np.asarray(cu_seqlens)
    total, H = np.asarray(x).shape[:2]
    pos = np.zeros(total, dtype=np.int64)
    for a, b in zip(cu[:-1], cu[1:]):
        pos[a:b] = np.arange(b - a)
    return np.broadcast_to(pos[:, None], (total, H))


def rope_fwd(q, k, v, rope_cos_sin, causal: bool = True, scale: float | None = None, lib=None):
    """Dense attention with rotary queries and keys (RoPE of
    MultiHeadAttentionWithRoPE, llm-from-scratch "Project Overview"; the
    positions-aware RoPE of the microLLM-rocm README): q and k of each row are
    rotated (rope_rotate) at their positions 0..T-1, then ``fwd``.  Returns
    (O, LSE) as ``fwd``."""
    return fwd(rope_rotate(q, _dense_positions(q), rope_cos_sin), rope_rotate(k, _dense_positions(k), rope_cos_sin),
               v, causal=causal, scale=scale, lib=lib)


def rope_bwd(q, k, v, dout, rope_cos_sin, causal: bool = True, scale: float | None = None, lib=None,
             err_terms: bool = False):
    """Backward of L = sum(dO * rope_fwd(q, k, v)) with respect to the
    unrotated q, k and v: ``bwd`` on the rotated q, k, then dq and dk taken
    back through the rotation (rope_rotate_t).  Returns the same dict as
    ``bwd`` (error scales carried through the rotation)."""
    pq, pk = _dense_positions(q), _dense_positions(k)
    r = bwd(rope_rotate(q, pq, rope_cos_sin), rope_rotate(k, pk, rope_cos_sin), v, dout, causal=causal,
            scale=scale, lib=lib, err_terms=err_terms)
    r["dq"] = rope_rotate_t(r["dq"], pq, rope_cos_sin)
    r["dk"] = rope_rotate_t(r["dk"], pk, rope_cos_sin)
    if err_terms:
        r["edq"] = _rope_err_t(r["edq"], pq, rope_cos_sin)
        r["edk"] = _rope_err_t(r["edk"], pk, rope_cos_sin)
    return r


def rope_varlen_fwd(q, k, v, cu_seqlens, rope_cos_sin, causal: bool = True, scale: float | None = None, lib=None):
    """``rope_fwd`` for a packed variable-length batch: positions restart at 0
    in every sequence (only position differences within a sequence reach
    the result)."""
    return varlen_fwd(rope_rotate(q, _varlen_positions(q, cu_seqlens), rope_cos_sin),
                      rope_rotate(k, _varlen_positions(k, cu_seqlens), rope_cos_sin), v, cu_seqlens,
                      causal=causal, scale=scale, lib=lib)


def rope_varlen_bwd(q, k, v, dout, cu_seqlens, rope_cos_sin, causal: bool = True, scale: float | None = None,
                    lib=None, err_terms: bool = False):
    """``rope_bwd`` for a packed variable-length batch."""
    pq, pk = _varlen_positions(q, cu_seqlens), _varlen_positions(k, cu_seqlens)
    r = varlen_bwd(rope_rotate(q, pq, rope_cos_sin), rope_rotate(k, pk, rope_cos_sin), v, dout, cu_seqlens,
                   causal=causal, scale=scale, lib=lib, err_terms=err_terms)
    r["dq"] = rope_rotate_t(r["dq"], pq, rope_cos_sin)
    r["dk"] = rope_rotate_t(r["dk"], pk, rope_cos_sin)
    if err_terms:
        r["edq"] = _rope_err_t(r["edq"], pq, rope_cos_sin)
        r["edk"] = _rope_err_t(r["edk"], pk, rope_cos_sin)
    return r


def decode_fwd(q, k_cache, v_cache, cache_lens, scale: float | None = None, lib=None, rope_cos_sin=None):
    """Attention of the newest Tq positions over a KV cache.

    q [B,Hq,Tq,D]; k_cache, v_cache [B,Hkv,S,D]; cache_lens [B] (keys held per
    row, including the Tq new ones).  Query t of row b attends to keys
    j <= cache_lens[b] - Tq + t.  With rope_cos_sin [positions, D] the
    queries are first rotated (rope_rotate) at their positions
    cache_lens[b] - Tq + t (the cache holds keys already rotated at theirs).
    Returns (O [B,Hq,Tq,D], LSE [B,Hq,Tq])."""
    lib = lib or load()
    if rope_cos_sin is not None:
        lens_ = np.asarray(cache_lens)
        Tq_ = np.asarray(q).shape[2]
        pos = lens_[:, None, None] - Tq_ + np.arange(Tq_)[None, None, :]
        q = rope_rotate(q, np.broadcast_to(pos, np.asarray(q).shape[:3]), rope_cos_sin)
    q, k, v = _c(q), _c(k_cache), _c(v_cache)
    lens = _cu(cache_lens)
    B, Hq, Tq, D = q.shape
    Hkv, S = k.shape[1], k.shape[2]
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    o = np.zeros_like(q)
    lse = np.zeros((B, Hq, Tq))
    st = lib.oracle_decode_fwd(_p(q), _p(k), _p(v), lens.ctypes.data_as(_I), _p(o), _p(lse), B, Hq, Hkv, Tq, S, D,
                               scale)
    if st:
        raise ValueError(f"oracle_decode_fwd status {st}")
    return o, lse


def paged_decode_fwd(q, k_pages, v_pages, block_table, cache_lens, scale: float | None = None, lib=None,
                     rope_cos_sin=None):
    """Cached attention over a paged KV cache.

    k_pages, v_pages [num_pages, Hkv, page_size, D] (each page holds page_size
    consecutive positions of one batch row, all K/V heads); block_table
    [B, max_pages] int: key position j of row b is row j % page_size of page
    block_table[b, j // page_size].  Only the pages that hold one of the row's
    cache_lens[b] keys are read.  Same queries, mask and results as
    ``decode_fwd`` over the gathered cache [B, Hkv, max_pages * page_size, D]."""
    kp, vp = _c(k_pages), _c(v_pages)
    bt = np.asarray(block_table)
    lens = np.asarray(cache_lens)
    B = q.shape[0]
    _, Hkv, psz, D = kp.shape
    S = bt.shape[1] * psz
    k = np.zeros((B, Hkv, S, D))
    v = np.zeros((B, Hkv, S, D))
    for b in range(B):
        for i in range((int(lens[b]) + psz - 1) // psz):
            page = int(bt[b, i])
            k[b, :, i * psz:(i + 1) * psz] = kp[page]
            v[b, :, i * psz:(i + 1) * psz] = vp[page]
    return decode_fwd(q, k, v, lens, scale=scale, lib=lib, rope_cos_sin=rope_cos_sin)


def e4m3_decode(codes):
    """Values of FP8 E4M3 codes (uint8): sign bit, 4 exponent bits (bias 7), 3
    mantissa bits; exponent 0 is subnormal (m/8 * 2^-6); no infinities; the
    two codes with all exponent and mantissa bits set are NaN."""
    c = np.asarray(codes).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return sign * val


def fp8_decode_fwd(q, k8, v8, k_scale, v_scale, cache_lens, scale: float | None = None, lib=None, rope_cos_sin=None):
    """Cached attention over FP8 E4M3 caches with per-tensor scales (the FP8
    quantize / dequantize and KV-cache work of the microLLM-rocm README,
    section "Why this project exists"): K = e4m3(k8) * k_scale,
    V = e4m3(v8) * v_scale, then ``decode_fwd``."""
    k = e4m3_decode(k8) * float(k_scale)
    v = e4m3_decode(v8) * float(v_scale)
    return decode_fwd(q, k, v, cache_lens, scale=scale, lib=lib, rope_cos_sin=rope_cos_sin)
