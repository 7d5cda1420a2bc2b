"""Seeded synthetic workloads for causal GQA attention.

This module only draws inputs: it holds no attention arithmetic, and both the
CUDA path's tests/benchmark and the CPU oracle's tests take their inputs from
here.  Every tensor is drawn on the CPU from ``torch.Generator().manual_seed``
in float32, then rounded to bf16, so the GPU and the oracle see identical
bits.  Draw order: (variable-length: the sequence lengths first), then Q, K,
V, dO.

The five workloads are shaped after the models the pages train: a tiny GQA
check, a Qwen3-0.6B-shaped layer, a GPT-2-small-shaped MHA layer, a long
context GQA layer (T = 4096, D = 128) and a packed variable-length batch.

The cached (decode) workloads put Tq new query positions per batch row
against a KV cache of capacity S holding cache_lens[b] keys: two are shaped
after the steady-decode rows the microLLM-rocm README reports (context 2048,
batch 8, Qwen2.5-0.5B and DeepSeek-R1-Distill-Qwen-1.5B attention shapes),
one is a long-context GQA cache larger than the L2 cache (per-row lengths
drawn between S/2 and S), and the same long-context cache is also paged
(pages of 64 and of 16 positions, shuffled over the pool).  Draw order:
cache lengths, Q, K cache, V cache (paged: K pages, V pages, then the page
permutation).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    Hq: int
    Hkv: int
    D: int
    B: int = 0              # dense only
    T: int = 0              # dense only
    num_seqs: int = 0       # variable length only
    min_len: int = 0
    max_len: int = 0
    q_std: float = 1.0
    causal: bool = True
    scale: float = field(default=0.0)

    @property
    def varlen(self) -> bool:
        return self.num_seqs > 0

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale else 1.0 / math.sqrt(self.D)


WORKLOADS = {
    "tiny": Workload("tiny", B=1, Hq=4, Hkv=2, T=128, D=64),
    "qwen3_0p6b_layer": Workload("qwen3_0p6b_layer", B=4, Hq=16, Hkv=8, T=512, D=128),
    "gpt2_small_mha": Workload("gpt2_small_mha", B=8, Hq=12, Hkv=12, T=1024, D=64),
    "long_gqa_t4096": Workload("long_gqa_t4096", B=2, Hq=32, Hkv=8, T=4096, D=128),
    "varlen16": Workload("varlen16", num_seqs=16, min_len=64, max_len=2048, Hq=16, Hkv=8, D=128, q_std=4.0),
}

HEADLINE = "long_gqa_t4096"


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Tq: int
    S: int                  # cache capacity (keys per row)
    D: int
    min_len: int            # cache_lens drawn uniformly in [min_len, max_len]
    max_len: int
    scale: float = field(default=0.0)
    page_size: int = 0      # > 0: paged cache of S / page_size pages per row
    fp8: bool = False       # E4M3 caches with per-tensor scales
    rope: bool = False      # queries rotated at their positions (rotary table of S rows)

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale else 1.0 / math.sqrt(self.D)


DECODE_WORKLOADS = {
    "decode_qwen25_0p5b_t2048_b8": DecodeWorkload("decode_qwen25_0p5b_t2048_b8", B=8, Hq=14, Hkv=2, Tq=1,
                                                  S=2048, D=64, min_len=2048, max_len=2048),
    "decode_r1distill_1p5b_t2048_b8": DecodeWorkload("decode_r1distill_1p5b_t2048_b8", B=8, Hq=12, Hkv=2, Tq=1,
                                                     S=2048, D=128, min_len=2048, max_len=2048),
    "decode_long_gqa_s32k": DecodeWorkload("decode_long_gqa_s32k", B=8, Hq=32, Hkv=8, Tq=1, S=32768, D=128,
                                           min_len=16384, max_len=32768),
}

DECODE_WORKLOADS["decode_paged_long_gqa_s32k_p64"] = DecodeWorkload(
    "decode_paged_long_gqa_s32k_p64", B=8, Hq=32, Hkv=8, Tq=1, S=32768, D=128, min_len=16384, max_len=32768,
    page_size=64)
DECODE_WORKLOADS["decode_paged_long_gqa_s32k_p16"] = DecodeWorkload(
    "decode_paged_long_gqa_s32k_p16", B=8, Hq=32, Hkv=8, Tq=1, S=32768, D=128, min_len=16384, max_len=32768,
    page_size=16)

DECODE_WORKLOADS["decode_fp8_long_gqa_s32k"] = DecodeWorkload(
    "decode_fp8_long_gqa_s32k", B=8, Hq=32, Hkv=8, Tq=1, S=32768, D=128, min_len=16384, max_len=32768, fp8=True)

DECODE_WORKLOADS["decode_rope_long_gqa_s32k"] = DecodeWorkload(
    "decode_rope_long_gqa_s32k", B=8, Hq=32, Hkv=8, Tq=1, S=32768, D=128, min_len=16384, max_len=32768, rope=True)

DECODE_HEADLINE = "decode_long_gqa_s32k"


def _randn(g, shape, std=1.0):
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        x = x * std
    return x.to(torch.bfloat16)


def dense_inputs(B, Hq, Hkv, T, D, seed=0, q_std=1.0):
    """Q,dO [B,Hq,T,D], K,V [B,Hkv,T,D], bf16, CPU."""
    g = torch.Generator().manual_seed(seed)
    q = _randn(g, (B, Hq, T, D), q_std)
    k = _randn(g, (B, Hkv, T, D))
    v = _randn(g, (B, Hkv, T, D))
    do = _randn(g, (B, Hq, T, D))
    return dict(q=q, k=k, v=v, do=do)


def varlen_lengths(num_seqs, min_len, max_len, g):
    return torch.randint(min_len, max_len + 1, (num_seqs,), generator=g, dtype=torch.int64)


def varlen_inputs(lengths, Hq, Hkv, D, seed=0, q_std=1.0, g=None):
    """Packed Q,dO [total,Hq,D], K,V [total,Hkv,D] bf16 and cu_seqlens int32 [N+1]."""
    if g is None:
        g = torch.Generator().manual_seed(seed)
    lengths = torch.as_tensor(lengths, dtype=torch.int64)
    cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
    if len(lengths):
        cu[1:] = torch.cumsum(lengths, 0).to(torch.int32)
    total = int(cu[-1])
    q = _randn(g, (total, Hq, D), q_std)
    k = _randn(g, (total, Hkv, D))
    v = _randn(g, (total, Hkv, D))
    do = _randn(g, (total, Hq, D))
    return dict(q=q, k=k, v=v, do=do, cu_seqlens=cu, max_seqlen=int(lengths.max()) if len(lengths) else 0)


def make_inputs(w: Workload, seed=0):
    """Inputs of a named workload (dense or variable length)."""
    if w.varlen:
        g = torch.Generator().manual_seed(seed)
        lengths = varlen_lengths(w.num_seqs, w.min_len, w.max_len, g)
        return varlen_inputs(lengths, w.Hq, w.Hkv, w.D, q_std=w.q_std, g=g)
    return dense_inputs(w.B, w.Hq, w.Hkv, w.T, w.D, seed=seed, q_std=w.q_std)



def decode_inputs(B, Hq, Hkv, Tq, S, D, cache_lens=None, min_len=None, max_len=None, seed=0):
    """q [B,Hq,Tq,D], k_cache/v_cache [B,Hkv,S,D] bf16 and cache_lens int32 [B], CPU.  The whole
    cache (rows past each length too) is drawn, so a kernel that reads past a row's length sees
    finite, wrong keys rather than zeros."""
    g = torch.Generator().manual_seed(seed)
    if cache_lens is None:
        lo = Tq if min_len is None else min_len
        hi = S if max_len is None else max_len
        cache_lens = torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64)
    lens = torch.as_tensor(cache_lens, dtype=torch.int32)
    q = _randn(g, (B, Hq, Tq, D))
    k = _randn(g, (B, Hkv, S, D))
    v = _randn(g, (B, Hkv, S, D))
    return dict(q=q, k_cache=k, v_cache=v, cache_lens=lens)


def paged_decode_inputs(B, Hq, Hkv, Tq, page_size, max_pages, D, cache_lens=None, min_len=None, max_len=None,
                        spare_pages=0, seed=0):
    """q [B,Hq,Tq,D], a page pool k_pages/v_pages [num_pages,Hkv,page_size,D] bf16 (num_pages =
    B * max_pages + spare_pages), block_table int32 [B, max_pages] and cache_lens int32 [B], CPU.
    The table is a random permutation of the pool's pages; entries past each row's last page are -1.
    Draw order: cache lengths, Q, K pages, V pages, the permutation."""
    g = torch.Generator().manual_seed(seed)
    S = page_size * max_pages
    if cache_lens is None:
        lo = Tq if min_len is None else min_len
        hi = S if max_len is None else max_len
        cache_lens = torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64)
    lens = torch.as_tensor(cache_lens, dtype=torch.int32)
    num_pages = B * max_pages + spare_pages
    q = _randn(g, (B, Hq, Tq, D))
    kp = _randn(g, (num_pages, Hkv, page_size, D))
    vp = _randn(g, (num_pages, Hkv, page_size, D))
    table = torch.randperm(num_pages, generator=g)[:B * max_pages].reshape(B, max_pages).to(torch.int32)
    for b in range(B):
        table[b, (int(lens[b]) + page_size - 1) // page_size:] = -1
    return dict(q=q, k_pages=kp, v_pages=vp, block_table=table, cache_lens=lens)


def make_decode_inputs(w: DecodeWorkload, seed=0):
    """The workload's inputs (CPU); with ``rope`` also ``rope_cs``, the
    rotary table of the cache's S positions."""
    if w.fp8:
        x = fp8_decode_inputs(w.B, w.Hq, w.Hkv, w.Tq, w.S, w.D, min_len=w.min_len, max_len=w.max_len, seed=seed)
    elif w.page_size:
        x = paged_decode_inputs(w.B, w.Hq, w.Hkv, w.Tq, w.page_size, w.S // w.page_size, w.D, min_len=w.min_len,
                                max_len=w.max_len, seed=seed)
    else:
        x = decode_inputs(w.B, w.Hq, w.Hkv, w.Tq, w.S, w.D, min_len=w.min_len, max_len=w.max_len, seed=seed)
    if w.rope:
        x["rope_cs"] = rope_cos_sin_table(w.S, w.D)
    return x


def rope_cos_sin_table(positions: int, D: int, base: float = 10000.0):
    """Rotary table [positions, D] float32: row p holds cos(p * theta_i) for
    i < D/2, then sin(p * theta_i), theta_i = base^(-2i/D) -- an input of both
    the kernels and the oracle (as the cos/sin caches serving stacks keep),
    computed in float64 and rounded once."""
    i = torch.arange(D // 2, dtype=torch.float64)
    theta = base ** (-2.0 * i / D)
    ang = torch.arange(positions, dtype=torch.float64)[:, None] * theta[None, :]
    return torch.cat([torch.cos(ang), torch.sin(ang)], dim=1).to(torch.float32)


def to_e4m3(x, scale: float):
    """E4M3 codes (uint8) of x / scale, rounded to nearest (PyTorch's float8_e4m3fn cast) -- input
    preparation: the kernels and the oracle both take the codes and the scale."""
    return (x.to(torch.float32) / scale).to(torch.float8_e4m3fn).view(torch.uint8)


def fp8_cache(x):
    """(codes, scale) of an f32 cache with one scale: amax maps to the format's largest finite value, 448."""
    scale = float(x.abs().max()) / 448.0
    return to_e4m3(x, scale), scale


def fp8_decode_inputs(B, Hq, Hkv, Tq, S, D, cache_lens=None, min_len=None, max_len=None, seed=0):
    """q bf16 [B,Hq,Tq,D]; k8, v8 uint8 [B,Hkv,S,D] E4M3 codes with scales k_scale, v_scale (caches drawn
    N(0,1) in f32, each mapped onto the E4M3 range by its own amax); cache_lens int32 [B]."""
    g = torch.Generator().manual_seed(seed)
    if cache_lens is None:
        lo = Tq if min_len is None else min_len
        hi = S if max_len is None else max_len
        cache_lens = torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64)
    lens = torch.as_tensor(cache_lens, dtype=torch.int32)
    q = _randn(g, (B, Hq, Tq, D))
    k8, ks = fp8_cache(torch.randn(B, Hkv, S, D, generator=g, dtype=torch.float32))
    v8, vs = fp8_cache(torch.randn(B, Hkv, S, D, generator=g, dtype=torch.float32))
    return dict(q=q, k8=k8, v8=v8, k_scale=ks, v_scale=vs, cache_lens=lens)
