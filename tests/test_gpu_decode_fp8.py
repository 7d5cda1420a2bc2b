"""Cached attention over FP8 (E4M3) K/V caches on the GPU against the fp64 oracle.

The oracle decodes the same E4M3 codes with the same per-tensor scales.
Cases: several shapes (D 64/128, Tq 1..4, G 1..8, more than 16 query rows,
a cache holding only the new queries), rows past each length filled with
E4M3 NaN codes (must not leak), rotary queries, a paged FP8 pool, and the
FP8 long-context workload at its full size.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL_REL_O, check, check_lse, to64
from causal_gqa_attention_fwd_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gq():
    import causal_gqa_attention_fwd_gb300 as g
    g.lib()
    oracle.set_threads(0)
    return g


def run_gpu(gq, x, scale, **kw):
    q, k8, v8, lens = (x[n].cuda() for n in ("q", "k8", "v8", "cache_lens"))
    return gq.attn_decode_fp8_fwd(q, k8, v8, x["k_scale"], x["v_scale"], lens, scale=scale, **kw)


def run_oracle(x, scale, **kw):
    return oracle.fp8_decode_fwd(to64(x["q"]), x["k8"].numpy(), x["v8"].numpy(), x["k_scale"], x["v_scale"],
                                 x["cache_lens"].numpy(), scale=scale, **kw)


CASES = [
    # B, Hq, Hkv, Tq, S, D, cache_lens
    (3, 8, 2, 1, 700, 128, [700, 1, 389]),
    (2, 14, 2, 2, 600, 64, [600, 130]),
    (2, 16, 2, 4, 640, 128, [640, 385]),
    (2, 4, 4, 1, 300, 64, [300, 129]),
    (4, 32, 8, 1, 4096, 128, None),
    (8, 32, 8, 1, 16384, 64, None),     # D = 64 with dozens of chunks per CTA: its rings wrap
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%d_Hq%d_Hkv%d_Tq%d_S%d_D%d" % c[:6])
def test_fp8_decode_matches_oracle(gq, case):
    B, Hq, Hkv, Tq, S, D, lens = case
    x = W.fp8_decode_inputs(B, Hq, Hkv, Tq, S, D, cache_lens=lens, seed=31)
    scale = 1.0 / np.sqrt(D)
    o, lse = run_gpu(gq, x, scale)
    assert gq.get_device_status() == 0
    ro, rlse = run_oracle(x, scale)
    check("o", o, ro, TOL_REL_O)
    check_lse(lse, rlse)


def test_fp8_ignores_nan_codes_past_length(gq):
    B, Hq, Hkv, Tq, S, D = 3, 8, 2, 2, 500, 128
    lens = [500, 2, 261]
    x = W.fp8_decode_inputs(B, Hq, Hkv, Tq, S, D, cache_lens=lens, seed=32)
    ref = run_oracle(x, 0.1)
    for b, n in enumerate(lens):
        x["k8"][b, :, n:] = 0x7F
        x["v8"][b, :, n:] = 0xFF
    o, lse = run_gpu(gq, x, 0.1)
    assert gq.get_device_status() == 0
    check("o", o, ref[0], TOL_REL_O)
    check_lse(lse, ref[1])


@pytest.mark.parametrize("D", [128, 64])
def test_fp8_rope_decode(gq, D):
    B, Hq, Hkv, Tq, S = 2, 8, 2, 3, 3000
    x = W.fp8_decode_inputs(B, Hq, Hkv, Tq, S, D, cache_lens=[3000, 1500], seed=33)
    tab = W.rope_cos_sin_table(S, D)
    o, lse = run_gpu(gq, x, 0.09, rope_cos_sin=tab.cuda())
    assert gq.get_device_status() == 0
    ro, rlse = run_oracle(x, 0.09, rope_cos_sin=tab.double().numpy())
    check("o", o, ro, TOL_REL_O)
    check_lse(lse, rlse)


PAGED_FP8_CASES = [
    # B, Hq, Hkv, Tq, page_size, max_pages, D, cache_lens
    (3, 8, 2, 1, 32, 30, 128, [960, 1, 333]),
    (3, 14, 2, 2, 16, 40, 64, [640, 2, 301]),   # 64-byte swizzle, 8 page boxes per chunk
    (2, 8, 8, 1, 128, 5, 64, [640, 129]),      # 64-byte swizzle, chunks inside a page
]


@pytest.mark.parametrize("case", PAGED_FP8_CASES, ids=lambda c: "B%d_Hq%d_Hkv%d_Tq%d_page%d_D%d" % (c[0], c[1], c[2], c[3], c[4], c[6]))
def test_paged_fp8_decode(gq, case):
    B, Hq, Hkv, Tq, psz, maxp, D, lens = case
    x = W.paged_decode_inputs(B, Hq, Hkv, Tq, psz, maxp, D, cache_lens=lens, spare_pages=2, seed=34)
    k8p, ks = W.fp8_cache(x["k_pages"].float())
    v8p, vs = W.fp8_cache(x["v_pages"].float())
    q, bt, ln = x["q"].cuda(), x["block_table"].cuda(), x["cache_lens"].cuda()
    o, lse = gq.attn_decode_paged_fp8_fwd(q, k8p.cuda(), v8p.cuda(), ks, vs, bt, ln, scale=0.1)
    assert gq.get_device_status() == 0
    ro, rlse = oracle.paged_decode_fwd(to64(x["q"]), oracle.e4m3_decode(k8p.numpy()) * ks,
                                       oracle.e4m3_decode(v8p.numpy()) * vs, x["block_table"].numpy(),
                                       x["cache_lens"].numpy(), scale=0.1)
    check("o", o, ro, TOL_REL_O)
    check_lse(lse, rlse)


@pytest.mark.parametrize("name", [n for n, w in W.DECODE_WORKLOADS.items() if w.fp8])
def test_fp8_decode_workloads_full(gq, name):
    w = W.DECODE_WORKLOADS[name]
    x = W.make_decode_inputs(w)
    o, lse = run_gpu(gq, x, w.softmax_scale)
    assert gq.get_device_status() == 0
    ro, rlse = run_oracle(x, w.softmax_scale)
    check("o", o, ro, TOL_REL_O)
    check_lse(lse, rlse)


def test_fp8_decode_is_deterministic(gq):
    """Many chunks per CTA, ragged lengths: repeated calls give the same bits."""
    x = W.fp8_decode_inputs(4, 32, 8, 1, 24000, 128, min_len=12000, max_len=24000, seed=35)
    o1, l1 = run_gpu(gq, x, 0.09)
    for _ in range(3):
        o2, l2 = run_gpu(gq, x, 0.09)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_fp8_one_hot_values_keep_chunks_apart(gq):
    """V row s is the unit vector of feature (s // 128) % D, so feature d of
    O is the softmax mass of the 128-key chunks d, d + D, ...: a chunk whose
    values were lost or taken from another chunk shows as one feature off by
    about 1 / (chunks in the row)."""
    B, Hq, Hkv, Tq, S, D = 4, 16, 4, 1, 20000, 128
    x = W.fp8_decode_inputs(B, Hq, Hkv, Tq, S, D, min_len=9000, max_len=20000, seed=36)
    one = 0x38  # E4M3 code of 1.0
    v8 = torch.zeros(S, D, dtype=torch.uint8)
    v8[torch.arange(S), (torch.arange(S) // 128) % D] = one
    x["v8"] = v8.expand(B, Hkv, S, D).contiguous()
    x["v_scale"] = 1.0
    o, lse = run_gpu(gq, x, 0.09)
    assert gq.get_device_status() == 0
    ro, rlse = run_oracle(x, 0.09)
    err = np.abs(to64(o) - ro).max()
    assert err < 2e-3 * ro.max() + 1e-4, f"max abs error {err:.3e} (largest feature {ro.max():.3e})"
    check("o", o, ro, TOL_REL_O)
    check_lse(lse, rlse)


def test_fp8_nan_codes_inside_the_cache(gq):
    """An E4M3 NaN code at a visible key makes NaN exactly where the oracle
    does (V: that feature of the group's rows; K: the whole rows that see
    it); everything else still matches."""
    B, Hq, Hkv, Tq, S, D = 2, 8, 2, 1, 700, 128
    x = W.fp8_decode_inputs(B, Hq, Hkv, Tq, S, D, cache_lens=[700, 300], seed=37)
    x["v8"][0, 1, 400, 5] = 0x7F
    x["v8"][1, 0, 17, 100] = 0xFF
    x["k8"][1, 1, 250, 3] = 0x7F
    o, lse = run_gpu(gq, x, 0.1)
    assert gq.get_device_status() == 0
    ro, rlse = run_oracle(x, 0.1)
    g, ref = to64(o), ro
    assert np.isnan(ref).any()
    np.testing.assert_array_equal(np.isnan(g), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.abs(g[ok] - ref[ok]).max() < 2e-2
    np.testing.assert_array_equal(np.isnan(to64(lse)), np.isnan(rlse))
