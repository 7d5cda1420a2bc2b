"""Cached (decode) attention on the GPU against the fp64 oracle.

Query t of batch row b attends to the keys j <= cache_lens[b] - Tq + t of its
own cache.  Cases cover: a cache holding only the new queries (len = Tq),
lengths just past a 128-key chunk edge, MHA (G = 1), G = 7, query-row blocks of
4 / 8 / 16 rows and more than 16 rows (two blocks), an unsplit key range
written directly, long items of several chunks, a split key range merged
afterwards, cache rows past each length filled with NaN, invalid lengths, and
the three decode workloads at their full sizes.
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


def run_gpu(gq, x, scale):
    q, k, v, lens = (x[n].cuda() for n in ("q", "k_cache", "v_cache", "cache_lens"))
    o, lse = gq.attn_decode_fwd(q, k, v, lens, scale=scale)
    return o, lse


def run_oracle(x, scale):
    return oracle.decode_fwd(to64(x["q"]), to64(x["k_cache"]), to64(x["v_cache"]), x["cache_lens"].numpy(),
                             scale=scale)


CASES = [
    # B, Hq, Hkv, Tq, S, D, cache_lens
    (3, 8, 2, 1, 300, 128, [300, 1, 129]),
    (3, 8, 2, 3, 1000, 64, [3, 1000, 517]),
    (2, 4, 4, 2, 257, 128, [257, 130]),
    (2, 16, 2, 4, 640, 128, [640, 385]),
    (2, 14, 2, 1, 700, 64, [700, 333]),
    (1, 2, 1, 1, 100, 64, [77]),
    (64, 32, 32, 1, 1024, 64, None),
    (4, 64, 16, 1, 16384, 128, None),
    (2, 8, 1, 5, 4500, 128, [4500, 4097]),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%d_Hq%d_Hkv%d_Tq%d_S%d_D%d" % c[:6])
def test_decode_matches_oracle(gq, case):
    B, Hq, Hkv, Tq, S, D, lens = case
    x = W.decode_inputs(B, Hq, Hkv, Tq, S, D, cache_lens=lens, seed=11)
    scale = 1.0 / np.sqrt(D)
    o, lse = run_gpu(gq, x, scale)
    assert gq.get_device_status() == 0
    ro, rlse = run_oracle(x, scale)
    check("o", o, ro, TOL_REL_O)
    check_lse(lse, rlse)


def test_decode_is_deterministic(gq):
    x = W.decode_inputs(4, 64, 16, 1, 16384, 128, seed=3)
    o1, l1 = run_gpu(gq, x, 0.09)
    o2, l2 = run_gpu(gq, x, 0.09)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_decode_ignores_cache_rows_past_length(gq):
    """Rows at or past cache_lens[b] are outside the cache: NaN there must not leak."""
    B, Hq, Hkv, Tq, S, D = 3, 8, 2, 2, 700, 128
    lens = [700, 2, 389]
    x = W.decode_inputs(B, Hq, Hkv, Tq, S, D, cache_lens=lens, seed=5)
    ref = run_oracle(x, 0.1)
    for b, n in enumerate(lens):
        x["k_cache"][b, :, n:] = float("nan")
        x["v_cache"][b, :, n:] = float("nan")
    o, lse = run_gpu(gq, x, 0.1)
    assert gq.get_device_status() == 0
    check("o", o, ref[0], TOL_REL_O)
    check_lse(lse, ref[1])


def test_decode_reports_invalid_lengths(gq):
    """A length below Tq or above S is reported (ATTN_ERR_SEQLENS); valid rows are still computed."""
    B, Hq, Hkv, Tq, S, D = 3, 8, 2, 2, 600, 64
    x = W.decode_inputs(B, Hq, Hkv, Tq, S, D, cache_lens=[600, 1, 601], seed=9)
    q, k, v, lens = (x[n].cuda() for n in ("q", "k_cache", "v_cache", "cache_lens"))
    o = torch.full_like(q, 7.0)
    lse = torch.full((B, Hq, Tq), 7.0, device="cuda")
    gq.attn_decode_fwd(q, k, v, lens, scale=0.125, o=o, lse=lse)
    assert gq.get_device_status() == 5
    assert gq.get_device_status() == 0            # cleared by the first read
    ok = {k_: t[:1] for k_, t in x.items() if k_ != "cache_lens"}
    ok["cache_lens"] = x["cache_lens"][:1]
    ro, rlse = run_oracle(ok, 0.125)
    check("o", o[:1], ro, TOL_REL_O)
    check_lse(lse[:1], rlse)
    assert bool((o[1:] == 7.0).all()) and bool((lse[1:] == 7.0).all())   # left unwritten


@pytest.mark.parametrize("name", [n for n, w in W.DECODE_WORKLOADS.items() if not w.page_size and not w.fp8])
def test_decode_workloads_full(gq, name):
    w = W.DECODE_WORKLOADS[name]
    x = W.make_decode_inputs(w)
    o, lse = run_gpu(gq, x, w.softmax_scale)
    assert gq.get_device_status() == 0
    ro, rlse = run_oracle(x, w.softmax_scale)
    check("o", o, ro, TOL_REL_O)
    check_lse(lse, rlse)


def test_decode_workspace_reuse(gq):
    """One workspace across calls: a unit cut into pieces in the first call is
    processed whole in the second, whose result must not pick up the first
    call's partials."""
    B, Hq, Hkv, Tq, S, D = 2, 8, 2, 1, 4096, 128
    ws = torch.empty(gq.attn_decode_workspace_size(B, Hq, Hkv, Tq, S, D), dtype=torch.uint8, device="cuda")
    for lens in ([4096, 4096], [100, 4096], [4096, 1]):
        x = W.decode_inputs(B, Hq, Hkv, Tq, S, D, cache_lens=lens, seed=len(lens) + lens[0])
        q, k, v, ln = (x[n].cuda() for n in ("q", "k_cache", "v_cache", "cache_lens"))
        o, lse = gq.attn_decode_fwd(q, k, v, ln, scale=0.1, workspace=ws)
        assert gq.get_device_status() == 0
        ro, rlse = run_oracle(x, 0.1)
        check("o", o, ro, TOL_REL_O)
        check_lse(lse, rlse)


ROPE_CASES = [
    # B, Hq, Hkv, Tq, S, D, cache_lens
    (3, 8, 2, 2, 700, 128, [700, 2, 389]),
    (2, 14, 2, 1, 600, 64, [600, 130]),
    (2, 4, 1, 3, 20000, 128, [20000, 16385]),
    (2, 16, 2, 4, 640, 128, [640, 385]),
]


@pytest.mark.parametrize("case", ROPE_CASES, ids=lambda c: "B%d_Hq%d_Hkv%d_Tq%d_S%d_D%d" % c[:6])
def test_rope_decode_matches_oracle(gq, case):
    """Queries rotated in the kernel at cache_lens[b] - Tq + t (positions up to 20K)."""
    B, Hq, Hkv, Tq, S, D, lens = case
    x = W.decode_inputs(B, Hq, Hkv, Tq, S, D, cache_lens=lens, seed=17)
    tab = W.rope_cos_sin_table(S, D)
    scale = 1.0 / np.sqrt(D)
    q, k, v, ln = (x[n].cuda() for n in ("q", "k_cache", "v_cache", "cache_lens"))
    o, lse = gq.attn_decode_fwd(q, k, v, ln, scale=scale, rope_cos_sin=tab.cuda())
    assert gq.get_device_status() == 0
    ro, rlse = oracle.decode_fwd(to64(x["q"]), to64(x["k_cache"]), to64(x["v_cache"]), x["cache_lens"].numpy(),
                                 scale=scale, rope_cos_sin=tab.double().numpy())
    check("o", o, ro, TOL_REL_O)
    check_lse(lse, rlse)
    plain, _ = run_gpu(gq, x, scale)
    assert not torch.equal(plain, o)


def test_decode_many_batch_rows(gq):
    """More batch rows than the kernel keeps lengths for in shared memory
    (they are then read from global memory), ragged lengths."""
    B, Hq, Hkv, Tq, S, D = 300, 4, 2, 1, 300, 64
    x = W.decode_inputs(B, Hq, Hkv, Tq, S, D, seed=23)
    o, lse = run_gpu(gq, x, 0.125)
    assert gq.get_device_status() == 0
    ro, rlse = run_oracle(x, 0.125)
    check("o", o, ro, TOL_REL_O)
    check_lse(lse, rlse)
