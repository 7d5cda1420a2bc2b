"""Cached attention over a paged KV cache on the GPU against the fp64 oracle.

The pool's pages are shuffled over the rows (a random permutation), table
entries past each row's last page are -1 and must never be read.  Cases
cover every page-size class (16, 32, 64: several pages per 128-key chunk;
128 and 256: chunks inside one page), lengths that end inside a page, Tq > 1,
G = 1 and 7, D = 64 and 128, more than 16 query rows, a pool with spare
pages, an invalid table entry (reported, nothing outside the pool read), and
the paged long-context workloads at their full size.
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
    q, kp, vp, bt, lens = (x[n].cuda() for n in ("q", "k_pages", "v_pages", "block_table", "cache_lens"))
    return gq.attn_decode_paged_fwd(q, kp, vp, bt, lens, scale=scale, **kw)


def run_oracle(x, scale):
    return oracle.paged_decode_fwd(to64(x["q"]), to64(x["k_pages"]), to64(x["v_pages"]), x["block_table"].numpy(),
                                   x["cache_lens"].numpy(), scale=scale)


CASES = [
    # B, Hq, Hkv, Tq, page_size, max_pages, D, cache_lens, spare pages
    (3, 8, 2, 1, 16, 40, 128, [640, 1, 145], 0),
    (3, 8, 2, 2, 32, 20, 64, [640, 33, 200], 3),
    (2, 14, 2, 1, 64, 12, 64, [768, 257], 0),
    (2, 4, 4, 3, 128, 6, 128, [768, 130], 5),
    (2, 16, 2, 4, 256, 3, 128, [768, 300], 0),
    (4, 32, 8, 1, 16, 256, 128, None, 7),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%d_Hq%d_Hkv%d_Tq%d_page%d_D%d" % (c[0], c[1], c[2], c[3], c[4], c[6]))
def test_paged_decode_matches_oracle(gq, case):
    B, Hq, Hkv, Tq, psz, maxp, D, lens, spare = case
    x = W.paged_decode_inputs(B, Hq, Hkv, Tq, psz, maxp, D, cache_lens=lens, spare_pages=spare, seed=21)
    scale = 1.0 / np.sqrt(D)
    o, lse = run_gpu(gq, x, scale)
    assert gq.get_device_status() == 0
    ro, rlse = run_oracle(x, scale)
    check("o", o, ro, TOL_REL_O)
    check_lse(lse, rlse)


def test_paged_equals_contiguous(gq):
    """The same cache laid out contiguously and paged gives the same bits."""
    B, Hq, Hkv, Tq, psz, maxp, D = 2, 8, 2, 1, 64, 20, 128
    x = W.paged_decode_inputs(B, Hq, Hkv, Tq, psz, maxp, D, cache_lens=[1280, 700], seed=4)
    S = psz * maxp
    k = torch.zeros(B, Hkv, S, D, dtype=torch.bfloat16)
    v = torch.zeros(B, Hkv, S, D, dtype=torch.bfloat16)
    for b in range(B):
        for i in range((int(x["cache_lens"][b]) + psz - 1) // psz):
            pg = int(x["block_table"][b, i])
            k[b, :, i * psz:(i + 1) * psz] = x["k_pages"][pg]
            v[b, :, i * psz:(i + 1) * psz] = x["v_pages"][pg]
    o1, l1 = run_gpu(gq, x, 0.1)
    o2, l2 = gq.attn_decode_fwd(x["q"].cuda(), k.cuda(), v.cuda(), x["cache_lens"].cuda(), scale=0.1)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_paged_reports_invalid_page(gq):
    """An entry naming no page of the pool is reported (ATTN_ERR_PAGES); only the pool is read."""
    B, Hq, Hkv, Tq, psz, maxp, D = 2, 8, 2, 1, 32, 10, 64
    x = W.paged_decode_inputs(B, Hq, Hkv, Tq, psz, maxp, D, cache_lens=[320, 200], seed=6)
    x["block_table"][1, 2] = B * maxp + 1000
    run_gpu(gq, x, 0.1)
    assert gq.get_device_status() == 11
    assert gq.get_device_status() == 0


@pytest.mark.parametrize("name", [n for n, w in W.DECODE_WORKLOADS.items() if w.page_size])
def test_paged_decode_workloads_full(gq, name):
    w = W.DECODE_WORKLOADS[name]
    x = W.make_decode_inputs(w)
    o, lse = run_gpu(gq, x, w.softmax_scale)
    assert gq.get_device_status() == 0
    ro, rlse = run_oracle(x, w.softmax_scale)
    check("o", o, ro, TOL_REL_O)
    check_lse(lse, rlse)


def test_paged_rope_decode(gq):
    B, Hq, Hkv, Tq, psz, maxp, D = 3, 8, 2, 2, 32, 40, 128
    x = W.paged_decode_inputs(B, Hq, Hkv, Tq, psz, maxp, D, cache_lens=[1280, 2, 777], seed=8)
    tab = W.rope_cos_sin_table(psz * maxp, D)
    o, lse = run_gpu(gq, x, 0.09, rope_cos_sin=tab.cuda())
    assert gq.get_device_status() == 0
    ro, rlse = oracle.paged_decode_fwd(to64(x["q"]), to64(x["k_pages"]), to64(x["v_pages"]),
                                       x["block_table"].numpy(), x["cache_lens"].numpy(), scale=0.09,
                                       rope_cos_sin=tab.double().numpy())
    check("o", o, ro, TOL_REL_O)
    check_lse(lse, rlse)
